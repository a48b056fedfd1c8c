"""Benchmark of compressed-KV decode attention (TurboQuant codes: product-quantised keys, MSE
values, attention on the packed bits).

The headline line is the long-context workload, the largest that fits one GPU: batch 1,
32 query / 8 KV heads, head_dim 128, 262144 cached tokens, K 3-bit product code (4 outlier
channels), V 2-bit MSE code, bf16 inputs.  One step = quantise the new token's K and V into
the packed cache, then decode attention over all 262144 tokens.  A ``per_workload`` block adds
the other decode workloads, each timed the same way:

* ``decode_gqa28x4_ctx32768_k3v4``: batch 1, 28/4 heads, 32768 tokens, K3/V4 (one step);
* ``asym_b8_ctx8192_kfp16_v4_tail255``: batch 8, FP16 keys, V 4-bit, FP16 tail of 255 tokens;
* ``serving_b32_ragged4k-16k_k4v4``: 32 ragged sequences, K4/V4, the workload's 128 decode
  steps: each appends one token per (sequence, KV head) and attends the grown cache.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead.
Metric: KV tokens/s = (tokens attended per sequence, summed over the batch) / step time.
Multi-GPU (torchrun): every rank runs its own independent replica (weak scaling, no
data-path collective); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "compressed-KV decode attention: KV tokens/s and % of GB300 HBM roofline"
UNIT = "KV tokens/s"
HEADLINE = "longctx_gqa32x8_ctx262144_k3v2"
PER_WORKLOAD = ["decode_gqa28x4_ctx32768_k3v4", "asym_b8_ctx8192_kfp16_v4_tail255",
                "serving_b32_ragged4k-16k_k4v4"]
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy test)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks sampling

class ClockSampler:
    """nvidia-smi sampling of SM clock, utilisation and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        loaded = [r for r in rows if (num(r[4]) or 0) >= 50]
        use = loaded or rows
        sm = [num(r[1]) for r in use if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "what": "median SM clock over samples with GPU utilisation >= 50%"}


# ------------------------------------------------------------------ distributed helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ timing helpers

class Graphs:
    """Captures a sequence of library calls once as a CUDA graph and replays it, so that the
    measurement is the GPU's time and not the Python launch loop's."""

    def __init__(self, dev):
        import torch
        self.torch = torch
        self.dev = dev
        self.stream = torch.cuda.current_stream(dev)

    def capture(self, fn, n):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(self.dev)
        cap.wait_stream(self.stream)
        with torch.cuda.graph(g, stream=cap):
            cs = torch.cuda.current_stream(self.dev)
            for i in range(n):
                fn(i, cs)
        self.stream.wait_stream(cap)
        g.replay()
        torch.cuda.synchronize()
        return g

    def time(self, g, ws):
        """Milliseconds of one replay of g (CUDA events on the replaying stream), max over
        ranks."""
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(ws)
        e0.record(self.stream)
        g.replay()
        e1.record(self.stream)
        torch.cuda.synchronize()
        barrier(ws)
        return max_over_ranks(e0.elapsed_time(e1), ws, self.dev)

    def busy(self, g, seconds):
        """Replays g for about `seconds` (untimed), so the clock sampler sees the GPU under
        load around a timed region."""
        torch = self.torch
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            g.replay()
            torch.cuda.synchronize()


def _elem_bytes(dt):
    import torch
    return torch.finfo(dt).bits // 8


def decode_bytes(w, tokens_total, out_dtype):
    """Algorithmic bytes of one decode-attention call: the packed K and V codes of every
    attended token and KV head, the queries and the outputs."""
    from kv_cache_quantization_gb300 import _binding as Bn
    code = Bn.tq_code_bytes(Bn.TQ_PROD, w.k_bits) + Bn.tq_code_bytes(Bn.TQ_MSE, w.v_bits)
    return (w.kv_heads * tokens_total * code
            + w.batch * w.q_heads * 128 * (_elem_bytes(w.in_dtype) + _elem_bytes(out_dtype)))


def roofline(bytes_, ms, workload, peak):
    from kv_cache_quantization_gb300.profiling import measured_traffic
    achieved = bytes_ / (ms * 1e-3) / 1e9
    traffic, note = measured_traffic(workload)
    return {"bound": "hbm", "achieved": achieved, "peak": peak[0], "unit": "GB/s",
            "frac": achieved / peak[0], "frac_of_nominal_7900": achieved / NOMINAL_HBM_GBS,
            "traffic": traffic, "traffic_note": note, "algorithmic_bytes": bytes_, "ms": ms,
            "peak_source": peak[1]}


# ------------------------------------------------------------------ symmetric workloads

class SymWorkload:
    """Codecs, packed caches and per-step inputs of a symmetric workload, quantised once (the
    prefill compaction, also timed)."""

    def __init__(self, w, dev):
        import torch

        from kv_cache_quantization_gb300 import api, synth
        self.w = w
        self.dev = dev
        self.api = api
        cap = synth.cache_capacity(w)
        lens0 = [min(int(x), w.context) for x in synth.seq_lengths(w)]
        # tokens in the cache before the timed steps: one-step workloads append their step's
        # token at len - 1; the decode loop appends at len, len + 1, ...
        self.loop = w.decode_steps > 0
        pre = lens0 if self.loop else [x - 1 for x in lens0]
        self.lens0 = lens0
        self.kc, self.vc = api.Codec.prod(w.k_bits, w.layer), api.Codec.mse(w.v_bits, w.layer)
        k, v = synth.make_kv(w, device=dev)
        self.kcache = api.ProdCache.empty(w.batch, w.kv_heads, cap, w.k_bits, device=dev)
        self.vcache = api.MSECache.empty(w.batch, w.kv_heads, cap, w.v_bits, device=dev)
        pre_t = torch.tensor(pre, dtype=torch.int32, device=dev)
        api.quantize_prod(self.kc, k, self.kcache, count=pre_t)
        api.quantize_mse(self.vc, v, self.vcache, count=pre_t)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        api.quantize_prod(self.kc, k, self.kcache, count=pre_t)
        api.quantize_mse(self.vc, v, self.vcache, count=pre_t)
        e1.record()
        torch.cuda.synchronize()
        self.compaction_eager_ms = e0.elapsed_time(e1)
        # the same two calls as a CUDA graph, replayed after an L2 flush: the GPU's time without
        # the Python launch overhead of the first call (the decode steps are timed the same way)
        g = Graphs(dev).capture(
            lambda i, cs: (api.quantize_prod(self.kc, k, self.kcache, count=pre_t, stream=cs),
                           api.quantize_mse(self.vc, v, self.vcache, count=pre_t, stream=cs)), 1)
        flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size,
                            dtype=torch.uint8, device=dev)
        reps = []
        for r in range(5):
            flush.fill_(r)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            reps.append(e0.elapsed_time(e1))
        del g, flush
        self.compaction_ms = sorted(reps)[len(reps) // 2]
        self.compaction_vectors = 2 * w.kv_heads * sum(pre)
        self.compaction_bytes = w.kv_heads * sum(pre) * (
            2 * 128 * _elem_bytes(w.in_dtype) + api.B.tq_code_bytes(api.B.TQ_PROD, w.k_bits)
            + api.B.tq_code_bytes(api.B.TQ_MSE, w.v_bits))
        del k, v
        self.cap = cap
        nsteps = w.decode_steps if self.loop else 4
        self.queries = [synth.make_queries(w, device=dev, step=i)[:, :, 0] for i in range(nsteps)]
        self.new_kv = [synth.make_new_tokens(w, device=dev, step=i) for i in range(nsteps)]
        if self.loop:
            # append positions of step s are lens0 + s, the attended lengths lens0 + s + 1
            self.lens = [torch.tensor([x + s for x in lens0], dtype=torch.int32, device=dev)
                         for s in range(nsteps + 1)]
            self.caches = [(self.kcache, self.vcache)]
        else:
            self.pos = pre_t
            self.lens = torch.tensor(lens0, dtype=torch.int32, device=dev)
            # rotating copies: every step reads its cache from HBM, not L2
            l2 = torch.cuda.get_device_properties(dev).L2_cache_size
            per = self.kcache.nbytes() + self.vcache.nbytes()
            self.copies = max(3, math.ceil(3 * l2 / per))
            self.caches = [(self.kcache, self.vcache)] + [
                (api.ProdCache(*(t.clone() for t in (self.kcache.idx, self.kcache.sgn,
                                                      self.kcache.xnorm, self.kcache.rnorm))),
                 api.MSECache(self.vcache.idx.clone(), self.vcache.xnorm.clone(), w.v_bits))
                for _ in range(self.copies - 1)]
            self.per_copy = per
        self.plan = api.DecodePlan(w.batch, w.q_heads, w.kv_heads, cap,
                                   max(lens0) + (w.decode_steps if self.loop else 0),
                                   w.in_dtype, w.out_dtype, device=dev)
        self.out = self.plan.new_out(dev)
        self.nsteps = nsteps

    def tokens(self, i):
        """Tokens attended (summed over the batch) at step i."""
        return sum(self.lens0) + (i + 1) * self.w.batch if self.loop else sum(self.lens0)

    def step(self, i, stream, kv=None, q=None):
        """One decode step through tq_decode_step: the new token's key and value are appended
        at pos and pos + 1 tokens are attended."""
        s = i % self.nsteps
        kn, vn = kv if kv is not None else self.new_kv[s]
        q = self.queries[s] if q is None else q
        if self.loop:
            kcache, vcache = self.caches[0]
            pos = self.lens[s]
        else:
            kcache, vcache = self.caches[i % self.copies]
            pos = self.pos
        self.plan.step(self.kc, self.vc, q, kn[:, :, 0], vn[:, :, 0], kcache, vcache, pos,
                       self.out, stream=stream)

    def decode_only(self, i, stream):
        s = i % self.nsteps
        if self.loop:
            kcache, vcache = self.caches[0]
            lens = self.lens[s + 1]
        else:
            kcache, vcache = self.caches[i % self.copies]
            lens = self.lens
        self.plan.run(self.kc, self.vc, self.queries[s], kcache, vcache, lens, self.out,
                      stream=stream)

    def l2_note(self):
        if self.loop:
            return (f"one cache of {self.kcache.nbytes() + self.vcache.nbytes() >> 20} MiB "
                    f"(> L2), appended in place by the decode loop")
        return f"{self.copies} rotating cache copies ({self.copies * self.per_copy >> 20} MiB > 3x L2)"

    def compaction(self, peak):
        ms = self.compaction_ms
        return {"vectors": self.compaction_vectors, "ms": ms,
                "vectors_per_s": self.compaction_vectors / (ms * 1e-3),
                "what": "quantise the cached K (product code) and V (MSE code) once",
                "timing": "CUDA-graph replay of the two calls after an L2 flush, median of 5",
                "eager_ms": self.compaction_eager_ms,
                "roofline": {"bound": "hbm", "unit": "GB/s", "peak": peak[0],
                             "achieved": self.compaction_bytes / (ms * 1e-3) / 1e9,
                             "frac": self.compaction_bytes / (ms * 1e-3) / 1e9 / peak[0],
                             "algorithmic_bytes": self.compaction_bytes,
                             "note": "input vectors read once, codes and norms written"}}


def measure_sym(w, args, dev, ws, peak, headline, clk=None):
    import torch
    g = Graphs(dev)
    S = SymWorkload(w, dev)
    n = w.decode_steps if S.loop else args.steps
    for i in range(max(args.warmup, 3)):
        S.step(i, g.stream)
    torch.cuda.synchronize()
    g_step = g.capture(S.step, n)
    g_dec = g.capture(S.decode_only, n)
    if headline:
        g.busy(g_step, 1.0)
    step_ms = g.time(g_step, ws) / n
    if headline:
        g.busy(g_step, 0.5)
    dec_ms = g.time(g_dec, ws) / n
    tokens = [S.tokens(i) for i in range(n)]
    mean_tokens = sum(tokens) / n
    dec_bytes = decode_bytes(w, mean_tokens, w.out_dtype)
    res = {
        "value": mean_tokens * ws / (step_ms * 1e-3), "unit": UNIT, "ms_per_step": step_ms,
        "steps": n, "tokens_attended_per_step": mean_tokens,
        "step": ("append one new K,V token per (sequence, KV head) at its length, then decode "
                 "attention over the grown cache; the workload's 128 steps" if S.loop else
                 "quantise the new K,V token at position len-1, then decode attention over len "
                 "tokens; the workload's one decode step, repeated"),
        "l2": S.l2_note(),
        "decode_call": roofline(dec_bytes, dec_ms, w.name, peak),
        "compaction": S.compaction(peak),
        "gpu_launches": 2 * n,
    }
    if not headline:
        return res
    # ---------------- end to end through the public API with host buffers: a step's inputs
    # (query, new key and value) travel as one packed pinned buffer, the output comes back
    parts = [S.queries[0], S.new_kv[0][0], S.new_kv[0][1]]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs = [0, sizes[0], sizes[0] + sizes[1]]
    h2d = sum(sizes)
    in_dev = torch.empty(h2d, dtype=torch.uint8, device=dev)
    q_dev, k_dev, v_dev = (in_dev[o:o + m].view(t.dtype).view(t.shape)
                           for o, m, t in zip(offs, sizes, parts))
    in_host = []
    for i in range(4):
        buf = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        for o, m, t in zip(offs, sizes, (S.queries[i], S.new_kv[i][0], S.new_kv[i][1])):
            buf[o:o + m].copy_(t.contiguous().cpu().view(-1).view(torch.uint8))
        in_host.append(buf)
    out_host = torch.empty(S.out.shape, dtype=S.out.dtype).pin_memory()
    d2h = S.out.numel() * S.out.element_size()

    def e2e_step(i, stream):
        in_dev.copy_(in_host[i % 4], non_blocking=True)
        S.step(i, stream, (k_dev, v_dev), q_dev)
        out_host.copy_(S.out, non_blocking=True)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(ws)
    e0.record(g.stream)
    for i in range(n):
        e2e_step(i, g.stream)
    e1.record(g.stream)
    torch.cuda.synchronize()
    eager_ms = max_over_ranks(e0.elapsed_time(e1) / n, ws, dev)
    graph_ms = g.time(g.capture(e2e_step, n), ws) / n
    res["e2e"] = {"value": mean_tokens * ws / (eager_ms * 1e-3), "unit": UNIT,
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                  "ms_per_step": eager_ms,
                  "timing": "eager Python loop over the steps; every step one pinned-host copy "
                            "in (query, new key and value packed), the library calls, the "
                            "output copied out",
                  "graph_value": mean_tokens * ws / (graph_ms * 1e-3),
                  "graph_ms_per_step": graph_ms,
                  "graph_timing": "the same steps captured once as a CUDA graph and replayed"}
    return res


# ------------------------------------------------------------------ asymmetric workload

def measure_asym(w, args, dev, ws, peak):
    """FP16 keys, 4-bit MSE values and an FP16 tail of 255 tokens per sequence.  The step is
    one decode-attention call over the compressed part and the tail."""
    import torch

    from kv_cache_quantization_gb300 import _binding as Bn
    from kv_cache_quantization_gb300 import api, synth
    g = Graphs(dev)
    lens_np = synth.seq_lengths(w)
    n_tok = int(sum(lens_np)) + w.batch * w.tail
    vc = api.Codec.mse(w.v_bits, w.layer)
    k, v = synth.make_kv(w, device=dev)
    kt, vt = synth.asym_tail(w, k, v)
    lens = torch.tensor([int(x) for x in lens_np], dtype=torch.int32, device=dev)
    tl = torch.full((w.batch,), w.tail, dtype=torch.int32, device=dev)
    base_v = api.MSECache.empty(w.batch, w.kv_heads, w.context, w.v_bits, device=dev)
    api.quantize_mse(vc, v, base_v, count=lens)
    k16 = k.to(torch.float16)
    del k, v
    torch.cuda.synchronize()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per = k16.numel() * 2 + base_v.nbytes() + kt.numel() * 4
    copies = max(3, math.ceil(3 * l2 / per))
    sets = [(k16, base_v, kt, vt)] + [
        (k16.clone(), api.MSECache(base_v.idx.clone(), base_v.xnorm.clone(), w.v_bits),
         kt.clone(), vt.clone()) for _ in range(copies - 1)]
    queries = [synth.make_queries(w, device=dev, step=i)[:, :, 0] for i in range(4)]
    plan = api.DecodePlan(w.batch, w.q_heads, w.kv_heads, w.context, int(max(lens_np)),
                          w.in_dtype, w.out_dtype, device=dev,
                          tail_capacity=synth.TAIL_CAPACITY)
    out = plan.new_out(dev)

    def step(i, stream):
        kk, vv, ktt, vtt = sets[i % copies]
        plan.run_asym(vc, queries[i % 4], kk, vv, lens, ktt, vtt, tl, out, stream=stream)

    for i in range(max(args.warmup, 3)):
        step(i, g.stream)
    ms = g.time(g.capture(step, args.steps), ws) / args.steps
    dec_bytes = (w.kv_heads * (int(sum(lens_np)) * (256 + Bn.tq_code_bytes(Bn.TQ_MSE, w.v_bits))
                               + w.batch * w.tail * 512)
                 + w.batch * w.q_heads * 128 * (_elem_bytes(w.in_dtype) + _elem_bytes(w.out_dtype)))
    return {"value": n_tok * ws / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "steps": args.steps, "tokens_attended_per_step": n_tok,
            "step": "decode attention over the compressed part (FP16 keys, 4-bit values) and "
                    "the FP16 tail",
            "l2": f"{copies} rotating copies ({copies * per >> 20} MiB > 3x L2)",
            "decode_call": roofline(dec_bytes, ms, w.name, peak), "gpu_launches": 2 * args.steps}


# ------------------------------------------------------------------ quality report

def quality_report(dev):
    """Attention-level KL divergence and top-1 agreement of compressed keys against exact keys
    (tq_attention_quality) on the 32K workload's data: every query head against its KV head's
    32768 keys, for 3-bit and 4-bit product codes; FP16 keys (the asymmetric mode) attend
    exactly up to FP16 rounding."""
    import torch

    from kv_cache_quantization_gb300 import api, synth
    w = synth.DECODE_32K
    k, _ = synth.make_kv(w, device=dev)
    q = synth.make_queries(w, device=dev)[0, :, 0].float()
    rep = {"workload": w.name, "queries": w.q_heads, "keys_per_query": w.context}
    for bits in (3, 4):
        kc = api.Codec.prod(bits, w.layer)
        cache = api.ProdCache.empty(1, w.kv_heads, w.context, bits, device=dev)
        api.quantize_prod(kc, k, cache)
        kls, agree = [], 0
        for h in range(w.kv_heads):
            one = api.ProdCache(cache.idx[:, h:h + 1], cache.sgn[:, h:h + 1],
                                cache.xnorm[:, h:h + 1], cache.rnorm[:, h:h + 1])
            one = api.ProdCache(*(t.contiguous() for t in (one.idx, one.sgn, one.xnorm, one.rnorm)))
            kl, te, tc = api.attention_quality(kc, q[h * w.group:(h + 1) * w.group], k[0, h],
                                               one, w.context)
            kls += kl.tolist()
            agree += int((te == tc).sum())
        rep[f"k{bits}_prod"] = {"kl_mean": sum(kls) / len(kls), "kl_max": max(kls),
                                "top1_agreement": agree / w.q_heads}
    torch.cuda.synchronize()
    return rep


# ------------------------------------------------------------------ our implementation

def describe(w, ws):
    return {"workload": w.name, "batch": w.batch, "q_heads": w.q_heads, "kv_heads": w.kv_heads,
            "head_dim": 128, "context": w.context, "k_bits": w.k_bits, "v_bits": w.v_bits,
            "tail": w.tail, "decode_steps": w.decode_steps, "layer": w.layer,
            "parallelism": f"replicas x{ws} (independent batches)"}


def run_ours(args):
    import torch

    from kv_cache_quantization_gb300 import synth

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peak = read_peaks()
    w = synth.WORKLOADS[args.workload]
    with ClockSampler(torch.cuda.current_device()) as clk:
        if w.k_bits == 0:
            head = measure_asym(w, args, dev, ws, peak)
        else:
            head = measure_sym(w, args, dev, ws, peak, headline=True)
    clocks = clk.summary()
    per = {}
    if not args.no_per_workload:
        for name in PER_WORKLOAD:
            if name == w.name:
                continue
            wl = synth.WORKLOADS[name]
            with ClockSampler(torch.cuda.current_device()) as c2:
                r = (measure_asym(wl, args, dev, ws, peak) if wl.k_bits == 0
                     else measure_sym(wl, args, dev, ws, peak, headline=False))
            r["config"] = describe(wl, ws)
            r["clocks"] = c2.summary()
            per[name] = r
            torch.cuda.empty_cache()
    result = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": ws,
        "steps": head["steps"], "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in; fp32 accumulation on packed codes (e4m3 x e4m3 key products, fp16 "
                 "value products)",
        "data": "synthetic (seeded N(0,1); keys with 4 outlier channels x10)",
        "config": dict(describe(w, ws), tokens_attended=head["tokens_attended_per_step"],
                       l2=head["l2"], step=head["step"],
                       timing="CUDA-graph replay of the K steps, CUDA events around it"),
        "roofline": dict(head["decode_call"],
                         kernel="tq_decode_attention (query operand + split decode with its "
                                "merge); the step is tq_decode_step (appends + operand in one "
                                "prologue launch, then the split decode)"),
        "e2e": head.get("e2e"),
        "gpu_launches": head["gpu_launches"],
        "clocks": clocks,
        "compaction": head.get("compaction"),
        "per_workload": per,
    }
    if not args.no_per_workload:
        result["quality"] = quality_report(dev)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = oracle_baseline(w, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ the CPU oracle

class OracleSample:
    """A bounded sample of the workload for the CPU oracle (as it stands): one KV head's GQA
    group over a prefix of the context.  One repetition quantises the sample's K and V and
    runs decode attention over it."""

    def __init__(self, w, sample_tokens=4096):
        import oracle.turboquant as o
        from kv_cache_quantization_gb300 import synth
        from kv_cache_quantization_gb300.synth import gaussian_matrix, layer_seeds

        self.o = o
        self.w = w
        self.n = min(w.context, sample_tokens)
        k, v = synth.make_kv(w, device="cpu", tokens=self.n)
        q = synth.make_queries(w, device="cpu")[:, :, 0]
        sp, ss = layer_seeds(w.layer)
        self.pi, self.s = o.rotation_from_gaussian(gaussian_matrix(sp)), gaussian_matrix(ss)
        self.ck = o.lloyd_max_codebook(128, w.k_bits - 1)[0] if w.k_bits else None
        self.cv = o.lloyd_max_codebook(128, w.v_bits)[0]
        self.kx = k[0, 0].double().numpy()
        self.vx = v[0, 0].double().numpy()
        self.q = q[0:1, :w.group].double().numpy()
        if not w.k_bits:
            # asymmetric: FP16 keys, and an FP16 tail of w.tail tokens after the sample
            import torch
            kt, vt = synth.make_kv(w, device="cpu", tokens=max(w.tail, 1))
            self.kx = k[0, 0].to(torch.float16).double().numpy()
            self.kt = kt[0:1, 0:1].to(torch.float16).double().numpy()
            self.vt = vt[0:1, 0:1].to(torch.float16).double().numpy()

    def rep(self):
        o = self.o
        if self.ck is None:
            vi, vn, _ = o.quantize_mse(self.vx, self.pi, self.cv)
            o.decode_attention_asym(self.q, self.kx[None, None], {"idx": vi[None, None], "n": vn[None, None]},
                                    [self.n], self.kt, self.vt, [self.w.tail], self.pi, self.cv)
            return
        kq = o.quantize_prod(self.kx, self.pi, self.s, self.ck)
        vi, vn, _ = o.quantize_mse(self.vx, self.pi, self.cv)
        o.decode_attention(self.q, {k: kq[k][None, None] for k in ("idx", "sign", "n", "gamma")},
                           {"idx": vi[None, None], "n": vn[None, None]}, [self.n], self.pi,
                           self.s, self.ck, self.cv)

    def tokens_per_s(self, seconds_per_rep):
        """KV tokens/s of a whole step equivalent: one of kv_heads heads per repetition."""
        return (self.n + (0 if self.ck is not None else self.w.tail)) / (seconds_per_rep * self.w.kv_heads)

    def describe(self, reps, el):
        what = "quantise K/V + attention" if self.ck is not None else "quantise V + attention with FP16 keys and tail"
        return (f"1 of {self.w.kv_heads} KV heads (its {self.w.group} query heads), {self.n} of "
                f"{self.w.context} tokens; {what}; {reps} reps in {el:.1f} s")


def _timed_reps(smp, budget_s):
    smp.rep()
    reps, t0 = 0, time.perf_counter()
    while True:
        smp.rep()
        reps += 1
        el = time.perf_counter() - t0
        if el > budget_s:
            return reps, el


def oracle_baseline(w, budget_s=15.0):
    """cpu_baseline object: the oracle timed on its bounded sample for about budget_s with the
    BLAS threads it has, and for a shorter while on one thread."""
    smp = OracleSample(w)
    reps, el = _timed_reps(smp, budget_s)
    out = {"value": smp.tokens_per_s(el / reps), "unit": UNIT, "cores": _blas_threads(),
           "kind": "oracle", "sample": smp.describe(reps, el)}
    # one thread: a fresh interpreter whose BLAS is limited to one thread from the start
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--single-thread-oracle",
                            "--workload", w.name, "--cpu-seconds", str(budget_s / 3)],
                           env=env, capture_output=True, text=True, timeout=300)
        out["single_thread_value"] = float(r.stdout.strip().splitlines()[-1])
    except Exception:
        out["single_thread_value"] = None
    return out


def single_thread_oracle(args):
    from kv_cache_quantization_gb300 import synth
    smp = OracleSample(synth.WORKLOADS[args.workload])
    reps, el = _timed_reps(smp, args.cpu_seconds)
    print(smp.tokens_per_s(el / reps))


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, W warm-up and K timed steps, each
    step one repetition of the bounded sample.  Only rank 0 runs."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from kv_cache_quantization_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    # size the sample so that the whole run stays within a few minutes
    smp = OracleSample(w, sample_tokens=1024 if args.steps + args.warmup > 60 else 4096)
    for _ in range(args.warmup):
        smp.rep()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        smp.rep()
    el = time.perf_counter() - t0
    value = smp.tokens_per_s(el / args.steps)
    tokens = int(sum(min(int(x), w.context) for x in synth.seq_lengths(w))) + w.batch * w.tail
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "ms_per_step_what": "one repetition of the bounded sample (measured)",
        "full_step_ms_extrapolated": tokens / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(describe(w, ws), tokens_attended=tokens),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
                         "sample": smp.describe(args.steps, el)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--single-thread-oracle", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.single_thread_oracle:
        single_thread_oracle(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
