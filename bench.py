"""Benchmark: one decode step of compressed-KV attention (quantise the new token's K and V
into the packed cache, then decode attention over the whole packed context), on the
Qwen2.5-7B-shaped GQA layer: batch 1, 28 query / 4 KV heads, head_dim 128, 32768 tokens,
K 3-bit product code, V 4-bit MSE code, bf16 inputs.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead.
Metric: KV tokens/s = (tokens attended per sequence, summed over the batch) / step time.
Multi-GPU (torchrun): every rank runs its own independent batch (weak scaling, no
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
FALLBACK_HBM_GBS = 6800.0


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks sampling

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


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


# ------------------------------------------------------------------ our implementation

def run_ours(args):
    import torch

    from kv_cache_quantization_gb300 import api, synth

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = synth.WORKLOADS[args.workload]
    if w.k_bits == 0:
        return run_ours_asym(args, w, ws, rank, dev)
    ctx = w.context
    # tokens attended per sequence this step (ragged for the serving workload); the cache
    # holds lens - 1 of them and the step appends the last one
    lens_np = synth.seq_lengths(w)
    lens_np[:] = [min(int(x), ctx) for x in lens_np]
    n_tok = int(sum(lens_np))
    kc, vc = api.Codec.prod(w.k_bits), api.Codec.mse(w.v_bits)

    # Prefill compaction: quantise the cached tokens once (not part of the timed step).
    k, v = synth.make_kv(w, device=dev)
    base_k = api.ProdCache.empty(w.batch, w.kv_heads, ctx, w.k_bits, device=dev)
    base_v = api.MSECache.empty(w.batch, w.kv_heads, ctx, w.v_bits, device=dev)
    pre = torch.tensor([int(x) - 1 for x in lens_np], dtype=torch.int32, device=dev)
    api.quantize_prod(kc, k, base_k, count=pre)
    api.quantize_mse(vc, v, base_v, count=pre)
    torch.cuda.synchronize()
    # compaction throughput (full cache, K and V), reported as an extra
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    api.quantize_prod(kc, k, base_k, count=pre)
    api.quantize_mse(vc, v, base_v, count=pre)
    ev1.record()
    torch.cuda.synchronize()
    compaction_ms = ev0.elapsed_time(ev1)
    del k, v

    # Rotate several cache copies so that each timed step reads from HBM, not L2.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = base_k.nbytes() + base_v.nbytes()
    copies = max(3, math.ceil(3 * l2 / per_copy))
    kcs = [base_k] + [api.ProdCache(*(t.clone() for t in (base_k.idx, base_k.sgn, base_k.xnorm,
                                                          base_k.rnorm))) for _ in range(copies - 1)]
    vcs = [base_v] + [api.MSECache(base_v.idx.clone(), base_v.xnorm.clone(), w.v_bits)
                      for _ in range(copies - 1)]
    steps_q = [synth.make_queries(w, device=dev, step=i)[:, :, 0] for i in range(4)]
    steps_kv = [synth.make_new_tokens(w, device=dev, step=i) for i in range(4)]
    pos = pre.clone()
    lens = torch.tensor([int(x) for x in lens_np], dtype=torch.int32, device=dev)
    plan = api.DecodePlan(w.batch, w.q_heads, w.kv_heads, ctx, int(max(lens_np)), w.in_dtype, w.out_dtype,
                          device=dev)
    out = plan.new_out(dev)
    stream = torch.cuda.current_stream(dev)

    def step(i, kv_new=None, q=None, stream=stream):
        kn, vn = kv_new if kv_new is not None else steps_kv[i % 4]
        c = i % copies
        api.quantize_prod(kc, kn, kcs[c], pos=pos, stream=stream)
        api.quantize_mse(vc, vn, vcs[c], pos=pos, stream=stream)
        plan.run(kc, vc, steps_q[i % 4] if q is None else q, kcs[c], vcs[c], lens, out,
                 stream=stream)

    def decode_only(i, stream=stream):
        c = i % copies
        plan.run(kc, vc, steps_q[i % 4], kcs[c], vcs[c], lens, out, stream=stream)

    # quantise K, quantise V, query fragments, split decode (its last CTA per head merges)
    launches_per_step = 4

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # The timed steps replay CUDA graphs captured from the same library calls, so that the
    # measurement is the GPU's time and not the Python launch loop's.
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            cs = torch.cuda.current_stream(dev)
            for i in range(args.steps):
                fn(i, stream=cs)
        stream.wait_stream(cap)
        return g

    g_step = capture(step)
    g_dec = capture(decode_only)
    g_step.replay()
    g_dec.replay()
    torch.cuda.synchronize()
    barrier(ws)

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(3):                 # untimed replays keep the clock sampler busy
            g_step.replay()
        torch.cuda.synchronize()
        barrier(ws)
        t0.record(stream)
        g_step.replay()                    # exactly args.steps steps
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        d0.record(stream)
        g_dec.replay()                     # the same decode-attention calls alone
        d1.record(stream)
        torch.cuda.synchronize()
    total_ms = t0.elapsed_time(t1)
    ms_per_step = max_over_ranks(total_ms / args.steps, ws, dev)
    dec_mean = max_over_ranks(d0.elapsed_time(d1) / args.steps, ws, dev)

    tokens_per_step = n_tok
    value = tokens_per_step * ws / (ms_per_step * 1e-3)
    # algorithmic bytes of one decode-attention call: packed K and V codes of every cached
    # token and head, the query and the output
    from kv_cache_quantization_gb300 import _binding as Bn
    code_bytes = (Bn.tq_code_bytes(Bn.TQ_PROD, w.k_bits) + Bn.tq_code_bytes(Bn.TQ_MSE, w.v_bits))
    dec_bytes = (w.kv_heads * n_tok * code_bytes
                 + w.batch * w.q_heads * 128 * (2 + torch.finfo(w.out_dtype).bits // 8))
    peak, peak_kind = read_peaks()
    achieved = dec_bytes / (dec_mean * 1e-3) / 1e9
    # compaction bytes: every cached vector read once (bf16) and its code written
    in_bytes = torch.finfo(w.in_dtype).bits // 8 * 128
    comp_bytes = w.kv_heads * (n_tok - w.batch) * (2 * in_bytes + code_bytes)
    traffic = None
    prof = os.path.join(ROOT, "profiles", "decode_attention_traffic.json")
    if os.path.exists(prof):
        try:
            traffic = json.load(open(prof)).get(args.workload)
        except Exception:
            traffic = None

    # ---------------- end to end through the public API with host buffers
    # a step's inputs (query, new key, new value) travel as one packed pinned buffer: one
    # host-to-device copy a step, the tensors the library sees are views into its device copy
    parts = [steps_q[0], steps_kv[0][0], steps_kv[0][1]]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs = [0, sizes[0], sizes[0] + sizes[1]]
    h2d = sum(sizes)
    in_dev = torch.empty(h2d, dtype=torch.uint8, device=dev)
    q_dev, k_dev, v_dev = (in_dev[o:o + n].view(t.dtype).view(t.shape)
                           for o, n, t in zip(offs, sizes, parts))
    in_host = []
    for i in range(4):
        buf = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        for o, n, t in zip(offs, sizes, (steps_q[i], steps_kv[i][0], steps_kv[i][1])):
            buf[o:o + n].copy_(t.contiguous().cpu().view(-1).view(torch.uint8))
        in_host.append(buf)
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d2h = out.numel() * out.element_size()
    def e2e_step(i, stream=stream):
        in_dev.copy_(in_host[i % 4], non_blocking=True)
        step(i, (k_dev, v_dev), q_dev, stream=stream)
        out_host.copy_(out, non_blocking=True)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(ws)
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_eager_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)
    # the same steps (copies in, library calls, copy out) captured once and replayed
    g_e2e = capture(e2e_step)
    g_e2e.replay()
    torch.cuda.synchronize()
    barrier(ws)
    e0.record(stream)
    g_e2e.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_graph_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)
    e2e_ms = min(e2e_graph_ms, e2e_eager_ms)

    result = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in / fp32 accumulate on packed K3/V4 codes",
        "data": "synthetic (seeded N(0,1) x lognormal(0,0.5) per channel)",
        "config": {"workload": w.name, "batch": w.batch, "q_heads": w.q_heads,
                   "kv_heads": w.kv_heads, "head_dim": 128, "context": ctx, "tokens_attended": n_tok,
                   "k_bits": w.k_bits, "v_bits": w.v_bits,
                   "parallelism": f"replicas x{ws} (independent batches)",
                   "l2": f"{copies} rotating cache copies ({copies * per_copy / 2**20:.0f} MiB > 3x L2)",
                   "step": "quantise new K,V token + decode attention over all tokens",
                   "timing": "CUDA-graph replay of the K steps, CUDA events around it"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "tq_decode_attention (query prep + split decode + merge)",
                     "algorithmic_bytes": dec_bytes, "ms": dec_mean,
                     "peak_source": peak_kind},
        "e2e": {"value": tokens_per_step * ws / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "timing": "every step: one pinned-host copy in (query, new key and value "
                          "packed), library calls, copy out; the faster of an eager Python "
                          "loop and one CUDA graph of the K steps",
                "ms_per_step_eager": e2e_eager_ms, "ms_per_step_graph": e2e_graph_ms},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "compaction": {"vectors": 2 * w.kv_heads * (n_tok - w.batch), "ms": compaction_ms,
                       "vectors_per_s": 2 * w.kv_heads * (n_tok - w.batch) / (compaction_ms * 1e-3),
                       "what": "quantise the cached K (product code) and V (MSE code) once",
                       "roofline": {"bound": "hbm", "unit": "GB/s", "peak": peak,
                                    "achieved": comp_bytes / (compaction_ms * 1e-3) / 1e9,
                                    "frac": comp_bytes / (compaction_ms * 1e-3) / 1e9 / peak,
                                    "algorithmic_bytes": comp_bytes,
                                    "note": "input vectors read once, codes and norms written"}},
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = oracle_baseline(w, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_ours_asym(args, w, ws, rank, dev):
    """Asymmetric workload: FP16 keys, 4-bit MSE values and an FP16 tail of 255 tokens per
    sequence.  The timed step is one decode-attention call over the compressed part and the
    tail (the tail's FP16 append is a copy, not part of this path)."""
    import torch

    from kv_cache_quantization_gb300 import api, synth

    lens_np = synth.seq_lengths(w)                       # compressed tokens per sequence
    tail = w.tail
    n_tok = int(sum(lens_np)) + w.batch * tail
    vc = api.Codec.mse(w.v_bits)
    k, v = synth.make_kv(w, device=dev)
    lens = torch.tensor([int(x) for x in lens_np], dtype=torch.int32, device=dev)
    tl = torch.full((w.batch,), tail, dtype=torch.int32, device=dev)
    tail_cap = 256
    base_v = api.MSECache.empty(w.batch, w.kv_heads, w.context, w.v_bits, device=dev)
    api.quantize_mse(vc, v, base_v, count=lens)
    k16 = k.to(torch.float16)
    kt = k16[:, :, w.context - tail_cap:].contiguous()
    vt = v[:, :, w.context - tail_cap:].to(torch.float16).contiguous()
    del k, v
    torch.cuda.synchronize()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = k16.numel() * 2 + base_v.nbytes() + kt.numel() * 4
    copies = max(3, math.ceil(3 * l2 / per_copy))
    sets = [(k16, base_v, kt, vt)] + [
        (k16.clone(), api.MSECache(base_v.idx.clone(), base_v.xnorm.clone(), w.v_bits), kt.clone(),
         vt.clone()) for _ in range(copies - 1)]
    steps_q = [synth.make_queries(w, device=dev, step=i)[:, :, 0] for i in range(4)]
    plan = api.DecodePlan(w.batch, w.q_heads, w.kv_heads, w.context, int(max(lens_np)), w.in_dtype,
                          w.out_dtype, device=dev, tail_capacity=tail_cap)
    out = plan.new_out(dev)
    stream = torch.cuda.current_stream(dev)

    def step(i, q=None, stream=stream):
        kk, vv, ktt, vtt = sets[i % copies]
        plan.run_asym(vc, steps_q[i % 4] if q is None else q, kk, vv, lens, ktt, vtt, tl, out,
                      stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.graph(g, stream=cap):
        cs = torch.cuda.current_stream(dev)
        for i in range(args.steps):
            step(i, stream=cs)
    stream.wait_stream(cap)
    g.replay()
    torch.cuda.synchronize()
    barrier(ws)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        barrier(ws)
        t0.record(stream)
        g.replay()
        t1.record(stream)
        torch.cuda.synchronize()
    ms_per_step = max_over_ranks(t0.elapsed_time(t1) / args.steps, ws, dev)
    value = n_tok * ws / (ms_per_step * 1e-3)
    from kv_cache_quantization_gb300 import _binding as Bn
    dec_bytes = (w.kv_heads * (int(sum(lens_np)) * (256 + Bn.tq_code_bytes(Bn.TQ_MSE, w.v_bits))
                               + w.batch * tail * 512)
                 + w.batch * w.q_heads * 128 * (2 + torch.finfo(w.out_dtype).bits // 8))
    peak, peak_kind = read_peaks()
    achieved = dec_bytes / (ms_per_step * 1e-3) / 1e9
    traffic = None
    prof = os.path.join(ROOT, "profiles", "decode_attention_traffic.json")
    if os.path.exists(prof):
        try:
            traffic = json.load(open(prof)).get(args.workload)
        except Exception:
            traffic = None
    # end to end: the query from pinned host memory in, the output back, every step
    q_host = [steps_q[i].cpu().pin_memory() for i in range(4)]
    q_dev = torch.empty_like(steps_q[0])
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    def e2e_step(i, stream=stream):
        q_dev.copy_(q_host[i % 4], non_blocking=True)
        step(i, q_dev, stream=stream)
        out_host.copy_(out, non_blocking=True)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(ws)
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_eager_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)
    g_e2e = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.graph(g_e2e, stream=cap):
        cs = torch.cuda.current_stream(dev)
        for i in range(args.steps):
            e2e_step(i, stream=cs)
    stream.wait_stream(cap)
    g_e2e.replay()
    torch.cuda.synchronize()
    barrier(ws)
    e0.record(stream)
    g_e2e.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_graph_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)
    e2e_ms = min(e2e_graph_ms, e2e_eager_ms)
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 queries, fp16 keys, 4-bit value codes / fp32 accumulate, bf16 out",
        "data": "synthetic (seeded N(0,1) x lognormal(0,0.5) per channel)",
        "config": {"workload": w.name, "batch": w.batch, "q_heads": w.q_heads,
                   "kv_heads": w.kv_heads, "head_dim": 128, "context": w.context,
                   "tokens_attended": n_tok, "k_bits": 0, "v_bits": w.v_bits, "tail": tail,
                   "parallelism": f"replicas x{ws} (independent batches)",
                   "l2": f"{copies} rotating copies ({copies * per_copy / 2**20:.0f} MiB > 3x L2)",
                   "step": "decode attention over the compressed part and the FP16 tail",
                   "timing": "CUDA-graph replay of the K steps, CUDA events around it"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "tq_decode_attention_asym (split decode + merge)",
                     "algorithmic_bytes": dec_bytes, "ms": ms_per_step, "peak_source": peak_kind},
        "e2e": {"value": n_tok * ws / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": q_dev.numel() * q_dev.element_size(),
                "d2h_bytes_per_step": out.numel() * out.element_size(), "ms_per_step": e2e_ms,
                "timing": "every step: pinned-host copy in, library call, copy out; the faster "
                          "of an eager Python loop and one CUDA graph of the K steps",
                "ms_per_step_eager": e2e_eager_ms, "ms_per_step_graph": e2e_graph_ms},
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
    }
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
            kt, vt = synth.make_kv(w, device="cpu", tokens=max(w.tail, 1))
            self.kx = k[0, 0].to(torch_f16()).double().numpy()
            self.kt = kt[0:1, 0:1].to(torch_f16()).double().numpy()
            self.vt = vt[0:1, 0:1].to(torch_f16()).double().numpy()

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


def oracle_baseline(w, budget_s=15.0):
    """cpu_baseline object: the oracle timed on its bounded sample for about budget_s."""
    smp = OracleSample(w)
    smp.rep()
    reps, t0 = 0, time.perf_counter()
    while True:
        smp.rep()
        reps += 1
        el = time.perf_counter() - t0
        if el > budget_s:
            break
    return {"value": smp.tokens_per_s(el / reps), "unit": UNIT, "cores": _blas_threads(),
            "kind": "oracle", "sample": smp.describe(reps, el)}


def torch_f16():
    import torch
    return torch.float16


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, W warm-up and K timed steps,
    each step one repetition of the bounded sample.  Only rank 0 runs."""
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
    ms = w.batch * w.context / value * 1e3
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name},
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
    ap.add_argument("--workload", default="decode_gqa28x4_ctx32768_k3v4")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
