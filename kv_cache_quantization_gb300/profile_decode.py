"""A short, plain run of one decode workload for profilers: the workload's cache is quantised
once, then `--calls` decode calls (or decode steps with `--step`) are launched one after the
other, with no CUDA graph and no timing loop, so that a profiler sees few launches.

    python -m kv_cache_quantization_gb300.profile_decode --workload longctx_gqa32x8_ctx262144_k3v2 --calls 3

Launch order: the prefill quantisation (quantize kernels), then per call the query-operand
kernel (or a step's prologue) and the split kernel (asymmetric workload: the split kernel and
its merge).
"""
from __future__ import annotations

import argparse

import torch

from . import api, synth


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="longctx_gqa32x8_ctx262144_k3v2")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--step", action="store_true", help="decode steps (appends + attention)")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    lens = [min(int(x), w.context) for x in synth.seq_lengths(w)]
    k, v = synth.make_kv(w, device=dev)
    q = synth.make_queries(w, device=dev)[:, :, 0]
    if w.k_bits == 0:
        vc = api.Codec.mse(w.v_bits, w.layer)
        lt = torch.tensor(lens, dtype=torch.int32, device=dev)
        vcache = api.MSECache.empty(w.batch, w.kv_heads, w.context, w.v_bits, device=dev)
        api.quantize_mse(vc, v, vcache, count=lt)
        kt, vt = synth.asym_tail(w, k, v)
        k16 = k.to(torch.float16)
        tl = torch.full((w.batch,), w.tail, dtype=torch.int32, device=dev)
        plan = api.DecodePlan(w.batch, w.q_heads, w.kv_heads, w.context, max(lens), w.in_dtype,
                              w.out_dtype, tail_capacity=synth.TAIL_CAPACITY, device=dev)
        out = plan.new_out(dev)
        for _ in range(args.calls):
            plan.run_asym(vc, q, k16, vcache, lt, kt, vt, tl, out)
    else:
        cap = synth.cache_capacity(w)
        kc, vc = api.Codec.prod(w.k_bits, w.layer), api.Codec.mse(w.v_bits, w.layer)
        kcache = api.ProdCache.empty(w.batch, w.kv_heads, cap, w.k_bits, device=dev)
        vcache = api.MSECache.empty(w.batch, w.kv_heads, cap, w.v_bits, device=dev)
        pre = torch.tensor([x - 1 for x in lens], dtype=torch.int32, device=dev)
        api.quantize_prod(kc, k, kcache, count=pre)
        api.quantize_mse(vc, v, vcache, count=pre)
        lt = pre + 1
        plan = api.DecodePlan(w.batch, w.q_heads, w.kv_heads, cap, max(lens), w.in_dtype,
                              w.out_dtype, device=dev)
        out = plan.new_out(dev)
        kn, vn = synth.make_new_tokens(w, device=dev)
        for _ in range(args.calls):
            if args.step:
                plan.step(kc, vc, q, kn[:, :, 0], vn[:, :, 0], kcache, vcache, pre, out)
            else:
                plan.run(kc, vc, q, kcache, vcache, lt, out)
    torch.cuda.synchronize()
    print(f"{w.name}: {args.calls} {'steps' if args.step else 'calls'} done")


if __name__ == "__main__":
    main()
