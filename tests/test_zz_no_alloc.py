"""tq_decode_attention_noalloc: decode attention for callers that cannot allocate device
memory (for example a runtime plugin whose enqueue call may not allocate, or a process whose
device memory belongs to another framework's pool).  It keeps its scratch in a static
device array inside the library instead of a caller-provided workspace.

Checked through the C ABI: after a call with a larger descriptor has filled the static array
with its own data, two calls in a row give bit for bit the output of the ordinary workspace
entry point (both run the same kernels with a fixed merge order), and a request that needs
more scratch than the static array is refused with TQ_ERR_SCRATCH_LIMIT before anything is
launched.  This file is collected last on purpose and does not depend on any state left by
other tests.
"""
import numpy as np
import pytest
import torch

from kv_cache_quantization_gb300 import _binding as B
from kv_cache_quantization_gb300 import api

pytestmark = pytest.mark.gpu


def _case(batch, hq, hkv, ctx, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    k = torch.randn(batch, hkv, ctx, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(batch, hkv, ctx, 128, generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn(batch, hq, 128, generator=g, device="cuda").to(torch.bfloat16)
    kc, vc = api.Codec.prod(3), api.Codec.mse(4)
    kcache = api.ProdCache.empty(batch, hkv, ctx, 3)
    vcache = api.MSECache.empty(batch, hkv, ctx, 4)
    api.quantize_prod(kc, k, kcache)
    api.quantize_mse(vc, v, vcache)
    lens = torch.full((batch,), ctx, dtype=torch.int32, device="cuda")
    return kc, vc, q, kcache, vcache, lens


def _rel(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def _noalloc(plan, kc, vc, q, kcache, vcache, lens):
    out = torch.full(plan.shape, float("nan"), device="cuda")
    st = B.tq_decode_attention_noalloc(plan.desc, kc.handle, vc.handle, q, kcache.c(),
                                       vcache.c(), lens, out,
                                       torch.cuda.current_stream().cuda_stream)
    assert st == B.TQ_OK, B.tq_status_string(st)
    return out


def test_noalloc_matches_workspace_entry_point():
    B.load()
    # a larger descriptor first: its records and operand images cover the bytes where the
    # smaller call below keeps its split tickets
    big = _case(8, 28, 4, 4096, 90)
    big_plan = api.DecodePlan(8, 28, 4, 4096, 4096, torch.bfloat16, torch.float32)
    assert B.tq_decode_workspace_bytes(big_plan.desc) <= B.tq_decode_noalloc_scratch_bytes()
    big_out = _noalloc(big_plan, *big)
    batch, hq, hkv, ctx = 2, 28, 4, 4096
    kc, vc, q, kcache, vcache, lens = _case(batch, hq, hkv, ctx, 91)
    plan = api.DecodePlan(batch, hq, hkv, ctx, ctx, q.dtype, torch.float32)
    assert B.tq_decode_workspace_bytes(plan.desc) <= B.tq_decode_noalloc_scratch_bytes()
    ref = plan.run(kc, vc, q, kcache, vcache, lens, plan.new_out())
    big_ref = big_plan.run(*big, big_plan.new_out())
    # two calls in a row share (and reuse) the static scratch
    outs = [_noalloc(plan, kc, vc, q, kcache, vcache, lens) for _ in range(2)]
    torch.cuda.synchronize()
    assert torch.equal(big_out, big_ref)
    for out in outs:
        assert torch.isfinite(out).all()
        assert torch.equal(out, ref), f"rel L2 {_rel(out, ref):.3g}"
    assert B.tq_device_status()[0] == B.TQ_OK


def test_noalloc_rejects_requests_beyond_the_static_scratch():
    B.load()
    # a very large batch: its per-query vectors alone exceed the static array
    desc = B.tq_attn_desc(2048, 32, 8, 128, 4096, 4096, 0, 0.0, B.TQ_BF16, B.TQ_F32)
    need = B.tq_decode_workspace_bytes(desc)
    assert need > B.tq_decode_noalloc_scratch_bytes()
    st = B.tq_decode_attention_noalloc(desc, None, None, 16, B.tq_prod_cache(16, 16, 16, 16),
                                       B.tq_mse_cache(16, 16), 16, 16, None)
    assert st == B.TQ_ERR_SCRATCH_LIMIT
    assert B.tq_status_string(st) == "TQ_ERR_SCRATCH_LIMIT"
