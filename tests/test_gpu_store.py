"""The FP16-tail store (tq_store_append) against a replay of its policy and the CPU oracle.

600 appends per sequence run through two compactions of the 256-slot tail.  After chosen
appends the lengths match the policy (compact when the tail fills) and decode attention on the
store (compressed part: FP16 keys and MSE-coded values; tail: FP16 keys and values) matches the
oracle's asymmetric attention over the same tokens, every query head on its own.  The
compressed values' codes match the oracle's quantisation of the FP16 tail values they came from.
"""
import numpy as np
import pytest
import torch

import oracle.turboquant as o
from kv_cache_quantization_gb300 import _binding as B
from kv_cache_quantization_gb300 import api
from parity import CodeStats, check_heads, match_mse_codes, oracle_codebook, oracle_constants, unpack_mse

pytestmark = pytest.mark.gpu

D = 128


def _draw(shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g, device="cuda").to(torch.bfloat16)


@pytest.mark.parametrize("vbits,hq,hkv", [(4, 8, 2), (2, 14, 2)])
def test_store_600_appends_two_compactions(vbits, hq, hkv):
    batch, T, cap, steps = 2, 256, 1024, 600
    vc = api.Codec.mse(vbits)
    store = api.TailStore(vc, batch, hkv, cap, tail_capacity=T)
    # sequence 1 starts with 64 compressed tokens (prefilled), sequence 0 empty
    pre_k = _draw((1, hkv, 64, D), 11)
    pre_v = _draw((1, hkv, 64, D), 12)
    store.k_f16[1:2, :, :64] = pre_k.to(torch.float16)
    one = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    api.quantize_mse(vc, torch.cat([torch.zeros_like(pre_v), pre_v]), store.v, count=one)
    store.comp_lens.copy_(one)
    comp, tail = [0, 64], [0, 0]
    checkpoints = {0: None, 254: None, 255: None, 300: None, 511: None, 599: None}
    plan = store.plan(hq)
    pi, _ = oracle_constants()
    cv = oracle_codebook(vbits)
    stats = CodeStats()
    new_k, new_v = [], []
    for st in range(steps):
        kn = _draw((batch, hkv, D), 1000 + st)
        vn = _draw((batch, hkv, D), 5000 + st)
        store.append(kn, vn)
        new_k.append(kn.to(torch.float16).cpu().numpy())
        new_v.append(vn.to(torch.float16).cpu().numpy())
        for b in range(batch):
            tail[b] += 1
            if tail[b] == T:
                comp[b] += T
                tail[b] = 0
        if st in checkpoints:
            q = _draw((batch, hq, D), 9000 + st)
            out = store.decode(plan, q, plan.new_out().fill_(float("nan")))
            torch.cuda.synchronize()
            assert store.comp_lens.tolist() == comp and store.tail_lens.tolist() == tail, st
            got = out.double().cpu().numpy()
            g = hq // hkv
            for b in range(batch):
                n_app = st + 1
                ks = np.stack([new_k[t][b] for t in range(n_app)], axis=1)   # [Hkv, n_app, D]
                vs = np.stack([new_v[t][b] for t in range(n_app)], axis=1)
                pre = 64 if b == 1 else 0
                for h in range(hkv):
                    keys = ks[h].astype(np.float64)
                    vals = vs[h].astype(np.float64)
                    if pre:
                        keys = np.concatenate([pre_k[0, h].to(torch.float16).double().cpu().numpy(),
                                               keys])
                        vals = np.concatenate([pre_v[0, h].float().cpu().numpy(), vals])
                    nc = comp[b]
                    gi, gx = unpack_mse(store.v, b, h, nc, vbits)
                    vcodes = match_mse_codes(vals[:nc], gi, gx, pi, cv, stats)
                    vd = {"idx": vcodes["idx"][None, None], "n": vcodes["n"][None, None]}
                    kt = keys[nc:][None, None]
                    vt = vals[nc:][None, None]
                    ref = o.decode_attention_asym(q[b:b + 1, h * g:(h + 1) * g].double().cpu().numpy(),
                                                  keys[:nc][None, None], vd, [nc], kt, vt,
                                                  [len(keys) - nc], pi, cv)[0]
                    check_heads(got[b, h * g:(h + 1) * g], ref, 1e-3,
                                f"append {st}, (b={b}, kv head={h})")
                    # the compressed keys are the FP16 tokens themselves
                    assert np.array_equal(store.k_f16[b, h, :nc].cpu().numpy().astype(np.float64),
                                          keys[:nc])
    assert B.tq_device_status() == (B.TQ_OK, 0)
    assert stats.idx_excluded < 1e-4 * stats.coords + 4, stats


def test_store_refuses_a_compaction_past_the_capacity():
    """A sequence whose tail fills when the compressed part has no room left keeps its state and
    raises TQ_FLAG_LEN_OVERFLOW; the other sequence carries on."""
    vc = api.Codec.mse(4)
    store = api.TailStore(vc, 2, 1, 256, tail_capacity=8)
    store.comp_lens.copy_(torch.tensor([252, 0], dtype=torch.int32))
    store.tail_lens.copy_(torch.tensor([7, 7], dtype=torch.int32))
    kn = _draw((2, 1, D), 1)
    store.append(kn, kn)
    st, flags = B.tq_device_status()
    assert st == B.TQ_ERR_DEVICE_STATUS and flags & B.TQ_FLAG_LEN_OVERFLOW
    assert store.comp_lens.tolist() == [252, 8] and store.tail_lens.tolist() == [7, 0]
