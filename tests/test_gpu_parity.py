"""GPU parity: the CUDA library through its C ABI against the CPU oracle.

Tolerances: index and sign codes bit-exact outside the boundary exclusions (see parity.py);
scores within 1e-4·‖q‖‖k‖; attention outputs within relative L2 1e-3 (fp32 out) or 1e-2
(bf16/fp16 out).  Excluded coordinates must stay below 1e-4 of all coordinates.
"""
import math

import numpy as np
import pytest
import torch

import oracle.turboquant as o
from kv_cache_quantization_gb300 import _binding as B
from kv_cache_quantization_gb300 import api, synth
from parity import (CodeStats, check_heads, match_mse_codes, match_prod_codes,
                    oracle_codebook, oracle_constants, rel_l2, report, unpack_mse, unpack_prod)

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.load()
    yield
    torch.cuda.synchronize()


def rand_x(shape, seed, dtype, lognormal=True, device="cuda"):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(*shape, generator=g, device=device)
    if lognormal:
        sc = torch.exp(0.5 * torch.randn(shape[-1], generator=g, device=device))
        x = x * sc
    return x.to(dtype)


def out_tol(dt):
    return 1e-3 if dt == torch.float32 else 1e-2


def check_flags_clear():
    st, flags = api.device_status()
    assert st == B.TQ_OK and flags == 0, f"device status flags {flags:#x}"


# ------------------------------------------------------------------ quantisation

@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_quantize_prod_codes(bits, dtype):
    bsz, h, t = 2, 3, 333
    x = rand_x((bsz, h, t, D), 100 + bits, dtype)
    x[0, 1, 5] = 0          # zero vector
    x[1, 2, 7] *= 1e-3      # tiny vector
    kc = api.Codec.prod(bits)
    cache = api.ProdCache.empty(bsz, h, t, bits)
    api.quantize_prod(kc, x, cache)
    check_flags_clear()
    pi, s = oracle_constants()
    c = oracle_codebook(bits - 1)
    stats = CodeStats()
    for b in range(bsz):
        for hh in range(h):
            gi, gs, gx, gr = unpack_prod(cache, b, hh, t, bits - 1)
            match_prod_codes(x[b, hh].double().cpu().numpy(), gi, gs, gx, gr, pi, s, c, stats)
    assert stats.idx_excluded < 1e-4 * stats.coords + 3, stats
    assert stats.sign_excluded < 1e-4 * stats.coords + 3, stats
    # zero vector: all signs one, norms zero
    assert cache.sgn[0, 1, 5].cpu().numpy().tolist() == [255] * 16
    assert cache.xnorm[0, 1, 5].item() == 0 and cache.rnorm[0, 1, 5].item() == 0


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_quantize_mse_codes(bits, dtype):
    bsz, h, t = 2, 2, 517
    x = rand_x((bsz, h, t, D), 200 + bits, dtype)
    vc = api.Codec.mse(bits)
    cache = api.MSECache.empty(bsz, h, t, bits)
    api.quantize_mse(vc, x, cache)
    check_flags_clear()
    pi, _ = oracle_constants()
    c = oracle_codebook(bits)
    stats = CodeStats()
    for b in range(bsz):
        for hh in range(h):
            gi, gx = unpack_mse(cache, b, hh, t, bits)
            match_mse_codes(x[b, hh].double().cpu().numpy(), gi, gx, pi, c, stats)
    assert stats.idx_excluded < 1e-4 * stats.coords + 2, stats


@pytest.mark.parametrize("kind,bits", [("prod", 2), ("prod", 3), ("prod", 4), ("prod", 5),
                                       ("mse", 2), ("mse", 3), ("mse", 4)])
def test_quantize_append_path_codes(kind, bits):
    """Few vectors (one new token per sequence and head) take the one-CTA-per-vector path."""
    bsz, h, t, cap = 5, 4, 2, 64
    x = rand_x((bsz, h, t, D), 900 + bits, torch.bfloat16)
    x[1, 2, 0] = 0
    pos = torch.tensor([0, 7, 30, 62, 1], dtype=torch.int32, device="cuda")
    pi, s = oracle_constants()
    stats = CodeStats()
    if kind == "prod":
        codec = api.Codec.prod(bits)
        cache = api.ProdCache.empty(bsz, h, cap, bits)
        api.quantize_prod(codec, x, cache, pos=pos)
        c = oracle_codebook(bits - 1)
    else:
        codec = api.Codec.mse(bits)
        cache = api.MSECache.empty(bsz, h, cap, bits)
        api.quantize_mse(codec, x, cache, pos=pos)
        c = oracle_codebook(bits)
    check_flags_clear()
    for b in range(bsz):
        p0 = int(pos[b])
        for hh in range(h):
            xs = x[b, hh].double().cpu().numpy()
            if kind == "prod":
                gi, gs, gx, gr = unpack_prod(cache, b, hh, p0 + t, bits - 1)
                match_prod_codes(xs, gi[p0:], gs[p0:], gx[p0:], gr[p0:], pi, s, c, stats)
            else:
                gi, gx = unpack_mse(cache, b, hh, p0 + t, bits)
                match_mse_codes(xs, gi[p0:], gx[p0:], pi, c, stats)


def test_quantize_positions_and_counts():
    """Appends land at pos[b] + t for t < count[b]; other slots stay untouched."""
    bsz, h, t, cap = 3, 2, 5, 128
    x = rand_x((bsz, h, t, D), 7, torch.bfloat16)
    kc = api.Codec.prod(3)
    cache = api.ProdCache.empty(bsz, h, cap, 3)
    cache.xnorm.fill_(-1)
    pos = torch.tensor([0, 10, 120], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([5, 2, 0], dtype=torch.int32, device="cuda")
    api.quantize_prod(kc, x, cache, pos=pos, count=cnt)
    check_flags_clear()
    xn = cache.xnorm.cpu()
    ref = x.float().norm(dim=-1).cpu()
    assert torch.allclose(xn[0, :, :5], ref[0], rtol=1e-6)
    assert torch.allclose(xn[1, :, 10:12], ref[1, :, :2], rtol=1e-6)
    assert (xn[0, :, 5:] == -1).all() and (xn[1, :, :10] == -1).all() and (xn[1, :, 12:] == -1).all()
    assert (xn[2] == -1).all()


def test_quantize_overflow_flag():
    """A token past the capacity is skipped and raises TQ_FLAG_POS_OVERFLOW."""
    x = rand_x((1, 1, 4, D), 8, torch.bfloat16)
    kc = api.Codec.prod(3)
    cache = api.ProdCache.empty(1, 1, 64, 3)
    pos = torch.tensor([62], dtype=torch.int32, device="cuda")
    api.quantize_prod(kc, x, cache, pos=pos)
    st, flags = api.device_status()
    assert st == B.TQ_ERR_DEVICE_STATUS and flags & B.TQ_FLAG_POS_OVERFLOW
    assert cache.xnorm[0, 0, 62].item() > 0 and cache.xnorm[0, 0, 63].item() > 0
    check_flags_clear()


# ------------------------------------------------------------------ scores (1024 keys x 64 queries)

def test_scores_fp32_1k():
    w = synth.SCORES_1K
    k, _ = synth.make_kv(w, device="cuda")
    q = synth.make_queries(w, device="cuda")[0, 0]                  # [64, 128] fp32
    kc = api.Codec.prod(w.k_bits)
    cache = api.ProdCache.empty(1, 1, w.context, w.k_bits)
    api.quantize_prod(kc, k, cache)
    scores = api.prod_scores(kc, q, cache, w.context).double().cpu().numpy()
    check_flags_clear()
    pi, s = oracle_constants()
    c = oracle_codebook(w.k_bits - 1)
    stats = CodeStats()
    x = k[0, 0].double().cpu().numpy()
    gi, gs, gx, gr = unpack_prod(cache, 0, 0, w.context, w.k_bits - 1)
    codes = match_prod_codes(x, gi, gs, gx, gr, pi, s, c, stats)
    qn = q.double().cpu().numpy()
    ref = o.prod_scores(qn, codes["idx"], codes["sign"], codes["n"], codes["gamma"], pi, s, c)
    bound = 1e-4 * np.linalg.norm(qn, axis=1)[:, None] * codes["n"][None, :]
    err = np.abs(scores - ref)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3g}"
    assert stats.idx_excluded < 1e-4 * stats.coords + 2


# ------------------------------------------------------------------ decode attention

def run_decode(batch, hq, hkv, lens, kbits, vbits, in_dtype, out_dtype, seed, sample=None,
               q_dtype=None, zero_tokens=(), layer=0):
    cap = max(64, (max(lens) + 63) // 64 * 64)
    k = rand_x((batch, hkv, cap, D), seed, in_dtype)
    v = rand_x((batch, hkv, cap, D), seed + 1, in_dtype)
    for (b, h, t) in zero_tokens:
        k[b, h, t] = 0
        v[b, h, t] = 0
    q = rand_x((batch, hq, D), seed + 2, q_dtype or in_dtype)
    kc, vc = api.Codec.prod(kbits, layer), api.Codec.mse(vbits, layer)
    kcache = api.ProdCache.empty(batch, hkv, cap, kbits)
    vcache = api.MSECache.empty(batch, hkv, cap, vbits)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    api.quantize_prod(kc, k, kcache, count=lens_t)
    api.quantize_mse(vc, v, vcache, count=lens_t)
    plan = api.DecodePlan(batch, hq, hkv, cap, max(lens), q.dtype, out_dtype)
    out = plan.new_out().fill_(float("nan"))   # every output element must be written
    plan.run(kc, vc, q, kcache, vcache, lens_t, out)
    got = out.double().cpu().numpy()
    check_flags_clear()
    pi, s = oracle_constants(layer)
    ck, cv = oracle_codebook(kbits - 1), oracle_codebook(vbits)
    g = hq // hkv
    stats = CodeStats()
    worst = 0.0
    pairs = sample or [(b, h) for b in range(batch) for h in range(hkv)]
    for b, h in pairs:
        n = lens[b]
        qq = q[b, h * g:(h + 1) * g].double().cpu().numpy()[None]
        if n == 0:
            assert np.all(got[b, h * g:(h + 1) * g] == 0)
            continue
        gi, gs, gx, gr = unpack_prod(kcache, b, h, n, kbits - 1)
        kcodes = match_prod_codes(k[b, h, :n].double().cpu().numpy(), gi, gs, gx, gr, pi, s, ck, stats)
        assert not kcodes["drop"].any()
        vi, vx = unpack_mse(vcache, b, h, n, vbits)
        vcodes = match_mse_codes(v[b, h, :n].double().cpu().numpy(), vi, vx, pi, cv, stats)
        kd = {key: kcodes[key][None, None] for key in ("idx", "sign", "n", "gamma")}
        vd = {key: vcodes[key][None, None] for key in ("idx", "n")}
        ref = o.decode_attention(qq, kd, vd, [n], pi, s, ck, cv)[0]
        worst = max(worst, check_heads(got[b, h * g:(h + 1) * g], ref, out_tol(out_dtype),
                                       f"(b={b}, kv head={h})"))
    assert stats.idx_excluded < 1e-4 * max(stats.coords, 1) + 4, stats
    assert stats.sign_excluded < 1e-4 * max(stats.coords, 1) + 4, stats
    return worst


@pytest.mark.parametrize("kbits,vbits,hq", [
    (3, 4, 8), (3, 2, 8), (4, 4, 8), (2, 1, 8), (5, 3, 8),      # G = 4 (query hi/lo columns)
    (4, 2, 8), (4, 2, 14),                                      # 4-bit keys, 2-bit values
    (4, 4, 14), (3, 3, 14), (2, 2, 12), (5, 4, 14),             # G = 7, 7, 6 (one column per head)
    (4, 1, 6), (2, 3, 4)])                                      # G = 3, 2
def test_decode_small(kbits, vbits, hq):
    run_decode(2, hq, 2, [300, 1000], kbits, vbits, torch.bfloat16, torch.float32,
               300 + 10 * kbits + vbits)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_decode_out_dtypes(out_dtype):
    run_decode(1, 7, 1, [777], 3, 4, torch.bfloat16, out_dtype, 400, q_dtype=torch.float32)


def test_decode_edge_lengths():
    """Empty, single-token, exactly-one-split and capacity-filling sequences, a zero vector,
    and plain multi-head attention (G = 1)."""
    run_decode(5, 4, 4, [0, 1, 256, 257, 1024], 3, 4, torch.bfloat16, torch.float32, 500,
               zero_tokens=[(1, 0, 0), (4, 3, 100)])


def test_decode_many_ragged_units():
    """160 (batch, KV head) units, more than half the SMs: several waves of splits without
    clusters, where splits without tokens leave at once; empty and one-token sequences."""
    rng = np.random.default_rng(161)
    lens = [int(x) for x in rng.integers(0, 900, size=40)]
    lens[3] = lens[17] = 0
    lens[5] = 1
    pairs = [(b, h) for b in (0, 3, 5, 17, 22, 39) for h in range(4)]
    run_decode(40, 8, 4, lens, 3, 4, torch.bfloat16, torch.float32, 650, sample=pairs)


def test_decode_operand_two_slices_per_cta():
    """24 (batch, KV head) units: the query-operand kernel takes two slices a CTA, here with
    one operand column per head (G = 7); ragged lengths taken largest first."""
    run_decode(6, 28, 4, [0, 5, 333, 1000, 2047, 64], 3, 4, torch.bfloat16, torch.float32, 660)


def test_decode_large_batch_natural_order():
    """180 sequences × 3 splits: more work items than the split kernel ranks, so the CTAs keep
    their natural order; the operand kernel takes four slices a CTA."""
    rng = np.random.default_rng(181)
    lens = [int(x) for x in rng.integers(0, 700, size=180)]
    lens[7] = 0
    lens[11] = 700
    pairs = [(b, h) for b in (0, 7, 11, 90, 179) for h in range(2)]
    run_decode(180, 4, 2, lens, 3, 2, torch.bfloat16, torch.float32, 670, sample=pairs)


def test_decode_group_of_eight():
    run_decode(1, 16, 2, [640], 3, 4, torch.float16, torch.float32, 600)


@pytest.mark.parametrize("hq,hkv,n,vbits", [(16, 2, 20000, 4), (7, 1, 30000, 2)])
def test_decode_records_in_several_chunks(hq, hkv, n, vbits):
    """Few (batch, KV head) units and a long context: many splits per sequence (53 of 8 heads,
    118 of 7 heads), so the merging split brings the records into shared memory in several
    chunks."""
    run_decode(1, hq, hkv, [n], 3, vbits, torch.bfloat16, torch.float32, 620 + hq)


def run_workload_decode(w, pairs):
    """A decode workload at its full size, in the configuration the benchmark times (one plan
    for the whole batch, its longest sequence as the plan's maximum); the oracle checks the
    listed (batch row, KV head) pairs."""
    kc, vc = api.Codec.prod(w.k_bits), api.Codec.mse(w.v_bits)
    k, v = synth.make_kv(w, device="cuda")
    q = synth.make_queries(w, device="cuda")[:, :, 0]
    lens = [min(int(x), w.context) for x in synth.seq_lengths(w)]
    kcache = api.ProdCache.empty(w.batch, w.kv_heads, w.context, w.k_bits)
    vcache = api.MSECache.empty(w.batch, w.kv_heads, w.context, w.v_bits)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    api.quantize_prod(kc, k, kcache, count=lens_t)
    api.quantize_mse(vc, v, vcache, count=lens_t)
    plan = api.DecodePlan(w.batch, w.q_heads, w.kv_heads, w.context, max(lens), q.dtype, w.out_dtype)
    out = plan.new_out().fill_(float("nan"))
    out = plan.run(kc, vc, q, kcache, vcache, lens_t, out).double().cpu().numpy()
    check_flags_clear()
    assert not np.isnan(out).any()
    pi, s = oracle_constants()
    ck, cv = oracle_codebook(w.k_bits - 1), oracle_codebook(w.v_bits)
    g = w.group
    stats = CodeStats()
    for b, h in pairs:
        n = lens[b]
        gi, gs, gx, gr = unpack_prod(kcache, b, h, n, w.k_bits - 1)
        kcodes = match_prod_codes(k[b, h, :n].double().cpu().numpy(), gi, gs, gx, gr, pi, s, ck, stats)
        vi, vx = unpack_mse(vcache, b, h, n, w.v_bits)
        vcodes = match_mse_codes(v[b, h, :n].double().cpu().numpy(), vi, vx, pi, cv, stats)
        kd = {key: kcodes[key][None, None] for key in ("idx", "sign", "n", "gamma")}
        vd = {key: vcodes[key][None, None] for key in ("idx", "n")}
        ref = o.decode_attention(q[b:b + 1, h * g:(h + 1) * g].double().cpu().numpy(), kd, vd, [n],
                                 pi, s, ck, cv)[0]
        check_heads(out[b, h * g:(h + 1) * g], ref, out_tol(w.out_dtype), f"(b={b}, kv head={h})")
    report(w.name, stats, f"pairs={len(pairs)}")
    assert stats.idx_excluded < 1e-4 * stats.coords, stats
    assert stats.sign_excluded < 1e-4 * stats.coords, stats


def test_decode_qwen7b_32k():
    """One decode step, B=1, 28/4 heads, 32768 tokens, K 3-bit prod, V 4-bit MSE, bf16."""
    run_workload_decode(synth.DECODE_32K, [(0, h) for h in range(4)])


def test_decode_longctx_262k():
    """B=1, 32/8 heads, 262144 tokens, K 3-bit prod (4 outlier channels), V 2-bit MSE: two of
    the eight KV heads checked against the oracle."""
    run_workload_decode(synth.LONG_262K, [(0, 0), (0, 5)])


def test_decode_serving_ragged_b32():
    """B=32 ragged 4096–16384 tokens, 28/4 heads, K 4-bit prod, V 4-bit MSE: the longest and
    the shortest sequences and two others checked against the oracle."""
    w = synth.SERVE_B32
    lens = [int(x) for x in synth.seq_lengths(w)]
    order = np.argsort(lens)
    pairs = [(int(order[-1]), 0), (int(order[0]), 3), (int(order[len(order) // 2]), 1), (7, 2)]
    run_workload_decode(w, pairs)


# ------------------------------------------------------------------ asymmetric mode

def run_asym(batch, hq, hkv, lens, tlens, vbits, out_dtype, seed, tail_cap=256, sample=None,
             tensors=None, name=None):
    """Asymmetric decode against the oracle.  tensors = (k fp16, v, k_tail fp16, v_tail fp16,
    q) of a workload recipe, or None for test-local draws."""
    cap = max(64, (max(lens) + 63) // 64 * 64)
    if tensors is None:
        k = rand_x((batch, hkv, cap, D), seed, torch.bfloat16).to(torch.float16)
        v = rand_x((batch, hkv, cap, D), seed + 1, torch.bfloat16)
        kt = rand_x((batch, hkv, tail_cap, D), seed + 2, torch.bfloat16).to(torch.float16)
        vt = rand_x((batch, hkv, tail_cap, D), seed + 3, torch.bfloat16).to(torch.float16)
        q = rand_x((batch, hq, D), seed + 4, torch.bfloat16)
    else:
        k, v, kt, vt, q = tensors
        cap = k.shape[2]
    vc = api.Codec.mse(vbits)
    vcache = api.MSECache.empty(batch, hkv, cap, vbits)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    tl_t = torch.tensor(tlens, dtype=torch.int32, device="cuda")
    api.quantize_mse(vc, v, vcache, count=lens_t)
    plan = api.DecodePlan(batch, hq, hkv, cap, max(lens), q.dtype, out_dtype, tail_capacity=tail_cap)
    out = plan.run_asym(vc, q, k, vcache, lens_t, kt, vt, tl_t, plan.new_out().fill_(float("nan")))
    got = out.double().cpu().numpy()
    check_flags_clear()
    assert not np.isnan(got).any()
    pi, _ = oracle_constants()
    cv = oracle_codebook(vbits)
    g = hq // hkv
    stats = CodeStats()
    for b, h in (sample or [(b, h) for b in range(batch) for h in range(hkv)]):
        n, tl = lens[b], tlens[b]
        vi, vx = unpack_mse(vcache, b, h, n, vbits)
        vcodes = match_mse_codes(v[b, h, :n].double().cpu().numpy(), vi, vx, pi, cv, stats)
        vd = {key: vcodes[key][None, None] for key in ("idx", "n")}
        ref = o.decode_attention_asym(q[b:b + 1, h * g:(h + 1) * g].double().cpu().numpy(),
                                      k[b:b + 1, h:h + 1, :n].double().cpu().numpy(), vd, [n],
                                      kt[b:b + 1, h:h + 1].double().cpu().numpy(),
                                      vt[b:b + 1, h:h + 1].double().cpu().numpy(), [tl], pi, cv)[0]
        if n + tl == 0:
            assert np.all(got[b, h * g:(h + 1) * g] == 0)
            continue
        check_heads(got[b, h * g:(h + 1) * g], ref, out_tol(out_dtype), f"(b={b}, kv head={h})")
    if name:
        report(name, stats, f"pairs={len(sample or [])}")
    assert stats.idx_excluded < 1e-4 * max(stats.coords, 1) + 4, stats


def test_asym_small():
    run_asym(3, 8, 2, [100, 0, 700], [255, 17, 0], 4, torch.float32, 700)


@pytest.mark.parametrize("vbits,hq,hkv", [(2, 8, 2), (3, 14, 2), (1, 16, 2), (4, 14, 2)])
def test_asym_value_bits_and_groups(vbits, hq, hkv):
    """Value codes as planes (1–3 bits) and the pair table (4 bits), G = 4 (fp16 weight pairs)
    and G = 7, 8 (one column per head); ragged compressed lengths across tile boundaries and
    tails of 0, 1 and 128 tokens."""
    run_asym(3, hq, hkv, [383, 129, 1000], [0, 1, 128], vbits, torch.float32, 710 + vbits)


def test_asym_b8_8k():
    """B=8, 28/4 heads, the workload's own inputs: 7937 FP16-key / 4-bit-value tokens and the
    last 255 tokens held as the FP16 tail, bf16 out; 8 of the 32 (batch, KV head) pairs checked
    against the oracle, every query head on its own."""
    w = synth.ASYM_8K
    lens = [int(x) for x in synth.seq_lengths(w)]
    k, v = synth.make_kv(w, device="cuda")
    kt, vt = synth.asym_tail(w, k, v)
    q = synth.make_queries(w, device="cuda")[:, :, 0]
    pairs = [(0, 0), (1, 3), (2, 1), (3, 2), (4, 0), (5, 3), (6, 2), (7, 1)]
    run_asym(w.batch, w.q_heads, w.kv_heads, lens, [w.tail] * w.batch, w.v_bits, w.out_dtype, 0,
             sample=pairs, tensors=(k.to(torch.float16), v, kt, vt, q), name=w.name)


# ------------------------------------------------------------------ workspace reuse

def test_workspace_reuse_across_descriptors():
    """One workspace serves a larger symmetric call, an asymmetric call and a smaller call in
    turn (each leaves its own data where the next keeps its split tickets); the smaller call's
    output is bit for bit that of a fresh workspace."""
    def case(batch, hq, hkv, n, seed):
        k = rand_x((batch, hkv, n, D), seed, torch.bfloat16)
        v = rand_x((batch, hkv, n, D), seed + 1, torch.bfloat16)
        q = rand_x((batch, hq, D), seed + 2, torch.bfloat16)
        kc, vc = api.Codec.prod(3), api.Codec.mse(4)
        kcache = api.ProdCache.empty(batch, hkv, n, 3)
        vcache = api.MSECache.empty(batch, hkv, n, 4)
        api.quantize_prod(kc, k, kcache)
        api.quantize_mse(vc, v, vcache)
        lens = torch.full((batch,), n, dtype=torch.int32, device="cuda")
        return kc, vc, q, kcache, vcache, lens, k, v
    big = case(16, 28, 4, 2048, 950)
    small = case(2, 14, 2, 1500, 960)
    big_plan = api.DecodePlan(16, 28, 4, 2048, 2048, torch.bfloat16, torch.float32)
    asym_plan = api.DecodePlan(16, 28, 4, 2048, 2048, torch.bfloat16, torch.float32,
                               tail_capacity=256)
    n = max(big_plan.workspace.numel(), asym_plan.workspace.numel())
    ws = torch.empty(n, dtype=torch.uint8, device="cuda").fill_(0xA5)
    big_plan.workspace = ws
    asym_plan.workspace = ws
    big_plan.run(*big[:6], big_plan.new_out())
    tl = torch.full((16,), 200, dtype=torch.int32, device="cuda")
    kt = big[6][:, :, :256].to(torch.float16).contiguous()
    vt = big[7][:, :, :256].to(torch.float16).contiguous()
    asym_plan.run_asym(big[1], big[2], big[6].to(torch.float16), big[4], big[5], kt, vt, tl,
                       asym_plan.new_out())
    fresh = api.DecodePlan(2, 14, 2, 1500, 1500, torch.bfloat16, torch.float32)
    ref = fresh.run(*small[:6], fresh.new_out())
    out = torch.full(fresh.shape, float("nan"), device="cuda")
    kc, vc, q, kcache, vcache, lens = small[:6]
    B.check(B.tq_decode_attention(fresh.desc, kc.handle, vc.handle, q, kcache.c(), vcache.c(),
                                  lens, out, ws, ws.numel(), torch.cuda.current_stream().cuda_stream),
            "tq_decode_attention")
    torch.cuda.synchronize()
    check_flags_clear()
    assert torch.equal(out, ref)


# ------------------------------------------------------------------ serving loop

def test_decode_serving_loop():
    """The ragged serving batch (B=32, 4096–16384 tokens, 28/4 heads, K 4-bit prod, V 4-bit
    MSE) for its 128 decode steps: every step (tq_decode_step) appends one new key and value
    per (sequence, KV head) at position len, attends the grown cache and returns len + 1.  The oracle replays the appends and checks four
    (sequence, KV head) pairs at steps 0, 1, 64 and 127, every query head on its own."""
    w = synth.SERVE_B32
    steps = w.decode_steps
    lens0 = [int(x) for x in synth.seq_lengths(w)]
    cap = synth.cache_capacity(w)
    kc, vc = api.Codec.prod(w.k_bits), api.Codec.mse(w.v_bits)
    k, v = synth.make_kv(w, device="cuda")
    kcache = api.ProdCache.empty(w.batch, w.kv_heads, cap, w.k_bits)
    vcache = api.MSECache.empty(w.batch, w.kv_heads, cap, w.v_bits)
    lens_t = torch.tensor(lens0, dtype=torch.int32, device="cuda")
    api.quantize_prod(kc, k, kcache, count=lens_t)
    api.quantize_mse(vc, v, vcache, count=lens_t)
    plan = api.DecodePlan(w.batch, w.q_heads, w.kv_heads, cap, max(lens0) + steps, w.in_dtype,
                          w.out_dtype)
    order = np.argsort(lens0)
    pairs = [(int(order[-1]), 0), (int(order[0]), 3), (int(order[len(order) // 2]), 1), (7, 2)]
    checkpoints = (0, 1, 64, steps - 1)
    new_kv, queries, outs = [], {}, {}
    lens_next = torch.empty_like(lens_t)
    for st in range(steps):
        kn, vn = synth.make_new_tokens(w, device="cuda", step=st)
        q = synth.make_queries(w, device="cuda", step=st)[:, :, 0]
        # one call: append at lens, attend lens + 1 tokens, lens + 1 written to lens_next
        out = plan.step(kc, vc, q, kn[:, :, 0].contiguous(), vn[:, :, 0].contiguous(), kcache,
                        vcache, lens_t, plan.new_out().fill_(float("nan")), lens_out=lens_next)
        lens_t, lens_next = lens_next, lens_t
        new_kv.append((kn[:, :, 0].double().cpu().numpy(), vn[:, :, 0].double().cpu().numpy()))
        if st in checkpoints:
            outs[st] = out.double().cpu().numpy()
            queries[st] = q.double().cpu().numpy()
    torch.cuda.synchronize()
    check_flags_clear()
    pi, s = oracle_constants(w.layer)
    ck, cv = oracle_codebook(w.k_bits - 1), oracle_codebook(w.v_bits)
    g = w.group
    stats = CodeStats()
    for b, h in pairs:
        n0 = lens0[b]
        n = n0 + steps
        xk = np.concatenate([k[b, h, :n0].double().cpu().numpy(),
                             np.stack([new_kv[t][0][b, h] for t in range(steps)])])
        xv = np.concatenate([v[b, h, :n0].double().cpu().numpy(),
                             np.stack([new_kv[t][1][b, h] for t in range(steps)])])
        gi, gs, gx, gr = unpack_prod(kcache, b, h, n, w.k_bits - 1)
        kcodes = match_prod_codes(xk, gi, gs, gx, gr, pi, s, ck, stats)
        assert not kcodes["drop"].any()
        vi, vx = unpack_mse(vcache, b, h, n, w.v_bits)
        vcodes = match_mse_codes(xv, vi, vx, pi, cv, stats)
        for st in checkpoints:
            m = n0 + st + 1
            kd = {key: kcodes[key][None, None, :m] for key in ("idx", "sign", "n", "gamma")}
            vd = {key: vcodes[key][None, None, :m] for key in ("idx", "n")}
            ref = o.decode_attention(queries[st][b:b + 1, h * g:(h + 1) * g], kd, vd, [m], pi, s,
                                     ck, cv)[0]
            check_heads(outs[st][b, h * g:(h + 1) * g], ref, out_tol(w.out_dtype),
                        f"step {st}, (b={b}, kv head={h})")
    report(w.name + " (128-step loop)", stats, f"pairs={len(pairs)}")
    assert stats.idx_excluded < 1e-4 * stats.coords, stats
    assert stats.sign_excluded < 1e-4 * stats.coords, stats


@pytest.mark.parametrize("kbits,vbits,hq,hkv,batch,vlayer", [
    (3, 2, 32, 8, 1, 0),     # the long-context shape (4-head groups, value planes)
    (3, 4, 28, 4, 3, 0),     # the 32K shape (7-head groups, value pair table)
    (4, 4, 28, 4, 6, 0),     # the serving shape (3-bit key indices)
    (5, 3, 8, 2, 2, 0),      # 4-bit key indices: the CUDA-core path
    (3, 2, 16, 4, 40, 0),    # 160 units: the appends as their own launch before the operand kernel
    (3, 2, 32, 8, 1, 1),     # the value codec's Π from another layer: one append CTA per vector
    (3, 4, 16, 4, 40, 1),    # the same in the appends' own launch (keys first, then values)
    (5, 3, 8, 2, 2, 1),
])
def test_decode_step_equals_separate_calls(kbits, vbits, hq, hkv, batch, vlayer):
    """tq_decode_step gives bit for bit the caches and outputs of tq_quantize_prod +
    tq_quantize_mse (one token at pos) + tq_decode_attention over pos + 1 tokens, over three
    chained steps (lens_out feeding the next step), with ragged lengths.  With the two codecs
    sharing Π (vlayer 0) the step quantises each key and value together in one CTA; with
    another Π for the values (vlayer 1) it appends them separately."""
    rng = np.random.default_rng(1700 + kbits * 10 + vbits)
    lens = [int(x) for x in rng.integers(1, 1500, size=batch)]
    cap = 1600
    kc, vc = api.Codec.prod(kbits), api.Codec.mse(vbits, layer=vlayer)
    k = rand_x((batch, hkv, cap, D), 1701, torch.bfloat16)
    v = rand_x((batch, hkv, cap, D), 1702, torch.bfloat16)
    caches = []
    for _ in range(2):
        kcache = api.ProdCache.empty(batch, hkv, cap, kbits)
        vcache = api.MSECache.empty(batch, hkv, cap, vbits)
        lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
        api.quantize_prod(kc, k, kcache, count=lt)
        api.quantize_mse(vc, v, vcache, count=lt)
        caches.append((kcache, vcache))
    plan = api.DecodePlan(batch, hq, hkv, cap, max(lens) + 3, torch.bfloat16, torch.float32)
    pos_a = torch.tensor(lens, dtype=torch.int32, device="cuda")
    pos_b = pos_a.clone()
    nxt = torch.empty_like(pos_a)
    for st in range(3):
        kn = rand_x((batch, hkv, D), 1710 + st, torch.bfloat16)
        vn = rand_x((batch, hkv, D), 1720 + st, torch.bfloat16)
        q = rand_x((batch, hq, D), 1730 + st, torch.bfloat16)
        out_a = plan.step(kc, vc, q, kn, vn, *caches[0], pos_a, plan.new_out(), lens_out=nxt)
        pos_a, nxt = nxt, pos_a
        api.quantize_prod(kc, kn[:, :, None], caches[1][0], pos=pos_b)
        api.quantize_mse(vc, vn[:, :, None], caches[1][1], pos=pos_b)
        pos_b = pos_b + 1
        out_b = plan.run(kc, vc, q, *caches[1], pos_b, plan.new_out())
        torch.cuda.synchronize()
        assert torch.equal(pos_a, pos_b)
        assert torch.equal(out_a, out_b), f"step {st}: max diff {(out_a - out_b).abs().max()}"
    check_flags_clear()
    for ta, tb in zip((caches[0][0].idx, caches[0][0].sgn, caches[0][0].xnorm, caches[0][0].rnorm,
                       caches[0][1].idx, caches[0][1].xnorm),
                      (caches[1][0].idx, caches[1][0].sgn, caches[1][0].xnorm, caches[1][0].rnorm,
                       caches[1][1].idx, caches[1][1].xnorm)):
        assert torch.equal(ta, tb)


# ------------------------------------------------------------------ quality report

@pytest.mark.parametrize("bits", [3, 4])
def test_attention_quality_report(bits):
    """KL divergence and top-1 positions of attention on compressed keys against exact keys
    (tq_attention_quality) match the oracle on the 1024-key workload's inputs: KL within
    2e-5 + 1e-3·KL, top-1 equal unless the oracle's two best scores are within rounding."""
    w = synth.SCORES_1K
    k, _ = synth.make_kv(w, device="cuda")
    q = synth.make_queries(w, device="cuda")[0, 0]
    kc = api.Codec.prod(bits)
    cache = api.ProdCache.empty(1, 1, w.context, bits)
    api.quantize_prod(kc, k, cache)
    kl, te, tc = api.attention_quality(kc, q, k[0, 0], cache, w.context)
    kl, te, tc = kl.double().cpu().numpy(), te.cpu().numpy(), tc.cpu().numpy()
    check_flags_clear()
    pi, s = oracle_constants()
    c = oracle_codebook(bits - 1)
    gi, gs, gx, gr = unpack_prod(cache, 0, 0, w.context, bits - 1)
    x = k[0, 0].double().cpu().numpy()
    codes = match_prod_codes(x, gi, gs, gx, gr, pi, s, c, CodeStats())
    qn = q.double().cpu().numpy()
    rkl, rte, rtc = o.attention_quality(qn, x, codes["idx"], codes["sign"], codes["n"],
                                        codes["gamma"], pi, s, c)
    assert np.all(np.abs(kl - rkl) <= 2e-5 + 1e-3 * rkl), np.max(np.abs(kl - rkl))
    exact = qn @ x.T
    comp = o.prod_scores(qn, codes["idx"], codes["sign"], codes["n"], codes["gamma"], pi, s, c)
    tol = 1e-4 * np.linalg.norm(qn, axis=1) * np.max(np.linalg.norm(x, axis=1))
    for i in range(len(qn)):
        assert te[i] == rte[i] or exact[i, te[i]] >= exact[i, rte[i]] - tol[i]
        assert tc[i] == rtc[i] or comp[i, tc[i]] >= comp[i, rtc[i]] - tol[i]
    # more key bits, closer attention
    assert rkl.mean() > 0


@pytest.mark.parametrize("layer", [1, 5])
def test_decode_other_layers(layer):
    """Codecs of other layers (rotation seed 42 + 7ℓ, sketch seed 43 + 7ℓ: independent Π and S
    per layer, QJL deep-dive §六): quantisation and decode attention match the oracle built from
    the same layer's constants."""
    run_decode(2, 8, 2, [500, 1200], 3, 4, torch.bfloat16, torch.float32, 1900 + layer,
               layer=layer)


def test_layers_have_independent_constants():
    """Different layers get different rotations: the codes of one input differ between layer 0
    and layer 1 codecs."""
    x = rand_x((1, 1, 64, D), 1950, torch.bfloat16)
    caches = []
    for layer in (0, 1):
        kc = api.Codec.prod(3, layer)
        cache = api.ProdCache.empty(1, 1, 64, 3)
        api.quantize_prod(kc, x, cache)
        caches.append(cache)
    torch.cuda.synchronize()
    assert not torch.equal(caches[0].idx, caches[1].idx)
    torch.testing.assert_close(caches[0].xnorm, caches[1].xnorm, rtol=1e-6, atol=0)


# ------------------------------------------------------------------ prefill chunks

@pytest.mark.parametrize("causal,kbits,vbits,hq,hkv,nq", [
    (True, 3, 4, 8, 2, 5), (False, 3, 2, 14, 2, 3), (True, 4, 4, 28, 4, 16)])
def test_prefill_attention(causal, kbits, vbits, hq, hkv, nq):
    """A chunk of nq queries per sequence over the compressed cache (tq_prefill_attention): with
    causal, query i attends the history and the chunk's first i + 1 tokens; without, the
    history only.  Every query head of every row against the oracle."""
    batch, hist = 2, [300, 1000]
    cap = 1088
    kc, vc = api.Codec.prod(kbits), api.Codec.mse(vbits)
    k = rand_x((batch, hkv, cap, D), 2100 + nq, torch.bfloat16)
    v = rand_x((batch, hkv, cap, D), 2200 + nq, torch.bfloat16)
    q = rand_x((batch, nq, hq, D), 2300 + nq, torch.bfloat16)
    kcache = api.ProdCache.empty(batch, hkv, cap, kbits)
    vcache = api.MSECache.empty(batch, hkv, cap, vbits)
    full = torch.tensor([h + nq for h in hist], dtype=torch.int32, device="cuda")
    api.quantize_prod(kc, k, kcache, count=full)
    api.quantize_mse(vc, v, vcache, count=full)
    lens = torch.tensor(hist, dtype=torch.int32, device="cuda")
    plan = api.PrefillPlan(batch, nq, hq, hkv, cap, max(hist) + nq, causal=causal)
    out = plan.run(kc, vc, q, kcache, vcache, lens, plan.new_out().fill_(float("nan")))
    got = out.double().cpu().numpy()
    check_flags_clear()
    pi, s = oracle_constants()
    ck, cv = oracle_codebook(kbits - 1), oracle_codebook(vbits)
    g = hq // hkv
    stats = CodeStats()
    for b in range(batch):
        n_all = hist[b] + nq
        for h in range(hkv):
            gi, gs, gx, gr = unpack_prod(kcache, b, h, n_all, kbits - 1)
            kcodes = match_prod_codes(k[b, h, :n_all].double().cpu().numpy(), gi, gs, gx, gr, pi,
                                      s, ck, stats)
            vi, vx = unpack_mse(vcache, b, h, n_all, vbits)
            vcodes = match_mse_codes(v[b, h, :n_all].double().cpu().numpy(), vi, vx, pi, cv, stats)
            for i in range(nq):
                n = hist[b] + (i + 1 if causal else 0)
                kd = {key: kcodes[key][None, None, :n] for key in ("idx", "sign", "n", "gamma")}
                vd = {key: vcodes[key][None, None, :n] for key in ("idx", "n")}
                ref = o.decode_attention(q[b:b + 1, i, h * g:(h + 1) * g].double().cpu().numpy(),
                                         kd, vd, [n], pi, s, ck, cv)[0]
                check_heads(got[b, i, h * g:(h + 1) * g], ref, 1e-3,
                            f"(b={b}, query {i}, kv head={h})")
    assert stats.idx_excluded < 1e-4 * stats.coords + 4, stats
