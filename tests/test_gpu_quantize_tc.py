"""GPU parity of the tensor-core quantiser (tiles of bf16 / fp16 vectors) against the oracle.

The tensor-core kernel takes every bf16 / fp16 call with more vectors than two per SM; the
basic code checks live in test_gpu_parity.py.  This file covers what is specific to it:
placement (pos / count) and the overflow flag on the tiled path, inputs whose magnitudes
stress the per-vector power-of-two scaling, and the full-size compaction workloads
(262144-token long context; 32 ragged sequences of 4096..16384 tokens), checked on sampled
vectors that the oracle recomputes one by one.
"""
import numpy as np
import pytest
import torch

from kv_cache_quantization_gb300 import _binding as B
from kv_cache_quantization_gb300 import api, synth
from parity import (CodeStats, match_mse_codes, match_prod_codes, oracle_codebook,
                    oracle_constants, unpack_mse, unpack_mse_at, unpack_prod, unpack_prod_at)

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.load()
    yield
    torch.cuda.synchronize()


def rand_x(shape, seed, dtype):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(*shape, generator=g, device="cuda")
    x = x * torch.exp(0.5 * torch.randn(shape[-1], generator=g, device="cuda"))
    return x.to(dtype)


def flags_clear():
    st, flags = api.device_status()
    assert st == B.TQ_OK and flags == 0, f"device status flags {flags:#x}"


def test_tiled_positions_and_counts():
    """Tiled path: vector t of sequence b lands at pos[b] + t when t < count[b]."""
    bsz, h, t, cap = 3, 4, 300, 704
    x = rand_x((bsz, h, t, D), 31, torch.bfloat16)
    kc = api.Codec.prod(3)
    cache = api.ProdCache.empty(bsz, h, cap, 3)
    cache.xnorm.fill_(-1)
    pos = torch.tensor([0, 100, 400], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([300, 17, 0], dtype=torch.int32, device="cuda")
    api.quantize_prod(kc, x, cache, pos=pos, count=cnt)
    flags_clear()
    xn = cache.xnorm.cpu()
    ref = x.float().norm(dim=-1).cpu()
    assert torch.allclose(xn[0, :, :300], ref[0], rtol=1e-6)
    assert (xn[0, :, 300:] == -1).all()
    assert torch.allclose(xn[1, :, 100:117], ref[1, :, :17], rtol=1e-6)
    assert (xn[1, :, :100] == -1).all() and (xn[1, :, 117:] == -1).all()
    assert (xn[2] == -1).all()
    pi, s = oracle_constants()
    c = oracle_codebook(2)
    stats = CodeStats()
    for hh in range(h):
        gi, gs, gx, gr = unpack_prod_at(cache, 1, hh, range(100, 117), 2)
        match_prod_codes(x[1, hh, :17].double().cpu().numpy(), gi, gs, gx, gr, pi, s, c, stats)


@pytest.mark.parametrize("layout", ["token-major", "short-rows"])
def test_tiled_copy_paths_with_counts(layout):
    """The tile copies take three paths: one copy per run of a long sequence, one per run
    starting at each vector of sequences shorter than 32 tokens, and one per vector when the
    token stride is not one vector ([batch, tokens, heads, 128] storage seen as [batch, heads,
    tokens, 128]).  Each is run with per-sequence counts that leave whole tiles empty; every
    stored slot's norm and a sample of its codes match the oracle, and untouched slots stay."""
    if layout == "token-major":
        bsz, h, t = 2, 4, 700
        base = rand_x((bsz, t, h, D), 41, torch.bfloat16)
        x = base.transpose(1, 2)                       # token stride = h vectors
        assert x.stride(2) == h * D
        counts = [700, 333]
    else:
        bsz, h, t = 8, 16, 20
        x = rand_x((bsz, h, t, D), 42, torch.bfloat16)
        counts = [20, 0, 7, 19, 1, 20, 13, 0]
    cnt = torch.tensor(counts, dtype=torch.int32, device="cuda")
    cap = (t + 63) // 64 * 64
    pi, s = oracle_constants()
    for kind in ("prod", "mse"):
        if kind == "prod":
            codec = api.Codec.prod(3)
            cache = api.ProdCache.empty(bsz, h, cap, 3)
            cache.xnorm.fill_(-1)
            api.quantize_prod(codec, x, cache, count=cnt)
        else:
            codec = api.Codec.mse(2)
            cache = api.MSECache.empty(bsz, h, cap, 2)
            cache.xnorm.fill_(-1)
            api.quantize_mse(codec, x, cache, count=cnt)
        flags_clear()
        xn = cache.xnorm.cpu()
        ref = x.float().norm(dim=-1).cpu()
        stats = CodeStats()
        c = oracle_codebook(2)
        for b in range(bsz):
            n = counts[b]
            assert torch.allclose(xn[b, :, :n], ref[b, :, :n], rtol=2e-6), (kind, b)
            assert (xn[b, :, n:] == -1).all(), (kind, b)
            if n == 0:
                continue
            for hh in (0, h - 1):
                toks = range(0, n, max(1, n // 12))
                xs = x[b, hh, list(toks)].double().cpu().numpy()
                if kind == "prod":
                    gi, gs, gx, gr = unpack_prod_at(cache, b, hh, toks, 2)
                    match_prod_codes(xs, gi, gs, gx, gr, pi, s, c, stats)
                else:
                    gi, gx = unpack_mse_at(cache, b, hh, toks, 2)
                    match_mse_codes(xs, gi, gx, pi, c, stats)
        assert stats.idx_excluded < 1e-4 * stats.coords + 3, stats


def test_tiled_overflow_flag():
    """Tiled path: tokens past the capacity are skipped and raise TQ_FLAG_POS_OVERFLOW."""
    x = rand_x((1, 4, 400, D), 32, torch.bfloat16)
    vc = api.Codec.mse(4)
    cache = api.MSECache.empty(1, 4, 448, 4)
    pos = torch.tensor([100], dtype=torch.int32, device="cuda")
    api.quantize_mse(vc, x, cache, pos=pos)
    st, flags = api.device_status()
    assert st == B.TQ_ERR_DEVICE_STATUS and flags & B.TQ_FLAG_POS_OVERFLOW
    assert (cache.xnorm[0, :, 100:448] > 0).all()
    flags_clear()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_magnitudes(dtype):
    """Vectors of very different magnitudes (each is rescaled by its own power of two)."""
    x = rand_x((1, 2, 320, D), 33, torch.float32)
    if dtype == torch.bfloat16:
        scales = [1e15, 1e-15, 2.0 ** -100, 1e30, 1.0]
    else:
        scales = [1e2, 1e-3, 2.0 ** -10, 1.0, 0.25]
    for i, sc in enumerate(scales):
        x[0, :, 40 * i:40 * (i + 1)] *= sc
    x[0, 1, 300] = 0
    x[0, 0, 301, :] = 0
    x[0, 0, 301, 17] = 3.0            # a single nonzero coordinate
    x = x.to(dtype)
    pi, s = oracle_constants()
    for bits in (2, 3, 4):
        kc = api.Codec.prod(bits)
        cache = api.ProdCache.empty(1, 2, 320, bits)
        api.quantize_prod(kc, x, cache)
        flags_clear()
        c = oracle_codebook(bits - 1)
        stats = CodeStats()
        for hh in range(2):
            gi, gs, gx, gr = unpack_prod(cache, 0, hh, 320, bits - 1)
            match_prod_codes(x[0, hh].double().cpu().numpy(), gi, gs, gx, gr, pi, s, c, stats)
        assert stats.idx_excluded < 1e-4 * stats.coords + 3, stats


def _sample(rng, lens, hkv, n):
    """n (b, h, t) triples with t < lens[b]."""
    b = rng.integers(0, len(lens), n)
    h = rng.integers(0, hkv, n)
    t = (rng.random(n) * np.asarray(lens)[b]).astype(np.int64)
    return b, h, t


def _check_sampled(w, k, v, kcache, vcache, lens, rng, n):
    pi, s = oracle_constants()
    ck, cv = oracle_codebook(w.k_bits - 1), oracle_codebook(w.v_bits)
    bs, hs, ts = _sample(rng, lens, w.kv_heads, n)
    stats = CodeStats()
    for b in np.unique(bs):
        for h in np.unique(hs[bs == b]):
            tt = np.sort(ts[(bs == b) & (hs == h)])
            gi, gs, gx, gr = unpack_prod_at(kcache, int(b), int(h), tt, w.k_bits - 1)
            xk = k[int(b), int(h)][torch.as_tensor(tt, device=k.device)].double().cpu().numpy()
            match_prod_codes(xk, gi, gs, gx, gr, pi, s, ck, stats)
            vi, vx = unpack_mse_at(vcache, int(b), int(h), tt, w.v_bits)
            xv = v[int(b), int(h)][torch.as_tensor(tt, device=v.device)].double().cpu().numpy()
            match_mse_codes(xv, vi, vx, pi, cv, stats)
    assert stats.idx_excluded < 1e-4 * stats.coords + 3, stats
    assert stats.sign_excluded < 1e-4 * stats.coords + 3, stats
    return stats


def test_compaction_longctx_262k_sampled():
    """Full-cache compaction of the 262144-token long-context layer (8 KV heads, keys with
    outlier channels): 2,097,152 keys and as many values in one call each."""
    w = synth.LONG_262K
    k, v = synth.make_kv(w, device="cuda")
    kc, vc = api.Codec.prod(w.k_bits), api.Codec.mse(w.v_bits)
    kcache = api.ProdCache.empty(w.batch, w.kv_heads, w.context, w.k_bits)
    vcache = api.MSECache.empty(w.batch, w.kv_heads, w.context, w.v_bits)
    api.quantize_prod(kc, k, kcache)
    api.quantize_mse(vc, v, vcache)
    flags_clear()
    # every token of every head was written: norms are positive
    assert (kcache.xnorm > 0).all() and (vcache.xnorm > 0).all() and (kcache.rnorm > 0).all()
    rng = np.random.default_rng(262144)
    lens = synth.seq_lengths(w)
    _check_sampled(w, k, v, kcache, vcache, lens, rng, 1536)
    # the last tile of the last head
    n = w.context
    gi, gs, gx, gr = unpack_prod_at(kcache, 0, w.kv_heads - 1, range(n - 200, n), w.k_bits - 1)
    pi, s = oracle_constants()
    match_prod_codes(k[0, -1, n - 200:].double().cpu().numpy(), gi, gs, gx, gr, pi, s,
                     oracle_codebook(w.k_bits - 1), CodeStats())


def test_compaction_serving_ragged_sampled():
    """Prefill compaction of 32 ragged sequences (4096..16384 tokens, 4 KV heads): every
    sequence passes its length as count; slots beyond it stay untouched."""
    w = synth.SERVE_B32
    k, v = synth.make_kv(w, device="cuda")
    lens = synth.seq_lengths(w)
    cnt = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kc, vc = api.Codec.prod(w.k_bits), api.Codec.mse(w.v_bits)
    kcache = api.ProdCache.empty(w.batch, w.kv_heads, w.context, w.k_bits)
    vcache = api.MSECache.empty(w.batch, w.kv_heads, w.context, w.v_bits)
    kcache.xnorm.fill_(-1)
    vcache.xnorm.fill_(-1)
    api.quantize_prod(kc, k, kcache, count=cnt)
    api.quantize_mse(vc, v, vcache, count=cnt)
    flags_clear()
    tok = torch.arange(w.context, device="cuda")[None, None, :]
    live = tok < cnt[:, None, None]
    assert (kcache.xnorm[live.expand_as(kcache.xnorm)] > 0).all()
    assert (kcache.xnorm[~live.expand_as(kcache.xnorm)] == -1).all()
    assert (vcache.xnorm[~live.expand_as(vcache.xnorm)] == -1).all()
    rng = np.random.default_rng(16384)
    _check_sampled(w, k, v, kcache, vcache, lens, rng, 1536)
