"""Paged caches (include/tq.h, tq_pages): a block table maps each sequence's tokens to pages of
a shared pool.  The same kernels serve both layouts and only the addresses differ, so a paged
cache must hold, token for token, the bytes of the flat cache written from the same inputs,
and a decode over it must give bit for bit the flat decode's output.  The flat layout is
checked against the oracle by test_gpu_parity.py.

Block tables here take their pages in a shuffled order from a pool with spare pages; entries
past a sequence's last page are -1, which the kernels must never read (a read would raise
TQ_FLAG_PAGE, and every test checks that the status word stays clear).
"""
import numpy as np
import pytest
import torch

from kv_cache_quantization_gb300 import _binding as B
from kv_cache_quantization_gb300 import api

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


def check_flags_clear():
    st, flags = api.device_status()
    assert st == B.TQ_OK and flags == 0, f"device status flags {flags:#x}"


def make_pages(used_tokens, page_tokens, max_pages, seed, spare=5):
    """A block table giving sequence b the pages for its first used_tokens[b] slots, drawn in
    a shuffled order from a pool with `spare` unused pages; other entries are -1."""
    need = [-(-u // page_tokens) for u in used_tokens]
    num_pages = sum(need) + spare
    order = np.random.default_rng(seed).permutation(num_pages)
    table = np.full((len(used_tokens), max_pages), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = order[k:k + n]
        k += n
    return api.Pages(torch.tensor(table, device="cuda"), page_tokens, num_pages)


def gather(pool: torch.Tensor, pages: api.Pages, token_dim: int) -> torch.Tensor:
    """The flat [batch][heads]... layout of a pool array whose dim 0 is the page and
    `token_dim` the slot in the page (negative entries read page 0; callers compare only the
    sequences' tokens)."""
    tab = pages.block_table.long().clamp(min=0)                     # [B, max_pages]
    g = pool[tab]                                                   # [B, max_pages, ...]
    td = token_dim + 1                                              # slot dim, after max_pages
    g = g.movedim(1, td - 1)                                        # max_pages beside the slots
    shape = list(g.shape)
    shape[td - 1:td + 1] = [shape[td - 1] * shape[td]]
    return g.reshape(shape)


def assert_prod_equal(flat: api.ProdCache, paged: api.ProdCache, ends):
    gi, gs = gather(paged.idx, paged.pages, 3), gather(paged.sgn, paged.pages, 2)
    gx, gr = gather(paged.xnorm, paged.pages, 2), gather(paged.rnorm, paged.pages, 2)
    for b, (lo, hi) in enumerate(ends):
        assert torch.equal(flat.idx[b, :, :, lo:hi], gi[b, :, :, lo:hi]), f"idx b={b}"
        assert torch.equal(flat.sgn[b, :, lo:hi], gs[b, :, lo:hi]), f"sgn b={b}"
        assert torch.equal(flat.xnorm[b, :, lo:hi], gx[b, :, lo:hi]), f"xnorm b={b}"
        assert torch.equal(flat.rnorm[b, :, lo:hi], gr[b, :, lo:hi]), f"rnorm b={b}"


def assert_mse_equal(flat: api.MSECache, paged: api.MSECache, ends):
    gi = gather(paged.idx, paged.pages, 2 if flat.bits == 4 else 3)
    gx = gather(paged.xnorm, paged.pages, 2)
    for b, (lo, hi) in enumerate(ends):
        if flat.bits == 4:
            assert torch.equal(flat.idx[b, :, lo:hi], gi[b, :, lo:hi]), f"nibbles b={b}"
        else:
            assert torch.equal(flat.idx[b, :, :, lo:hi], gi[b, :, :, lo:hi]), f"planes b={b}"
        assert torch.equal(flat.xnorm[b, :, lo:hi], gx[b, :, lo:hi]), f"xnorm b={b}"


def caches(batch, heads, kbits, vbits, used, page_tokens, max_pages, seed):
    pages_k = make_pages(used, page_tokens, max_pages, seed)
    pages_v = make_pages(used, page_tokens, max_pages, seed + 1)
    cap = page_tokens * max_pages
    flat = (api.ProdCache.empty(batch, heads, cap, kbits), api.MSECache.empty(batch, heads, cap, vbits))
    paged = (api.ProdCache.empty_paged(pages_k, heads, kbits),
             api.MSECache.empty_paged(pages_v, heads, vbits))
    return flat, paged, cap


# ------------------------------------------------------------------ quantisation

@pytest.mark.parametrize("dtype,tokens", [
    (torch.bfloat16, 700),   # the tensor-core quantiser
    (torch.float32, 700),    # the FFMA tile quantiser
    (torch.bfloat16, 1),     # one vector per (sequence, head): the append kernel
])
@pytest.mark.parametrize("page_tokens", [64, 192, 256])
@pytest.mark.parametrize("kbits,vbits", [(3, 2), (4, 4)])
def test_paged_quantize_equals_flat(dtype, tokens, page_tokens, kbits, vbits):
    batch, heads = 3, 4
    pos = [0, 64, 130] if tokens > 1 else [5, 700, 1023]
    count = [tokens, min(tokens, 333), tokens]
    used = [p + c for p, c in zip(pos, count)]
    max_pages = -(-1152 // page_tokens)
    (kf, vf), (kp, vp), cap = caches(batch, heads, kbits, vbits, used, page_tokens, max_pages,
                                     seed=10 * page_tokens + kbits)
    assert kf.capacity == cap == kp.capacity
    x = rand_x((batch, heads, tokens, D), 7 + tokens, dtype)
    y = rand_x((batch, heads, tokens, D), 8 + tokens, dtype)
    kc, vc = api.Codec.prod(kbits), api.Codec.mse(vbits)
    p = torch.tensor(pos, dtype=torch.int32, device="cuda")
    n = torch.tensor(count, dtype=torch.int32, device="cuda")
    for k, v in ((kf, vf), (kp, vp)):
        api.quantize_prod(kc, x, k, pos=p, count=n)
        api.quantize_mse(vc, y, v, pos=p, count=n)
    torch.cuda.synchronize()
    check_flags_clear()
    ends = list(zip(pos, used))
    assert_prod_equal(kf, kp, ends)
    assert_mse_equal(vf, vp, ends)


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("kbits,vbits,hq,hkv,batch,page_tokens", [
    (3, 2, 32, 8, 1, 256),    # the long-context shape, one run per 256-token stage
    (3, 4, 28, 4, 3, 64),     # 7-head groups, value pair table, four runs per stage
    (4, 4, 28, 4, 6, 192),    # pages that straddle the stages
    (2, 1, 16, 4, 2, 512),
])
def test_paged_decode_equals_flat(kbits, vbits, hq, hkv, batch, page_tokens):
    rng = np.random.default_rng(300 + kbits * 10 + vbits)
    lens = [int(x) for x in rng.integers(1, 3000, size=batch)]
    lens[0] = 3000
    max_pages = -(-3072 // page_tokens)
    (kf, vf), (kp, vp), cap = caches(batch, hkv, kbits, vbits, lens, page_tokens, max_pages,
                                     seed=500 + page_tokens)
    k = rand_x((batch, hkv, 3000, D), 31, torch.bfloat16)
    v = rand_x((batch, hkv, 3000, D), 32, torch.bfloat16)
    q = rand_x((batch, hq, D), 33, torch.bfloat16)
    kc, vc = api.Codec.prod(kbits), api.Codec.mse(vbits)
    lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for kk, vv in ((kf, vf), (kp, vp)):
        api.quantize_prod(kc, k, kk, count=lt)
        api.quantize_mse(vc, v, vv, count=lt)
    plan = api.DecodePlan(batch, hq, hkv, cap, max(lens), torch.bfloat16, torch.float32)
    out_f = plan.run(kc, vc, q, kf, vf, lt, plan.new_out())
    out_p = plan.run(kc, vc, q, kp, vp, lt, plan.new_out())
    torch.cuda.synchronize()
    check_flags_clear()
    assert torch.isfinite(out_f).all()
    assert torch.equal(out_f, out_p), f"max diff {(out_f - out_p).abs().max()}"


@pytest.mark.parametrize("hq,hkv,batch,page_tokens,vlayer", [
    (32, 8, 1, 256, 0),     # the appends inside the step's prologue, key and value together
    (16, 4, 40, 64, 0),     # 160 units: the appends as their own launch
    (32, 8, 1, 192, 1),     # the value codec's Π from another layer: one append CTA per vector
    (16, 4, 40, 128, 1),
])
def test_paged_step_equals_flat(hq, hkv, batch, page_tokens, vlayer):
    """Three chained decode steps (append at pos, attend pos + 1) on both layouts."""
    rng = np.random.default_rng(900 + batch)
    lens = [int(x) for x in rng.integers(1, 1500, size=batch)]
    max_pages = -(-1600 // page_tokens)
    (kf, vf), (kp, vp), cap = caches(batch, hkv, 3, 2, [x + 3 for x in lens], page_tokens,
                                     max_pages, seed=77 + batch)
    kc, vc = api.Codec.prod(3), api.Codec.mse(2, layer=vlayer)
    k = rand_x((batch, hkv, 1500, D), 41, torch.bfloat16)
    v = rand_x((batch, hkv, 1500, D), 42, torch.bfloat16)
    lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for kk, vv in ((kf, vf), (kp, vp)):
        api.quantize_prod(kc, k, kk, count=lt)
        api.quantize_mse(vc, v, vv, count=lt)
    plan = api.DecodePlan(batch, hq, hkv, cap, max(lens) + 3, torch.bfloat16, torch.float32)
    pos_f, pos_p = lt.clone(), lt.clone()
    for st in range(3):
        kn = rand_x((batch, hkv, D), 50 + st, torch.bfloat16)
        vn = rand_x((batch, hkv, D), 60 + st, torch.bfloat16)
        q = rand_x((batch, hq, D), 70 + st, torch.bfloat16)
        nf, np_ = torch.empty_like(pos_f), torch.empty_like(pos_p)
        out_f = plan.step(kc, vc, q, kn, vn, kf, vf, pos_f, plan.new_out(), lens_out=nf)
        out_p = plan.step(kc, vc, q, kn, vn, kp, vp, pos_p, plan.new_out(), lens_out=np_)
        torch.cuda.synchronize()
        assert torch.equal(out_f, out_p), f"step {st}: max diff {(out_f - out_p).abs().max()}"
        assert torch.equal(nf, np_)
        pos_f, pos_p = nf, np_
    check_flags_clear()
    ends = [(0, x + 3) for x in lens]
    assert_prod_equal(kf, kp, ends)
    assert_mse_equal(vf, vp, ends)


# ------------------------------------------------------------------ checks

def test_paged_bad_entry_is_skipped_and_flagged():
    """A table entry outside [0, num_pages) for written or attended tokens: the kernels skip
    that page and raise TQ_FLAG_PAGE; the other pages are written as usual."""
    batch, heads, P, max_pages = 2, 4, 64, 8
    used = [300, 200]
    pk = make_pages(used, P, max_pages, seed=3)
    pv = make_pages(used, P, max_pages, seed=4)
    tab = pk.block_table.clone()
    tab[1, 2] = pk.num_pages            # tokens 128..191 of sequence 1
    bad = api.Pages(tab, P, pk.num_pages)
    kp = api.ProdCache.empty_paged(bad, heads, 3)
    vp = api.MSECache.empty_paged(pv, heads, 2)
    kf = api.ProdCache.empty(batch, heads, P * max_pages, 3)
    kc, vc = api.Codec.prod(3), api.Codec.mse(2)
    x = rand_x((batch, heads, 300, D), 91, torch.bfloat16)
    n = torch.tensor(used, dtype=torch.int32, device="cuda")
    api.quantize_prod(kc, x, kp, count=n)
    api.quantize_prod(kc, x, kf, count=n)
    api.quantize_mse(vc, x, vp, count=n)
    torch.cuda.synchronize()
    st, flags = api.device_status()
    assert st == B.TQ_ERR_DEVICE_STATUS and flags == B.TQ_FLAG_PAGE
    good = api.ProdCache(kp.idx, kp.sgn, kp.xnorm, kp.rnorm, pk)   # gathers through valid pages
    assert_prod_equal(kf, good, [(0, 300), (0, 128)])
    plan = api.DecodePlan(batch, 8, heads, P * max_pages, 300, torch.bfloat16, torch.float32)
    q = rand_x((batch, 8, D), 92, torch.bfloat16)
    plan.run(kc, vc, q, kp, vp, n, plan.new_out())
    torch.cuda.synchronize()
    st, flags = api.device_status()
    assert st == B.TQ_ERR_DEVICE_STATUS and flags == B.TQ_FLAG_PAGE
    check_flags_clear()


def test_paged_argument_checks():
    """Host checks: page sizes, the capacity they imply, and the calls that take flat caches
    only."""
    kc, vc = api.Codec.prod(3), api.Codec.mse(2)
    pk = make_pages([256], 64, 4, seed=1)
    kp = api.ProdCache.empty_paged(pk, 1, 3)
    x = rand_x((1, 1, 256, D), 5, torch.bfloat16)
    s = torch.cuda.current_stream().cuda_stream
    # pages of 96 slots (not a multiple of 64), two of them: capacity 192
    bad_size = B.tq_pages(pk.block_table.data_ptr(), 2, 96, pk.num_pages)
    c = B.tq_prod_cache(kp.idx.data_ptr(), kp.sgn.data_ptr(), kp.xnorm.data_ptr(),
                        kp.rnorm.data_ptr(), B.ctypes.pointer(bad_size))
    assert B.tq_quantize_prod(kc.handle, x, B.TQ_BF16, 1, 1, 192, 256 * D, 256 * D, D, None, None,
                              c, 192, s) == B.TQ_ERR_INVALID_ARG
    # capacity other than max_pages · page_tokens
    assert B.tq_quantize_prod(kc.handle, x, B.TQ_BF16, 1, 1, 256, 256 * D, 256 * D, D, None, None,
                              kp.c(), 512, s) == B.TQ_ERR_INVALID_ARG
    q = torch.zeros(1, D, dtype=torch.float32, device="cuda")
    out = torch.empty(1, 256, dtype=torch.float32, device="cuda")
    assert B.tq_prod_scores(kc.handle, q, 1, D, kp.c(), 256, 256, out, 256, s) == \
        B.TQ_ERR_UNSUPPORTED
    # 5-bit keys decode on CUDA cores, which take flat caches only
    kc5 = api.Codec.prod(5)
    k5 = api.ProdCache.empty_paged(pk, 1, 5)
    v2 = api.MSECache.empty_paged(make_pages([256], 64, 4, seed=2), 1, 2)
    plan = api.DecodePlan(1, 2, 1, 256, 256, torch.bfloat16, torch.float32)
    lens = torch.tensor([256], dtype=torch.int32, device="cuda")
    with pytest.raises(B.TQError) as e:
        plan.run(kc5, vc, rand_x((1, 2, D), 6, torch.bfloat16), k5, v2, lens, plan.new_out())
    assert e.value.status == B.TQ_ERR_UNSUPPORTED
    check_flags_clear()


@pytest.mark.parametrize("causal", [True, False])
def test_paged_prefill_equals_flat(causal):
    """A chunk of queries per sequence (tq_prefill_attention): each query row reads its
    sequence's pages through the block table."""
    batch, nq, hq, hkv, P = 2, 5, 16, 4, 128
    hist = [300, 1000]
    used = [h + nq for h in hist]
    max_pages = -(-1088 // P)
    (kf, vf), (kp, vp), cap = caches(batch, hkv, 3, 4, used, P, max_pages, seed=880)
    kc, vc = api.Codec.prod(3), api.Codec.mse(4)
    k = rand_x((batch, hkv, max(used), D), 81, torch.bfloat16)
    v = rand_x((batch, hkv, max(used), D), 82, torch.bfloat16)
    q = rand_x((batch, nq, hq, D), 83, torch.bfloat16)
    full = torch.tensor(used, dtype=torch.int32, device="cuda")
    for kk, vv in ((kf, vf), (kp, vp)):
        api.quantize_prod(kc, k, kk, count=full)
        api.quantize_mse(vc, v, vv, count=full)
    lens = torch.tensor(hist, dtype=torch.int32, device="cuda")
    plan = api.PrefillPlan(batch, nq, hq, hkv, cap, max(used), causal=causal)
    out_f = plan.run(kc, vc, q, kf, vf, lens, plan.new_out())
    out_p = plan.run(kc, vc, q, kp, vp, lens, plan.new_out())
    torch.cuda.synchronize()
    check_flags_clear()
    assert torch.isfinite(out_f).all()
    assert torch.equal(out_f, out_p), f"max diff {(out_f - out_p).abs().max()}"
