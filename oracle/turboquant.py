"""CPU oracle for TurboQuant KV-cache compression and compressed-domain decode attention.

TEST INFRASTRUCTURE ONLY.  This module is a plain, slow, float64 NumPy restatement of what
the GPU library computes.  Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  It shares no
code, tables or constants with the CUDA library and never imports it.

Sources (cited by page title and section):

* [QJL] "TurboQuant QJL投影深度剖析：揭秘注意力分数背后的无偏内积估计器原理" (bjdmk.com.cn)
  - §二 step 1: store ||x||, rotate x/||x|| by a random orthogonal Π obtained by QR.
  - §二 step 2: Lloyd-Max (continuous 1-D k-means) codebook for the rotated-coordinate law,
    per-coordinate decision-boundary lookup.
  - §二 step 3: residual r = x - x̃ projected by a Gaussian S, keep sign bits (d/8 bytes)
    and ||r||.
  - §四: E[<g, sign(g r)>]-type identity; the constant √(π/2)/d.
  - §五: estimator <y, x̃_mse> + ||r||·√(π/2)/d·<Sᵀ signs, y>, unbiased; quantize() returns
    (MSE indices, QJL sign bytes, residual norm, original norm), all bit-packed.
  - §六: read path rotates the query forward (q Πᵀ) and pre-sketches it (q Sᵀ).
* [MLX] MLX-port article (cf-1.com), "背景": keys use the full two-stage quantiser
  (Algorithm 2), values the MSE-only quantiser (Algorithm 1); "对称 vs 非对称":
  asymmetric mode keeps K in FP16 and quantises V only, and compression is judged by the KL
  divergence and top-1 agreement of the distributions with and without it.

Readings where the pages are silent:

* index = number of decision boundaries <= y (a tie goes to the upper cell);
* sign bit = 1 iff (S r)_j >= 0, so a zero residual stores all ones;
* a zero vector stores ||x|| = 0, every index in the upper middle cell, ||r|| = 0;
* norms are float32 on the device, float64 here;
* index codes are bit planes (LSB-first coordinates), except 4-bit MSE codes which are
  nibble-packed (coordinate 2k in the low nibble of byte k).

Parity pins: every function here is pinned by the tests in ``tests/test_oracle_pins.py``
(closed forms, Monte-Carlo unbiasedness, brute force, printed page values).  No function
is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np
from scipy import special

QJL_SCALE_NUMERATOR = math.sqrt(math.pi / 2.0)  # the √(π/2) of [QJL] §四/§五


# ---------------------------------------------------------------------------------------
# Codebook: Lloyd-Max on the rotated-coordinate law            [QJL] §二 step 2
# ---------------------------------------------------------------------------------------

def coordinate_density(t, d: int):
    """Density of one coordinate of a uniform point on S^{d-1}:
    f(t) = Γ(d/2) / (√π Γ((d-1)/2)) · (1 - t²)^((d-3)/2) on [-1, 1]   ([QJL] §二 step 1,
    "scaled Beta law")."""
    t = np.asarray(t, dtype=np.float64)
    logc = special.gammaln(d / 2.0) - 0.5 * math.log(math.pi) - special.gammaln((d - 1) / 2.0)
    out = np.zeros_like(t)
    inside = np.abs(t) < 1.0
    out[inside] = np.exp(logc + (d - 3) / 2.0 * np.log1p(-t[inside] ** 2))
    return out


def coordinate_cdf(t, d: int):
    """P(T <= t).  T² ~ Beta(1/2, (d-1)/2), so F(t) = 1/2 + sign(t)/2 · I_{t²}(1/2, (d-1)/2)."""
    t = np.clip(np.asarray(t, dtype=np.float64), -1.0, 1.0)
    return 0.5 + 0.5 * np.sign(t) * special.betainc(0.5, (d - 1) / 2.0, t * t)


def coordinate_first_moment(a, b, d: int):
    """∫_a^b t f(t) dt = C_d [-(1-t²)^((d-1)/2) / (d-1)]_a^b  (f as in coordinate_density)."""
    logc = special.gammaln(d / 2.0) - 0.5 * math.log(math.pi) - special.gammaln((d - 1) / 2.0)
    c = math.exp(logc)

    def prim(t):
        t = np.clip(np.asarray(t, dtype=np.float64), -1.0, 1.0)
        return -c * np.power(1.0 - t * t, (d - 1) / 2.0) / (d - 1)

    return prim(b) - prim(a)


def lloyd_max_codebook(d: int, bits: int, tol: float = 1e-15, max_iter: int = 200000):
    """Optimal scalar quantiser for the coordinate law by Lloyd's iteration ([QJL] §二 step 2:
    "continuous 1-D k-means").  Alternates (1) decision boundaries = midpoints of adjacent
    centroids and (2) centroid = conditional mean of the cell, until the centroids move by
    less than ``tol``.  Returns (centroids ascending, boundaries ascending), float64,
    unit-sphere scale."""
    levels = 1 << bits
    c = np.linspace(-2.5, 2.5, levels) / math.sqrt(d)
    for _ in range(max_iter):
        bnd = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate(([-1.0], bnd, [1.0]))
        mass = np.diff(coordinate_cdf(edges, d))
        moment = coordinate_first_moment(edges[:-1], edges[1:], d)
        new = moment / mass
        moved = np.max(np.abs(new - c))
        c = new
        if moved < tol:
            break
    # The coordinate law is symmetric and the start is symmetric, so the fixed point is
    # too; remove the last-ulp asymmetry so that the middle boundary is exactly 0.
    c = 0.5 * (c - c[::-1])
    bnd = 0.5 * (c[:-1] + c[1:])
    return c, bnd


def codebook_mse(centroids, d: int):
    """Per-coordinate distortion E[(T - c[idx(T)])²] of the codebook under the coordinate law."""
    c = np.asarray(centroids, dtype=np.float64)
    bnd = 0.5 * (c[:-1] + c[1:])
    edges = np.concatenate(([-1.0], bnd, [1.0]))
    # E[T²] over each cell minus 2 c E[T] + c² P: use E[T²] = 1/d overall.
    mass = np.diff(coordinate_cdf(edges, d))
    moment = coordinate_first_moment(edges[:-1], edges[1:], d)
    return 1.0 / d - np.sum(2.0 * c * moment - c * c * mass)


# ---------------------------------------------------------------------------------------
# Rotation Π from a Gaussian matrix                              [QJL] §二 step 1
# ---------------------------------------------------------------------------------------

def rotation_from_gaussian(g):
    """Π = Q of the QR factorisation G = Q R, with column signs fixed so that diag(R) > 0
    (which makes Π a deterministic function of G).  y = Π x rotates a column vector."""
    g = np.asarray(g, dtype=np.float64)
    q, r = np.linalg.qr(g)
    s = np.sign(np.diag(r))
    s[s == 0] = 1.0
    return q * s[None, :]


# ---------------------------------------------------------------------------------------
# Quantisers                                                      [QJL] §二, §五
# ---------------------------------------------------------------------------------------

def quantize_mse(x, pi, centroids):
    """TurboQuant-MSE (Algorithm 1): n = ||x||; y = Π x / n; idx_j = #{boundaries <= y_j},
    everything in float64.  (A float32 implementation may pick the neighbouring cell only
    where y_j lies within float32 rounding of a boundary, far inside the 1e-6 band that
    ``boundary_exclusion`` marks.)
    Returns (idx int64 [..., d], n float64 [...], y float64 [..., d])."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(centroids, dtype=np.float64)
    bnd = 0.5 * (c[:-1] + c[1:])
    n = np.sqrt(np.sum(x * x, axis=-1))
    safe = np.where(n > 0, n, 1.0)
    u = x / safe[..., None]
    u = np.where((n > 0)[..., None], u, 0.0)
    y = u @ np.asarray(pi, dtype=np.float64).T
    idx = np.searchsorted(bnd, y, side="right")
    return idx.astype(np.int64), n, y


def prod_residual(x, n, idx, pi, s, centroids):
    """Second stage of TurboQuant-prod for given MSE indices ([QJL] §二 step 3):
    x̃ = n Πᵀ c[idx], r = x - x̃, γ = ||r||, z = S r, sign_j = [z_j >= 0].
    Returns (sign bool [..., d], gamma [...], z [..., d])."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(centroids, dtype=np.float64)
    x_tilde = np.asarray(n, dtype=np.float64)[..., None] * (c[idx] @ np.asarray(pi, dtype=np.float64))
    r = x - x_tilde
    gamma = np.sqrt(np.sum(r * r, axis=-1))
    z = r @ np.asarray(s, dtype=np.float64).T
    return z >= 0.0, gamma, z


def quantize_prod(x, pi, s, centroids):
    """TurboQuant-prod (Algorithm 2) with a (b-1)-bit codebook ``centroids``: the MSE stage
    followed by the 1-bit QJL sketch of the residual ([QJL] §二, §五).  Returns a dict with
    idx, sign (bool), n, gamma and the decision quantities y (unit-sphere rotated
    coordinates) and z = S r."""
    idx, n, y = quantize_mse(x, pi, centroids)
    sign, gamma, z = prod_residual(x, n, idx, pi, s, centroids)
    return {"idx": idx, "sign": sign, "n": n, "gamma": gamma, "y": y, "z": z}


def dequantize_mse(idx, n, pi, centroids):
    """v̂ = n Πᵀ c[idx]."""
    c = np.asarray(centroids, dtype=np.float64)
    return np.asarray(n, dtype=np.float64)[..., None] * (c[idx] @ np.asarray(pi, dtype=np.float64))


def dequantize_prod(idx, sign, n, gamma, pi, s, centroids):
    """k̂ = n Πᵀ c[idx] + γ·√(π/2)/d · Sᵀ (2·sign - 1): the vector whose inner product with
    any y equals the [QJL] §五 estimator (an independent second path to the same number)."""
    d = np.asarray(pi).shape[0]
    pm = 2.0 * np.asarray(sign, dtype=np.float64) - 1.0
    qjl = (QJL_SCALE_NUMERATOR / d) * np.asarray(gamma, dtype=np.float64)[..., None] * (
        pm @ np.asarray(s, dtype=np.float64))
    return dequantize_mse(idx, n, pi, centroids) + qjl


def prod_scores(q, idx, sign, n, gamma, pi, s, centroids):
    """Estimator of <q, k> for every (query, key) pair ([QJL] §五, §六):
    score = n·<Π q, c[idx]> + γ·√(π/2)/d·<S q, 2·sign - 1>.
    q: [nq, d]; codes: [nk, d]; returns [nq, nk]."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    c = np.asarray(centroids, dtype=np.float64)
    q_rot = q @ np.asarray(pi, dtype=np.float64).T  # Π q as rows  (q Πᵀ)
    q_sk = q @ np.asarray(s, dtype=np.float64).T    # S q as rows  (q Sᵀ)
    pm = 2.0 * np.asarray(sign, dtype=np.float64) - 1.0
    mse = (q_rot @ c[idx].T) * np.asarray(n, dtype=np.float64)[None, :]
    qjl = (q_sk @ pm.T) * ((QJL_SCALE_NUMERATOR / d) * np.asarray(gamma, dtype=np.float64))[None, :]
    return mse + qjl


# ---------------------------------------------------------------------------------------
# Attention                                                       [QJL] §六
# ---------------------------------------------------------------------------------------

def softmax_attention(q, keys, values, scale):
    """Exact single-query attention: softmax(scale · keys q) · values, dense, float64.
    q: [d]; keys, values: [n, d].  An empty key set returns zeros."""
    if keys.shape[0] == 0:
        return np.zeros(values.shape[-1], dtype=np.float64)
    logits = scale * (np.asarray(keys, dtype=np.float64) @ np.asarray(q, dtype=np.float64))
    w = np.exp(logits - np.max(logits))
    w /= np.sum(w)
    return w @ np.asarray(values, dtype=np.float64)


def decode_attention(q, k_codes, v_codes, seq_lens, pi, s, k_centroids, v_centroids, scale=None):
    """Decode attention on the compressed cache: for batch b and query head h (KV head
    h // G), logits = scale·estimator(q, k_t) over t < seq_lens[b], weights softmax, output
    Σ_t w_t v̂_t.  q: [B, Hq, d].  k_codes: dict(idx [B,Hkv,T,d], sign, n, gamma);
    v_codes: dict(idx [B,Hkv,T,d], n).  Returns float64 [B, Hq, d]."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    hkv = k_codes["idx"].shape[1]
    g = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((bsz, hq, d))
    for b in range(bsz):
        ln = int(seq_lens[b])
        for kh in range(hkv):
            sl = (b, kh, slice(0, ln))
            k_hat = dequantize_prod(k_codes["idx"][sl], k_codes["sign"][sl], k_codes["n"][sl],
                                    k_codes["gamma"][sl], pi, s, k_centroids)
            v_hat = dequantize_mse(v_codes["idx"][sl], v_codes["n"][sl], pi, v_centroids)
            for j in range(g):
                h = kh * g + j
                out[b, h] = softmax_attention(q[b, h], k_hat, v_hat, scale)
    return out


def decode_attention_asym(q, k_plain, v_codes, seq_lens, k_tail, v_tail, tail_lens, pi,
                          v_centroids, scale=None):
    """Asymmetric mode ([MLX] "对称 vs 非对称": K in FP16, V quantised): one softmax over the
    compressed segment (FP16 keys k_plain[:, :, :seq_len], MSE-coded values) and the FP16
    tail segment (k_tail/v_tail[:, :, :tail_len]).  Returns float64 [B, Hq, d]."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    hkv = k_plain.shape[1]
    g = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((bsz, hq, d))
    for b in range(bsz):
        ln, tl = int(seq_lens[b]), int(tail_lens[b])
        for kh in range(hkv):
            v_hat = dequantize_mse(v_codes["idx"][b, kh, :ln], v_codes["n"][b, kh, :ln], pi,
                                   v_centroids)
            keys = np.concatenate([np.asarray(k_plain[b, kh, :ln], dtype=np.float64),
                                   np.asarray(k_tail[b, kh, :tl], dtype=np.float64)])
            vals = np.concatenate([v_hat, np.asarray(v_tail[b, kh, :tl], dtype=np.float64)])
            for j in range(g):
                h = kh * g + j
                out[b, h] = softmax_attention(q[b, h], keys, vals, scale)
    return out


# ---------------------------------------------------------------------------------------
# Quality of compressed attention        [MLX] "对称 vs 非对称": KL divergence and top-1
# ---------------------------------------------------------------------------------------

def softmax_kl(a, b):
    """KL(softmax(a) ‖ softmax(b)) along the last axis: Σ_t p_t (log p_t − log q_t) with
    log p = a − log Σ e^a and log q = b − log Σ e^b."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    la = a - special.logsumexp(a, axis=-1, keepdims=True)
    lb = b - special.logsumexp(b, axis=-1, keepdims=True)
    return np.sum(np.exp(la) * (la - lb), axis=-1)


def attention_quality(q, keys, idx, sign, n, gamma, pi, s, centroids, scale=None):
    """Attention-level counterpart of the pages' KLD / top-1 comparison: for each query q_i,
    the attention weights over exact keys, softmax(scale·⟨q_i, k_t⟩), against those over the
    estimator scores of the compressed keys ([QJL] §五).  Returns (KL(exact ‖ compressed),
    argmax over exact, argmax over compressed) per query."""
    q = np.asarray(q, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    exact = scale * (q @ np.asarray(keys, dtype=np.float64).T)
    comp = scale * prod_scores(q, idx, sign, n, gamma, pi, s, centroids)
    return softmax_kl(exact, comp), np.argmax(exact, axis=-1), np.argmax(comp, axis=-1)


# ---------------------------------------------------------------------------------------
# Bit packing ([QJL] §二 step 3: d sign bits in d/8 bytes; §五: everything bit-packed)
# ---------------------------------------------------------------------------------------

def pack_bits(bits):
    """bool/int [..., d] -> uint8 [..., d/8]; coordinate j at byte j // 8, bit j % 8."""
    bits = np.asarray(bits).astype(np.uint8) & 1
    d = bits.shape[-1]
    b = bits.reshape(bits.shape[:-1] + (d // 8, 8))
    weights = (1 << np.arange(8)).astype(np.uint16)
    return (b.astype(np.uint16) * weights).sum(axis=-1).astype(np.uint8)


def unpack_bits(packed, d: int):
    """Inverse of pack_bits."""
    packed = np.asarray(packed, dtype=np.uint8)
    shifts = np.arange(8, dtype=np.uint8)
    bits = (packed[..., :, None] >> shifts) & 1
    return bits.reshape(packed.shape[:-1] + (d,)).astype(np.uint8)


def pack_index_planes(idx, bits: int):
    """int [..., d] -> uint8 [..., bits, d/8]; plane p holds bit p of every index."""
    idx = np.asarray(idx, dtype=np.int64)
    planes = [pack_bits((idx >> p) & 1) for p in range(bits)]
    return np.stack(planes, axis=-2)


def unpack_index_planes(packed, d: int):
    packed = np.asarray(packed, dtype=np.uint8)
    bits = packed.shape[-2]
    idx = np.zeros(packed.shape[:-2] + (d,), dtype=np.int64)
    for p in range(bits):
        idx |= unpack_bits(packed[..., p, :], d).astype(np.int64) << p
    return idx


def pack_nibbles(idx):
    """int [..., d] (values < 16) -> uint8 [..., d/2]; byte k = idx[2k] | idx[2k+1] << 4."""
    idx = np.asarray(idx, dtype=np.int64)
    lo = idx[..., 0::2]
    hi = idx[..., 1::2]
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_nibbles(packed, d: int):
    packed = np.asarray(packed, dtype=np.int64)
    out = np.zeros(packed.shape[:-1] + (d,), dtype=np.int64)
    out[..., 0::2] = packed & 15
    out[..., 1::2] = packed >> 4
    return out


def pack_mse_codes(idx, bits: int):
    """Packed MSE code bytes of one vector: nibbles for 4-bit codes, bit planes otherwise
    (flattened to [..., bits*d/8])."""
    if bits == 4:
        return pack_nibbles(idx)
    p = pack_index_planes(idx, bits)
    return p.reshape(p.shape[:-2] + (-1,))


# ---------------------------------------------------------------------------------------
# Parity exclusions (decision quantities close to a decision boundary)
# ---------------------------------------------------------------------------------------

def boundary_exclusion(y, centroids, eps=1e-6):
    """For each rotated coordinate: (excluded, alternative index).  A coordinate is excluded
    when it lies within eps of a decision boundary (unit-sphere units), where a float32
    evaluation may legitimately pick the neighbouring cell; the alternative is that
    neighbouring cell (the other side of the nearest boundary)."""
    c = np.asarray(centroids, dtype=np.float64)
    bnd = 0.5 * (c[:-1] + c[1:])
    y = np.asarray(y, dtype=np.float64)
    dist = np.abs(y[..., None] - bnd)
    k = np.argmin(dist, axis=-1)            # nearest boundary separates cells k and k+1
    excluded = np.take_along_axis(dist, k[..., None], axis=-1)[..., 0] < eps
    idx = np.searchsorted(bnd, y, side="right")
    alt = np.where(idx == k, k + 1, k)
    return excluded, alt.astype(np.int64)


def sign_exclusion(z, n, d, eps=1e-6):
    """True where a QJL sign bit lies within eps of its decision boundary.  The sign decides
    on z_j = (S r)_j.  Measured in the same unit-sphere units as the index band, the decision
    quantity is the projection of the unit-sphere residual r/||x|| onto the unit direction of
    row j of S, i.e. z_j / (||x||·||S_j||), and E||S_j||² = d for a Gaussian S.  So a bit is
    excluded when |z_j| < eps·√d·||x||.  For a Gaussian S independent of x, z_j ~ N(0, ||r||²)
    and the excluded share of a vector's bits is erf(eps·√d·||x|| / (√2·||r||))."""
    z = np.asarray(z, dtype=np.float64)
    n = np.asarray(n, dtype=np.float64)[..., None]
    return np.abs(z) < eps * math.sqrt(d) * n
