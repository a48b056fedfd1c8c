"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each ``pin_*`` takes the oracle namespace ``o`` as an argument so that
``test_oracle_planted.py`` can run the same pins on a copy of the oracle with one mistake
planted and require that some pin fails.  None of these checks retypes the oracle's own
formula: each compares against a closed form, an independent quadrature, a printed value,
a brute-force loop or a Monte-Carlo expectation.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy import integrate

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rotation(o, seed, d=128):
    return o.rotation_from_gaussian(np.random.default_rng(seed).standard_normal((d, d)))


def _sketch(seed, d=128):
    return np.random.default_rng(seed).standard_normal((d, d))


# --------------------------------------------------------------------------- rotation

def pin_rotation(o):
    """Π orthogonal, det ±1, and Πᵀ G upper triangular with a positive diagonal (so Π is the
    sign-fixed Q of G = Q R, QJL deep-dive §二 step 1)."""
    g = np.random.default_rng(42).standard_normal((128, 128))
    pi = o.rotation_from_gaussian(g)
    assert np.max(np.abs(pi.T @ pi - np.eye(128))) < 1e-12
    assert abs(abs(np.linalg.det(pi)) - 1.0) < 1e-9
    r = pi.T @ g
    assert np.max(np.abs(np.tril(r, -1))) < 1e-10
    assert np.all(np.diag(r) > 0)


# --------------------------------------------------------------------------- codebook

def _density_indep(t, d):
    # written independently of the oracle: normalised (1 - t^2)^((d-3)/2)
    logc = math.lgamma(d / 2) - 0.5 * math.log(math.pi) - math.lgamma((d - 1) / 2)
    return math.exp(logc) * (1 - t * t) ** ((d - 3) / 2) if abs(t) < 1 else 0.0


def pin_codebook_closed_form_1bit(o):
    """B = 1: the optimal levels are ±E|T| = ±Γ(d/2)/(√π Γ((d+1)/2))."""
    for d in (16, 128, 1000):
        c, b = o.lloyd_max_codebook(d, 1)
        e_abs = math.exp(math.lgamma(d / 2) - 0.5 * math.log(math.pi) - math.lgamma((d + 1) / 2))
        assert abs(c[1] - e_abs) < 1e-13 and abs(c[0] + e_abs) < 1e-13
        assert b[0] == 0.0


def pin_codebook_centroid_condition(o):
    """Each level is the conditional mean of its cell and each boundary the midpoint of its
    neighbours (Lloyd-Max optimality), checked with adaptive quadrature of an independently
    written density."""
    d = 128
    for bits in (2, 3, 4):
        c, b = o.lloyd_max_codebook(d, bits)
        assert np.all(np.diff(c) > 0)
        np.testing.assert_allclose(b, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-15)
        np.testing.assert_allclose(c, -c[::-1], rtol=0, atol=1e-15)
        edges = [-1.0] + list(b) + [1.0]
        for k in range(len(c)):
            lo, hi = edges[k], edges[k + 1]
            m0 = integrate.quad(lambda t: _density_indep(t, d), lo, hi, epsabs=1e-14,
                                epsrel=1e-13, limit=200)[0]
            m1 = integrate.quad(lambda t: t * _density_indep(t, d), lo, hi, epsabs=1e-14,
                                epsrel=1e-13, limit=200)[0]
            assert abs(m1 / m0 - c[k]) < 1e-9 * max(1.0, abs(c[k])), (bits, k)


def pin_codebook_gaussian_limit(o):
    """For large d the scaled levels approach the classical Gaussian Lloyd-Max table."""
    ref = golden("gaussian_lloyd_max.json")
    d = 1 << 16
    for bits in (1, 2, 3, 4):
        c, _ = o.lloyd_max_codebook(d, bits, tol=1e-12)
        pos = c[len(c) // 2:] * math.sqrt(d)
        np.testing.assert_allclose(pos, ref["levels_positive"][str(bits)], rtol=0, atol=2e-4)
        mse = o.codebook_mse(c, d) * d
        assert abs(mse - ref["mse"][str(bits)]) < 2e-4 * max(1.0, ref["mse"][str(bits)] * 10)


def pin_codebook_mse_monotone(o):
    d = 128
    m = [o.codebook_mse(o.lloyd_max_codebook(d, b)[0], d) for b in (1, 2, 3, 4)]
    assert all(m[i] > m[i + 1] > 0 for i in range(3))


# --------------------------------------------------------------------------- quantisers

def pin_mse_index_is_nearest_level(o):
    """Midpoint boundaries make the boundary count equal to the nearest level: brute force
    over all levels, away from ties."""
    rng = np.random.default_rng(7)
    pi = _rotation(o, 42)
    for bits in (1, 2, 3, 4):
        c, b = o.lloyd_max_codebook(128, bits)
        x = rng.standard_normal((200, 128)) * np.exp(0.5 * rng.standard_normal(128))
        idx, n, y = o.quantize_mse(x, pi, c)
        np.testing.assert_allclose(n, np.linalg.norm(x, axis=1), rtol=1e-14)
        # y is the rotated unit vector: Πᵀ y n reproduces x
        np.testing.assert_allclose((y @ pi) * n[:, None], x, rtol=0, atol=1e-11)
        brute = np.argmin(np.abs(y[..., None] - c[None, None, :]), axis=-1)
        excl, _ = o.boundary_exclusion(y, c)
        assert np.array_equal(idx[~excl], brute[~excl])


def pin_mse_distortion(o):
    """E||v - v̂||² / ||v||² over random directions equals d times the codebook's per-coordinate
    distortion (rotation invariance + the quantiser of QJL deep-dive §二)."""
    rng = np.random.default_rng(11)
    pi = _rotation(o, 42)
    for bits in (2, 4):
        c, _ = o.lloyd_max_codebook(128, bits)
        v = rng.standard_normal((4000, 128))
        idx, n, _ = o.quantize_mse(v, pi, c)
        vh = o.dequantize_mse(idx, n, pi, c)
        rel = np.sum((v - vh) ** 2, axis=1) / np.sum(v * v, axis=1)
        expect = 128 * o.codebook_mse(c, 128)
        assert abs(rel.mean() - expect) < 4 * rel.std() / math.sqrt(len(rel)) + 1e-12


def pin_value_cos_sim_pages(o):
    """QJL deep-dive §七: value reconstruction cos_sim ≈ 0.94 at 2 bits, 0.997 at 4 bits.
    Gaussian vectors give 0.940 and 0.995; the 4-bit page figure (likely on model
    activations) is held as a lower bound."""
    ref = golden("pages_constants.json")
    rng = np.random.default_rng(3)
    pi = _rotation(o, 42)
    v = rng.standard_normal((3000, 128))
    cos = {}
    for bits in (2, 4):
        c, _ = o.lloyd_max_codebook(128, bits)
        idx, n, _ = o.quantize_mse(v, pi, c)
        vh = o.dequantize_mse(idx, n, pi, c)
        cos[bits] = np.mean(np.sum(v * vh, 1) / np.linalg.norm(v, axis=1) / np.linalg.norm(vh, axis=1))
    assert abs(cos[2] - ref["value_cos_sim_2bit"]["value"]) < 0.005
    assert cos[4] > 0.994 and cos[4] < ref["value_cos_sim_4bit"]["value"] + 0.002


def pin_qjl_identity(o):
    """QJL deep-dive §四: for Gaussian S, E[√(π/2)/d <S q, sign(S r)>] = <q, r>/||r||.
    Monte-Carlo over independent sketches, within 4 standard errors."""
    rng = np.random.default_rng(5)
    d = 128
    q = rng.standard_normal(d)
    r = rng.standard_normal(d)
    truth = q @ r / np.linalg.norm(r)
    vals = []
    for m in range(3000):
        s = rng.standard_normal((d, d))
        vals.append(math.sqrt(math.pi / 2) / d * ((s @ q) @ np.where(s @ r >= 0, 1.0, -1.0)))
    vals = np.array(vals)
    # the oracle's constant must be the one used here
    assert abs(o.QJL_SCALE_NUMERATOR - math.sqrt(math.pi / 2)) < 1e-15
    assert abs(vals.mean() - truth) < 4 * vals.std() / math.sqrt(len(vals))


def pin_estimator_unbiased(o):
    """QJL deep-dive §五: E_S[estimate] = <q, x> for fixed x, q, Π: Monte-Carlo over sketch
    seeds (and a second run over rotation seeds), within 4 standard errors."""
    rng = np.random.default_rng(9)
    d = 128
    x = rng.standard_normal(d) * np.exp(0.5 * rng.standard_normal(d))
    q = rng.standard_normal(d) * np.exp(0.5 * rng.standard_normal(d))
    truth = q @ x
    for bits in (2, 3):
        c, _ = o.lloyd_max_codebook(d, bits - 1)
        for vary_pi in (False, True):
            est = []
            for m in range(600):
                pi = _rotation(o, 1000 + m if vary_pi else 42)
                s = _sketch(50000 + m)
                k = o.quantize_prod(x[None], pi, s, c)
                est.append(o.prod_scores(q[None], k["idx"], k["sign"], k["n"], k["gamma"], pi,
                                         s, c)[0, 0])
            est = np.array(est)
            assert abs(est.mean() - truth) < 4 * est.std() / math.sqrt(len(est)), (bits, vary_pi)


def pin_estimator_equals_dequantized_dot(o):
    """The estimator equals <q, k̂> for the dequantised k̂ (an independent path), 1e-12."""
    rng = np.random.default_rng(13)
    pi = _rotation(o, 42)
    s = _sketch(43)
    c, _ = o.lloyd_max_codebook(128, 2)
    x = rng.standard_normal((50, 128))
    q = rng.standard_normal((7, 128))
    k = o.quantize_prod(x, pi, s, c)
    sc = o.prod_scores(q, k["idx"], k["sign"], k["n"], k["gamma"], pi, s, c)
    kh = o.dequantize_prod(k["idx"], k["sign"], k["n"], k["gamma"], pi, s, c)
    np.testing.assert_allclose(sc, q @ kh.T, rtol=1e-12, atol=1e-10)


def pin_residual_definition(o):
    """γ = ||x - x̃_mse|| and the signs are those of S (x - x̃_mse), with x̃_mse the MSE
    dequantisation (QJL deep-dive §二 step 3)."""
    rng = np.random.default_rng(17)
    pi = _rotation(o, 42)
    s = _sketch(43)
    c, _ = o.lloyd_max_codebook(128, 3)
    x = rng.standard_normal((40, 128)) * 3.0
    k = o.quantize_prod(x, pi, s, c)
    xt = o.dequantize_mse(k["idx"], k["n"], pi, c)
    r = x - xt
    np.testing.assert_allclose(k["gamma"], np.linalg.norm(r, axis=1), rtol=1e-12)
    assert np.array_equal(k["sign"], (s @ r.T).T >= 0)


def pin_zero_vector(o):
    """A zero vector: ||x|| = 0, indices in the upper middle cell, ||r|| = 0, all signs 1."""
    pi = _rotation(o, 42)
    s = _sketch(43)
    c, _ = o.lloyd_max_codebook(128, 2)
    k = o.quantize_prod(np.zeros((1, 128)), pi, s, c)
    assert k["n"][0] == 0 and k["gamma"][0] == 0
    assert np.all(k["idx"] == len(c) // 2)
    assert np.all(k["sign"])


# --------------------------------------------------------------------------- packing

def pin_packing_golden(o):
    g = golden("packing_example.json")
    j = np.arange(128)
    planes = o.pack_index_planes(j % 4, 2)
    assert planes.shape == (2, 16)
    assert np.all(planes[0] == g["planes_2bit"]["plane0_byte"])
    assert np.all(planes[1] == g["planes_2bit"]["plane1_byte"])
    sign = (j % 8 == 0) | (j == 127)
    assert list(o.pack_bits(sign)) == g["sign_bytes"]
    nib = o.pack_nibbles(j % 16)
    assert list(nib[:8]) == g["nibble_bytes_first8"] and list(nib[8:16]) == g["nibble_bytes_first8"]
    assert o.pack_bits(np.ones(128)).nbytes == golden("pages_constants.json")[
        "sign_bytes_per_vector_d128"]["value"]
    rng = np.random.default_rng(0)
    for bits in (1, 2, 3, 4):
        idx = rng.integers(0, 1 << bits, size=(5, 128))
        assert np.array_equal(o.unpack_index_planes(o.pack_index_planes(idx, bits), 128), idx)
    idx = rng.integers(0, 16, size=(5, 128))
    assert np.array_equal(o.unpack_nibbles(o.pack_nibbles(idx), 128), idx)


# --------------------------------------------------------------------------- attention

def _brute_attention(q, keys, vals, scale):
    """Pure-Python loops: softmax(scale * <q, k_t>) weighted sum of values."""
    n = len(keys)
    if n == 0:
        return [0.0] * len(q)
    logits = [scale * sum(qi * ki for qi, ki in zip(q, keys[t])) for t in range(n)]
    mx = max(logits)
    w = [math.exp(l - mx) for l in logits]
    tot = sum(w)
    return [sum(w[t] * vals[t][j] for t in range(n)) / tot for j in range(len(q))]


def pin_attention_brute_force(o):
    """decode_attention (estimator keys, MSE values, GQA head mapping h -> h // G) against
    a pure-Python loop over dequantised keys/values, tiny sizes, ragged lengths 0..7."""
    rng = np.random.default_rng(21)
    d = 128
    pi = _rotation(o, 42)
    s = _sketch(43)
    kc, _ = o.lloyd_max_codebook(d, 2)
    vc, _ = o.lloyd_max_codebook(d, 2)
    bsz, hkv, g, t = 3, 2, 3, 7
    lens = [7, 0, 3]
    x_k = rng.standard_normal((bsz, hkv, t, d))
    x_v = rng.standard_normal((bsz, hkv, t, d))
    q = rng.standard_normal((bsz, hkv * g, d))
    kq = o.quantize_prod(x_k, pi, s, kc)
    vi, vn, _ = o.quantize_mse(x_v, pi, vc)
    out = o.decode_attention(q, kq, {"idx": vi, "n": vn}, lens, pi, s, kc, vc)
    scale = 1 / math.sqrt(d)
    for b in range(bsz):
        for h in range(hkv * g):
            kh = h // g
            ln = lens[b]
            keys = o.dequantize_prod(kq["idx"][b, kh, :ln], kq["sign"][b, kh, :ln],
                                     kq["n"][b, kh, :ln], kq["gamma"][b, kh, :ln], pi, s, kc)
            vals = o.dequantize_mse(vi[b, kh, :ln], vn[b, kh, :ln], pi, vc)
            ref = _brute_attention(list(q[b, h]), keys.tolist(), vals.tolist(), scale)
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-10, atol=1e-12)


def pin_asym_concatenation(o):
    """Asymmetric mode: one softmax over FP16 keys of the compressed segment and the FP16
    tail equals brute force over the concatenated key/value lists."""
    rng = np.random.default_rng(23)
    d = 128
    pi = _rotation(o, 42)
    vc, _ = o.lloyd_max_codebook(d, 4)
    bsz, hkv, g = 2, 1, 2
    k = rng.standard_normal((bsz, hkv, 5, d)).astype(np.float16)
    v = rng.standard_normal((bsz, hkv, 5, d))
    kt = rng.standard_normal((bsz, hkv, 3, d)).astype(np.float16)
    vt = rng.standard_normal((bsz, hkv, 3, d)).astype(np.float16)
    q = rng.standard_normal((bsz, hkv * g, d))
    vi, vn, _ = o.quantize_mse(v, pi, vc)
    lens, tlens = [5, 2], [3, 0]
    out = o.decode_attention_asym(q, k, {"idx": vi, "n": vn}, lens, kt, vt, tlens, pi, vc)
    for b in range(bsz):
        for h in range(hkv * g):
            vals = o.dequantize_mse(vi[b, 0, :lens[b]], vn[b, 0, :lens[b]], pi, vc)
            keys = np.concatenate([k[b, 0, :lens[b]], kt[b, 0, :tlens[b]]]).astype(np.float64)
            allv = np.concatenate([vals, vt[b, 0, :tlens[b]].astype(np.float64)])
            ref = _brute_attention(list(q[b, h]), keys.tolist(), allv.tolist(), 1 / math.sqrt(d))
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-10, atol=1e-12)


def pin_boundary_exclusion_rate(o):
    """The share of rotated coordinates within eps of a boundary is ≈ 2·eps·Σ f(boundary);
    checked with a wide eps so the Monte-Carlo count is large, and the 1e-6 rate is below
    1e-4 of coordinates for every bit width used."""
    rng = np.random.default_rng(29)
    pi = _rotation(o, 42)
    x = rng.standard_normal((8000, 128))
    for bits in (2, 3, 4):
        c, b = o.lloyd_max_codebook(128, bits)
        _, _, y = o.quantize_mse(x, pi, c)
        eps = 2e-3
        excl, alt = o.boundary_exclusion(y, c, eps=eps)
        expect = 2 * eps * sum(_density_indep(t, 128) for t in b)
        got = excl.mean()
        assert abs(got - expect) < 5 * math.sqrt(expect / excl.size) + 0.02 * expect
        assert 2e-6 * sum(_density_indep(t, 128) for t in b) < 1e-4
        idx, _, _ = o.quantize_mse(x, pi, c)
        assert np.all(np.abs(alt - idx) == 1)


def pin_sign_exclusion_rate(o):
    """The share of QJL sign bits that the parity checks skip matches its closed form.  With a
    fresh Gaussian sketch S for every vector (independent of x), (S r)_j ~ N(0, ||r||²)
    exactly, so the share of the vector's bits inside the band |z_j| < eps·√d·||x|| is
    erf(eps·√d·||x|| / (√2·||r||)).  Checked per index width with a wide eps (so the count is
    large) and for the 1e-6 band: the expected share stays below 1e-4.  A band with d in
    place of √d, ||r|| in place of ||x||, or a tenfold width misses the closed form."""
    from scipy import special
    rng = np.random.default_rng(31)
    d = 128
    pi = _rotation(o, 42)
    nvec = 1500
    for ibits in (1, 2, 3):
        c, _ = o.lloyd_max_codebook(d, ibits)
        eps = 1e-3
        got = 0
        expect = 0.0
        expect_1e6 = 0.0
        for v in range(nvec):
            x = rng.standard_normal((1, d)) * np.exp(0.5 * rng.standard_normal(d))
            s = rng.standard_normal((d, d))
            k = o.quantize_prod(x, pi, s, c)
            got += int(o.sign_exclusion(k["z"], k["n"], d, eps=eps).sum())
            ratio = math.sqrt(d) * k["n"][0] / (math.sqrt(2.0) * k["gamma"][0])
            expect += d * special.erf(eps * ratio)
            expect_1e6 += d * special.erf(1e-6 * ratio)
        total = nvec * d
        sd = math.sqrt(expect * (1 - expect / total))
        assert abs(got - expect) < 5 * sd + 0.02 * expect, (ibits, got, expect)
        assert expect_1e6 / total < 1e-4, (ibits, expect_1e6 / total)


def pin_softmax_kl(o):
    """KL of softmax distributions: zero for equal inputs and invariant to a shift of either
    input; the two-token case equals the Bernoulli KL written out; random small vectors equal
    a pure-Python double loop; never negative."""
    assert abs(o.softmax_kl([0.3, -1.2, 2.0], [0.3, -1.2, 2.0])) < 1e-15
    a, b = 0.7, -0.4
    pa, pb = 1 / (1 + math.exp(-a)), 1 / (1 + math.exp(-b))
    bern = pa * math.log(pa / pb) + (1 - pa) * math.log((1 - pa) / (1 - pb))
    assert abs(o.softmax_kl([a, 0.0], [b, 0.0]) - bern) < 1e-14
    rng = np.random.default_rng(37)
    for _ in range(20):
        x = rng.standard_normal(5) * 3
        y = rng.standard_normal(5) * 3
        zx = sum(math.exp(v) for v in x)
        zy = sum(math.exp(v) for v in y)
        brute = sum(math.exp(x[t]) / zx * (math.log(math.exp(x[t]) / zx) - math.log(math.exp(y[t]) / zy))
                    for t in range(5))
        assert abs(o.softmax_kl(x, y) - brute) < 1e-12
        assert abs(o.softmax_kl(x + 4.0, y - 2.5) - brute) < 1e-12
        assert o.softmax_kl(x, y) >= 0


def pin_attention_quality(o):
    """attention_quality: exact scores are scale·⟨q, k⟩ and compressed scores the estimator
    (checked against a loop over the dequantised keys); the argmaxes match brute force."""
    rng = np.random.default_rng(41)
    pi = _rotation(o, 42)
    s = _sketch(43)
    c, _ = o.lloyd_max_codebook(128, 2)
    keys = rng.standard_normal((12, 128))
    q = rng.standard_normal((3, 128))
    k = o.quantize_prod(keys, pi, s, c)
    kl, te, tc = o.attention_quality(q, keys, k["idx"], k["sign"], k["n"], k["gamma"], pi, s, c)
    kh = o.dequantize_prod(k["idx"], k["sign"], k["n"], k["gamma"], pi, s, c)
    scale = 1 / math.sqrt(128)
    for i in range(3):
        ex = [scale * float(np.dot(q[i], keys[t])) for t in range(12)]
        cp = [scale * float(np.dot(q[i], kh[t])) for t in range(12)]
        assert te[i] == max(range(12), key=lambda t: ex[t])
        assert tc[i] == max(range(12), key=lambda t: cp[t])
        zx = sum(math.exp(v) for v in ex)
        zy = sum(math.exp(v) for v in cp)
        brute = sum(math.exp(ex[t]) / zx * (ex[t] - cp[t]) for t in range(12)) - math.log(zx) + math.log(zy)
        assert abs(kl[i] - brute) < 1e-10


ALL_PINS = [
    pin_rotation, pin_codebook_closed_form_1bit, pin_codebook_centroid_condition,
    pin_codebook_gaussian_limit, pin_codebook_mse_monotone, pin_mse_index_is_nearest_level,
    pin_mse_distortion, pin_value_cos_sim_pages, pin_qjl_identity, pin_estimator_unbiased,
    pin_estimator_equals_dequantized_dot, pin_residual_definition, pin_zero_vector,
    pin_packing_golden, pin_attention_brute_force, pin_asym_concatenation,
    pin_boundary_exclusion_rate, pin_sign_exclusion_rate, pin_softmax_kl, pin_attention_quality,
]
