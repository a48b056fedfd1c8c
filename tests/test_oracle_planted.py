"""Plant one mistake at a time in a private copy of the oracle (CPU only) and require that
at least one pin catches it: the pins are sensitive to the plausible slips (a dropped term,
a wrong sign or index, a transposed operand, a wrong constant)."""
import importlib.util
import math
import os

import numpy as np
import pytest

from oracle_pins import ALL_PINS

ORACLE_FILE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "turboquant.py")


def fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_copy", ORACLE_FILE)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def plant_drop_qjl(o):
    orig = o.prod_scores

    def f(q, idx, sign, n, gamma, pi, s, c):
        return orig(q, idx, sign, n, np.zeros_like(gamma), pi, s, c)
    o.prod_scores = f


def plant_flip_qjl_sign(o):
    o.QJL_SCALE_NUMERATOR = -o.QJL_SCALE_NUMERATOR


def plant_wrong_qjl_constant(o):
    o.QJL_SCALE_NUMERATOR = math.pi / 2


def plant_transposed_rotation(o):
    orig = o.quantize_mse

    def f(x, pi, c):
        return orig(x, np.asarray(pi).T, c)
    o.quantize_mse = f


def plant_no_sign_fix(o):
    o.rotation_from_gaussian = lambda g: np.linalg.qr(np.asarray(g, dtype=np.float64))[0]


def plant_cell_midpoint_levels(o):
    def f(d, bits, tol=1e-15, max_iter=0):
        levels = 1 << bits
        edges = np.linspace(-3, 3, levels + 1) / math.sqrt(d)
        c = 0.5 * (edges[:-1] + edges[1:])
        return c, 0.5 * (c[:-1] + c[1:])
    o.lloyd_max_codebook = f


def plant_residual_sign(o):
    orig = o.prod_residual

    def f(x, n, idx, pi, s, c):
        sign, gamma, z = orig(x, n, idx, pi, s, c)
        return ~sign, gamma, -z
    o.prod_residual = f


def plant_gqa_mapping(o):
    """Query head h reads KV head h % Hkv instead of h // G."""
    orig_dec = o.decode_attention

    def g(q, k_codes, v_codes, seq_lens, pi, s, kc, vc, scale=None):
        out = orig_dec(q, k_codes, v_codes, seq_lens, pi, s, kc, vc, scale)
        hq, hkv = out.shape[1], k_codes["idx"].shape[1]
        return out[:, [(h % hkv) * (hq // hkv) for h in range(hq)]]
    o.decode_attention = g


def plant_msb_first(o):
    """Coordinate j stored at bit 7 - j % 8 instead of bit j % 8."""
    orig = o.pack_bits

    def f(bits):
        b = np.asarray(bits)
        return orig(b.reshape(b.shape[:-1] + (-1, 8))[..., ::-1].reshape(b.shape))
    o.pack_bits = f


def plant_mse_norm_dropped(o):
    orig = o.dequantize_mse
    o.dequantize_mse = lambda idx, n, pi, c: orig(idx, np.ones_like(np.asarray(n, dtype=float)), pi, c)


def plant_ties_down_and_shift(o):
    orig = o.quantize_mse

    def f(x, pi, c):
        idx, n, y = orig(x, pi, c)
        return np.maximum(idx - (y > 0.05), 0), n, y
    o.quantize_mse = f


def plant_sign_band_power_of_d(o):
    """Sign band eps·d·||x|| instead of eps·√d·||x||."""
    o.sign_exclusion = lambda z, n, d, eps=1e-6: np.abs(np.asarray(z)) < eps * d * np.asarray(n)[..., None]


def plant_sign_band_residual_norm(o):
    """Sign band scaled by the residual's norm (||r|| ≈ ||S r|| / √d) instead of ||x||."""
    def band(z, n, d, eps=1e-6):
        z = np.asarray(z, dtype=np.float64)
        rn = np.linalg.norm(z, axis=-1, keepdims=True) / math.sqrt(d)
        return np.abs(z) < eps * math.sqrt(d) * rn
    o.sign_exclusion = band


def plant_sign_band_tenfold(o):
    orig = o.sign_exclusion
    o.sign_exclusion = lambda z, n, d, eps=1e-6: orig(z, n, d, eps * 10)


def plant_kl_reversed(o):
    """KL(compressed ‖ exact) instead of KL(exact ‖ compressed)."""
    orig = o.softmax_kl
    o.softmax_kl = lambda a, b: orig(b, a)


def plant_kl_unnormalised(o):
    """Log-probabilities without the log-partition term."""
    def f(a, b):
        a = np.asarray(a, dtype=float)
        b = np.asarray(b, dtype=float)
        p = np.exp(a - np.max(a, axis=-1, keepdims=True))
        p /= p.sum(axis=-1, keepdims=True)
        return np.sum(p * (a - b), axis=-1)
    o.softmax_kl = f


PLANTS = [plant_drop_qjl, plant_flip_qjl_sign, plant_wrong_qjl_constant,
          plant_transposed_rotation, plant_no_sign_fix, plant_cell_midpoint_levels,
          plant_residual_sign, plant_gqa_mapping, plant_msb_first, plant_mse_norm_dropped,
          plant_ties_down_and_shift, plant_sign_band_power_of_d, plant_sign_band_residual_norm,
          plant_sign_band_tenfold, plant_kl_reversed, plant_kl_unnormalised]


@pytest.mark.parametrize("plant", PLANTS, ids=lambda p: p.__name__)
def test_planted_mistake_is_caught(plant):
    o = fresh_oracle()
    plant(o)
    failures = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception as e:  # any failure of any pin counts as caught
            failures.append(pin.__name__)
            break
    assert failures, f"no pin caught {plant.__name__}"
