"""Seeded synthetic workloads.

This module only draws random numbers: it holds none of the quantiser's or the attention's
arithmetic, so both the CUDA library's tests and the CPU oracle can take their inputs from
it.  Recipes:

* Gaussian matrices for the rotation and the sketch: ``numpy.random.default_rng(seed)``
  standard normals, d x d, seed 42 + 7*layer for the rotation's Gaussian and 43 + 7*layer
  for S (per-layer seed convention of the QJL deep-dive article, §六 "store").
* Activations: N(0, 1) entries, each (head, channel) scaled by exp(0.5 * N(0, 1))
  (lognormal(0, 0.5)), drawn in float32 and rounded once to the workload's input dtype.
  Long-context keys instead carry 4 outlier channels scaled by 10 and no lognormal scale.
* Ragged serving lengths: uniform integers in [4096, 16384], ``default_rng(2005)``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

HEAD_DIM = 128


def gaussian_matrix(seed: int, d: int = HEAD_DIM) -> np.ndarray:
    """d x d standard normal matrix from ``default_rng(seed)`` (float64)."""
    return np.random.default_rng(seed).standard_normal((d, d))


def layer_seeds(layer: int):
    """(rotation seed, sketch seed) for a layer: 42 + 7*layer and 43 + 7*layer."""
    return 42 + 7 * layer, 43 + 7 * layer


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    q_heads: int
    kv_heads: int
    context: int                 # max tokens per sequence held in the cache
    k_bits: int                  # total bits of the key product code; 0 = keys kept FP16
    v_bits: int                  # bits of the value MSE code
    in_dtype: torch.dtype
    out_dtype: torch.dtype
    queries: int = 1             # queries per (batch, head) (scores workload: 64)
    tail: int = 0                # FP16 tail tokens (asymmetric mode)
    ragged: Optional[tuple] = None   # (lo, hi, seed) for uniform ragged lengths
    outlier_channels: int = 0
    decode_steps: int = 0
    layer: int = 0
    data_seed: int = 1000

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads


# The five synthetic workloads (shapes of a Qwen2.5-7B-like GQA layer and of the
# long-context / serving cases).
SCORES_1K = Workload("scores_d128_n1024_fp32", 1, 1, 1, 1024, 3, 0, torch.float32,
                     torch.float32, queries=64, data_seed=1001)
DECODE_32K = Workload("decode_gqa28x4_ctx32768_k3v4", 1, 28, 4, 32768, 3, 4, torch.bfloat16,
                      torch.float32, data_seed=1002)
ASYM_8K = Workload("asym_b8_ctx8192_kfp16_v4_tail255", 8, 28, 4, 8192, 0, 4, torch.bfloat16,
                   torch.bfloat16, tail=255, data_seed=1003)
LONG_262K = Workload("longctx_gqa32x8_ctx262144_k3v2", 1, 32, 8, 262144, 3, 2, torch.bfloat16,
                     torch.float32, outlier_channels=4, data_seed=1004)
SERVE_B32 = Workload("serving_b32_ragged4k-16k_k4v4", 32, 28, 4, 16384, 4, 4, torch.bfloat16,
                     torch.float32, ragged=(4096, 16384, 2005), decode_steps=128, data_seed=1005)

WORKLOADS = {w.name: w for w in (SCORES_1K, DECODE_32K, ASYM_8K, LONG_262K, SERVE_B32)}


def seq_lengths(w: Workload) -> np.ndarray:
    """Cached tokens per sequence before decoding (compressed part only for the asymmetric
    workload, whose last ``tail`` tokens stay FP16)."""
    if w.ragged is not None:
        lo, hi, seed = w.ragged
        return np.random.default_rng(seed).integers(lo, hi, size=w.batch, endpoint=True)
    return np.full(w.batch, w.context - w.tail, dtype=np.int64)


def _generator(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def channel_scales(w: Workload, which: str, device="cpu") -> torch.Tensor:
    """lognormal(0, 0.5) scale per (head, channel) for the workload's "q", "k" or "v"
    activations: [1, heads, 1, HEAD_DIM] float32, fixed for the whole workload."""
    heads = w.q_heads if which == "q" else w.kv_heads
    gen = _generator("cpu", w.data_seed * 10 + "qkv".index(which))
    z = torch.randn(1, heads, 1, HEAD_DIM, generator=gen, dtype=torch.float32)
    return torch.exp(0.5 * z).to(device)


def _draw(w: Workload, which: str, shape, gen, device) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if w.outlier_channels:
        if which == "k":
            ch = np.random.default_rng(w.data_seed).choice(HEAD_DIM, w.outlier_channels,
                                                           replace=False)
            x[..., torch.as_tensor(ch, device=device)] *= 10.0
        return x
    return x * channel_scales(w, which, device)


def make_kv(w: Workload, device="cpu", tokens: Optional[int] = None):
    """Keys and values [B, Hkv, T, d] in the workload's input dtype (T = context unless
    given).  Long-context keys: N(0,1) with 4 seeded outlier channels x10; values N(0,1)."""
    t = w.context if tokens is None else tokens
    gen = _generator(device, w.data_seed)
    shape = (w.batch, w.kv_heads, t, HEAD_DIM)
    k = _draw(w, "k", shape, gen, device)
    v = _draw(w, "v", shape, gen, device)
    return k.to(w.in_dtype), v.to(w.in_dtype)


def make_queries(w: Workload, device="cpu", step: int = 0):
    """Queries [B, Hq, queries, d] in the input dtype; ``step`` picks an independent draw
    for each decode step."""
    gen = _generator(device, w.data_seed * 1000 + 17 + step)
    return _draw(w, "q", (w.batch, w.q_heads, w.queries, HEAD_DIM), gen, device).to(w.in_dtype)


def make_new_tokens(w: Workload, device="cpu", step: int = 0):
    """One new key and value per (batch, kv head) for decode step ``step``: [B, Hkv, 1, d]."""
    gen = _generator(device, w.data_seed * 1000 + 500 + step)
    shape = (w.batch, w.kv_heads, 1, HEAD_DIM)
    k = _draw(w, "k", shape, gen, device)
    v = _draw(w, "v", shape, gen, device)
    return k.to(w.in_dtype), v.to(w.in_dtype)


def cache_capacity(w: Workload) -> int:
    """Tokens per (sequence, KV head) a cache for the workload must hold: its context, or its
    longest sequence after the decode steps' appends if that is more, in whole 64-token
    blocks."""
    need = max(w.context, int(seq_lengths(w).max()) + w.decode_steps)
    return (need + 63) // 64 * 64


TAIL_CAPACITY = 256   # FP16 tail slots per (sequence, KV head): at most min_compress - 1 used


def asym_tail(w: Workload, k: torch.Tensor, v: torch.Tensor):
    """FP16 tail of the asymmetric workload, [B, Hkv, TAIL_CAPACITY, d]: slots t < w.tail hold
    the last w.tail tokens of each sequence (the ones not in the compressed part), the rest
    are zero."""
    shape = (w.batch, w.kv_heads, TAIL_CAPACITY, HEAD_DIM)
    kt = torch.zeros(shape, dtype=torch.float16, device=k.device)
    vt = torch.zeros(shape, dtype=torch.float16, device=v.device)
    start = w.context - w.tail
    kt[:, :, :w.tail] = k[:, :, start:w.context].to(torch.float16)
    vt[:, :, :w.tail] = v[:, :, start:w.context].to(torch.float16)
    return kt, vt
