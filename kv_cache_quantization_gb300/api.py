"""PyTorch-facing convenience layer over the C ABI.

PyTorch only owns memory and streams here: caches and workspaces are torch tensors whose
addresses are handed to libtq.so; every step of quantisation and attention runs in the
library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
from typing import Optional

import numpy as np
import torch

from . import _binding as B

HEAD_DIM = B.TQ_HEAD_DIM

_DT = {torch.float32: B.TQ_F32, torch.float16: B.TQ_F16, torch.bfloat16: B.TQ_BF16}


def tq_dtype(dt: torch.dtype) -> int:
    if dt not in _DT:
        raise TypeError(f"unsupported dtype {dt}")
    return _DT[dt]


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ host constants

def lloyd_max_codebook(index_bits: int, d: int = HEAD_DIM) -> np.ndarray:
    """Ascending Lloyd-Max levels for the sphere-coordinate law (library host code)."""
    out = np.zeros(1 << index_bits, dtype=np.float64)
    B.check(B.tq_lloyd_max_codebook(d, index_bits, out.ctypes.data), "tq_lloyd_max_codebook")
    return out


def rotation_from_gaussian(g: np.ndarray) -> np.ndarray:
    """Π = sign-fixed Q of G = QR (library host code)."""
    g = np.ascontiguousarray(g, dtype=np.float64)
    d = g.shape[0]
    out = np.zeros((d, d), dtype=np.float64)
    B.check(B.tq_rotation_from_gaussian(d, g.ctypes.data, out.ctypes.data),
            "tq_rotation_from_gaussian")
    return out


def layer_constants(layer: int = 0, d: int = HEAD_DIM):
    """(Π, S) of a layer from the per-layer Gaussians (seeds 42 + 7ℓ and 43 + 7ℓ)."""
    from .synth import gaussian_matrix, layer_seeds
    sp, ss = layer_seeds(layer)
    return rotation_from_gaussian(gaussian_matrix(sp, d)), gaussian_matrix(ss, d)


# ------------------------------------------------------------------ codec

class Codec:
    """Owns a tq_codec (device copies of Π, Πᵀ, Sᵀ, M and the codebook)."""

    def __init__(self, kind: int, bits: int, pi: np.ndarray, s: Optional[np.ndarray] = None,
                 centroids: Optional[np.ndarray] = None):
        self.kind = kind
        self.bits = bits
        self.index_bits = bits - 1 if kind == B.TQ_PROD else bits
        if centroids is None:
            centroids = lloyd_max_codebook(self.index_bits)
        self.pi = np.ascontiguousarray(pi, dtype=np.float64)
        self.s = None if s is None else np.ascontiguousarray(s, dtype=np.float64)
        self.centroids = np.ascontiguousarray(centroids, dtype=np.float64)
        h = ctypes.c_void_p()
        B.check(B.tq_codec_create(HEAD_DIM, kind, bits, self.pi.ctypes.data,
                                  0 if self.s is None else self.s.ctypes.data,
                                  self.centroids.ctypes.data, h), "tq_codec_create")
        self.handle = h

    @classmethod
    def prod(cls, bits: int, layer: int = 0) -> "Codec":
        pi, s = layer_constants(layer)
        return cls(B.TQ_PROD, bits, pi, s)

    @classmethod
    def mse(cls, bits: int, layer: int = 0) -> "Codec":
        pi, _ = layer_constants(layer)
        return cls(B.TQ_MSE, bits, pi)

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            B.tq_codec_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------ caches

def _cap(capacity: int) -> int:
    a = B.TQ_CAPACITY_ALIGN
    return (capacity + a - 1) // a * a


@dataclasses.dataclass
class Pages:
    """A block table over a page pool (include/tq.h, tq_pages): token t of sequence b lives in
    slot t % page_tokens of page block_table[b, t // page_tokens]."""
    block_table: torch.Tensor   # int32 [batch, max_pages], on the device
    page_tokens: int
    num_pages: int

    def __post_init__(self):
        if self.block_table.dtype != torch.int32 or self.block_table.dim() != 2:
            raise ValueError("block_table must be int32 [batch, max_pages]")
        self.block_table = self.block_table.contiguous()
        self._c = B.tq_pages(self.block_table.data_ptr(), self.block_table.shape[1],
                             self.page_tokens, self.num_pages)

    @property
    def max_pages(self):
        return self.block_table.shape[1]

    @property
    def capacity(self):
        """Slots per sequence."""
        return self.max_pages * self.page_tokens

    def c(self):
        return ctypes.pointer(self._c)


def _pages_ptr(pages):
    return None if pages is None else pages.c()


@dataclasses.dataclass
class ProdCache:
    """Packed key cache [batch][heads][capacity] (layout of include/tq.h); with `pages` the
    arrays are a page pool [num_pages][heads][page_tokens] addressed through a block table."""
    idx: torch.Tensor      # uint8 [B, H, b-1, cap, 16]
    sgn: torch.Tensor      # uint8 [B, H, cap, 16]
    xnorm: torch.Tensor    # float32 [B, H, cap]
    rnorm: torch.Tensor    # float32 [B, H, cap]
    pages: Optional[Pages] = None

    @classmethod
    def empty(cls, batch, heads, capacity, bits, device="cuda"):
        cap = _cap(capacity)
        return cls(torch.zeros(batch, heads, bits - 1, cap, 16, dtype=torch.uint8, device=device),
                   torch.zeros(batch, heads, cap, 16, dtype=torch.uint8, device=device),
                   torch.zeros(batch, heads, cap, dtype=torch.float32, device=device),
                   torch.zeros(batch, heads, cap, dtype=torch.float32, device=device))

    @classmethod
    def empty_paged(cls, pages: Pages, heads, bits, device="cuda"):
        """A zeroed page pool of pages.num_pages pages for the block table `pages`."""
        c = cls.empty(pages.num_pages, heads, pages.page_tokens, bits, device)
        if c.capacity != pages.page_tokens:
            raise ValueError("page_tokens must be a multiple of TQ_CAPACITY_ALIGN")
        c.pages = pages
        return c

    @property
    def capacity(self):
        return self.pages.capacity if self.pages is not None else self.sgn.shape[2]

    def c(self):
        return B.tq_prod_cache(self.idx.data_ptr(), self.sgn.data_ptr(), self.xnorm.data_ptr(),
                               self.rnorm.data_ptr(), _pages_ptr(self.pages))

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in (self.idx, self.sgn, self.xnorm, self.rnorm))


@dataclasses.dataclass
class MSECache:
    """Packed value cache [batch][heads][capacity]: bit planes, or nibbles for 4 bits; with
    `pages` a page pool as for ProdCache."""
    idx: torch.Tensor      # uint8 [B, H, bits, cap, 16] or [B, H, cap, 64]
    xnorm: torch.Tensor    # float32 [B, H, cap]
    bits: int
    pages: Optional[Pages] = None

    @classmethod
    def empty(cls, batch, heads, capacity, bits, device="cuda"):
        cap = _cap(capacity)
        if bits == 4:
            idx = torch.zeros(batch, heads, cap, 64, dtype=torch.uint8, device=device)
        else:
            idx = torch.zeros(batch, heads, bits, cap, 16, dtype=torch.uint8, device=device)
        return cls(idx, torch.zeros(batch, heads, cap, dtype=torch.float32, device=device), bits)

    @classmethod
    def empty_paged(cls, pages: Pages, heads, bits, device="cuda"):
        """A zeroed page pool of pages.num_pages pages for the block table `pages`."""
        c = cls.empty(pages.num_pages, heads, pages.page_tokens, bits, device)
        if c.xnorm.shape[2] != pages.page_tokens:
            raise ValueError("page_tokens must be a multiple of TQ_CAPACITY_ALIGN")
        c.pages = pages
        return c

    @property
    def capacity(self):
        return self.pages.capacity if self.pages is not None else self.xnorm.shape[2]

    def c(self):
        return B.tq_mse_cache(self.idx.data_ptr(), self.xnorm.data_ptr(), _pages_ptr(self.pages))

    def nbytes(self):
        return self.idx.numel() + self.xnorm.numel() * 4


# ------------------------------------------------------------------ calls

def _x_args(x: torch.Tensor):
    if x.dim() != 4 or x.shape[-1] != HEAD_DIM or x.stride(-1) != 1:
        raise ValueError("x must be [batch, heads, tokens, 128] with contiguous last dim")
    bsz, h, t, _ = x.shape
    return bsz, h, t, x.stride(0), x.stride(1), x.stride(2)


def quantize_prod(codec: Codec, x: torch.Tensor, cache: ProdCache, pos=None, count=None,
                  stream=None):
    bsz, h, t, sb, sh, st = _x_args(x)
    B.check(B.tq_quantize_prod(codec.handle, x, tq_dtype(x.dtype), bsz, h, t, sb, sh, st, pos,
                               count, cache.c(), cache.capacity, _stream(stream)),
            "tq_quantize_prod")


def quantize_mse(codec: Codec, x: torch.Tensor, cache: MSECache, pos=None, count=None,
                 stream=None):
    bsz, h, t, sb, sh, st = _x_args(x)
    B.check(B.tq_quantize_mse(codec.handle, x, tq_dtype(x.dtype), bsz, h, t, sb, sh, st, pos,
                              count, cache.c(), cache.capacity, _stream(stream)),
            "tq_quantize_mse")


def prod_scores(codec: Codec, q: torch.Tensor, keys: ProdCache, n: int, out=None, stream=None):
    """[nq, n] raw estimator scores of fp32 queries q [nq, 128] against keys[0, 0, :n]."""
    q = q.contiguous()
    if out is None:
        out = torch.empty(q.shape[0], n, dtype=torch.float32, device=q.device)
    B.check(B.tq_prod_scores(codec.handle, q, q.shape[0], q.stride(0), keys.c(), keys.capacity,
                             n, out, out.stride(0), _stream(stream)), "tq_prod_scores")
    return out


def attention_quality(codec: Codec, q: torch.Tensor, k: torch.Tensor, keys: ProdCache, n: int,
                      softmax_scale=None, stream=None):
    """(KL [nq], top-1 position over exact keys [nq], over compressed keys [nq]) for fp32
    queries q [nq, 128] against the exact keys k [n, 128] and their codes keys[0, 0, :n]."""
    q = q.contiguous()
    k = k.contiguous()
    nq = q.shape[0]
    scratch = torch.empty(B.tq_attention_quality_scratch_bytes(nq, n), dtype=torch.uint8,
                          device=q.device)
    kl = torch.empty(nq, dtype=torch.float32, device=q.device)
    te = torch.empty(nq, dtype=torch.int32, device=q.device)
    tc = torch.empty(nq, dtype=torch.int32, device=q.device)
    B.check(B.tq_attention_quality(codec.handle, q, nq, k, tq_dtype(k.dtype), keys.c(),
                                   keys.capacity, n, softmax_scale or 0.0, scratch,
                                   scratch.numel(), kl, te, tc, _stream(stream)),
            "tq_attention_quality")
    return kl, te, tc


class DecodePlan:
    """A decode-attention configuration with its workspace (allocated once, reused)."""

    def __init__(self, batch, q_heads, kv_heads, capacity, max_seq_len, q_dtype=torch.bfloat16,
                 out_dtype=torch.float32, tail_capacity=0, softmax_scale=None, device="cuda"):
        self.desc = B.tq_attn_desc(batch, q_heads, kv_heads, HEAD_DIM, _cap(capacity),
                                   max_seq_len, tail_capacity,
                                   softmax_scale if softmax_scale else 0.0,
                                   tq_dtype(q_dtype), tq_dtype(out_dtype))
        nbytes = B.tq_decode_workspace_bytes(self.desc)
        if nbytes == 0:
            raise ValueError("invalid decode-attention configuration")
        # caller-owned scratch; the library clears what must start at zero on every call
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.out_dtype = out_dtype
        self.shape = (batch, q_heads, HEAD_DIM)

    def new_out(self, device="cuda"):
        return torch.empty(self.shape, dtype=self.out_dtype, device=device)

    def run(self, kc: Codec, vc: Codec, q, k: ProdCache, v: MSECache, seq_lens, out, stream=None):
        B.check(B.tq_decode_attention(self.desc, kc.handle, vc.handle, q, k.c(), v.c(), seq_lens,
                                      out, self.workspace, self.workspace.numel(),
                                      _stream(stream)), "tq_decode_attention")
        return out

    def step(self, kc: Codec, vc: Codec, q, k_new, v_new, k: ProdCache, v: MSECache, pos, out,
             lens_out=None, stream=None):
        """Appends k_new, v_new [batch, kv_heads, 128] at pos[b] and attends pos[b] + 1 tokens."""
        if k_new.dtype != v_new.dtype or not (k_new.is_contiguous() and v_new.is_contiguous()):
            raise ValueError("k_new and v_new must be contiguous and of one dtype")
        B.check(B.tq_decode_step(self.desc, kc.handle, vc.handle, q, k_new, v_new,
                                 tq_dtype(k_new.dtype), k.c(), v.c(), pos, lens_out, out,
                                 self.workspace, self.workspace.numel(), _stream(stream)),
                "tq_decode_step")
        return out

    def run_asym(self, vc: Codec, q, k_f16, v: MSECache, seq_lens, k_tail, v_tail, tail_lens,
                 out, stream=None):
        B.check(B.tq_decode_attention_asym(self.desc, vc.handle, q, k_f16, v.c(), seq_lens,
                                           k_tail, v_tail, tail_lens, out, self.workspace,
                                           self.workspace.numel(), _stream(stream)),
                "tq_decode_attention_asym")
        return out


class PrefillPlan:
    """Attention of chunks of n_queries queries per sequence over a compressed cache
    (tq_prefill_attention), with its workspace."""

    def __init__(self, batch, n_queries, q_heads, kv_heads, capacity, max_seq_len, causal=True,
                 q_dtype=torch.bfloat16, out_dtype=torch.float32, device="cuda"):
        self.desc = B.tq_attn_desc(batch, q_heads, kv_heads, HEAD_DIM, _cap(capacity), max_seq_len,
                                   0, 0.0, tq_dtype(q_dtype), tq_dtype(out_dtype))
        self.n_queries = n_queries
        self.causal = 1 if causal else 0
        nbytes = B.tq_prefill_workspace_bytes(self.desc, n_queries)
        if nbytes == 0:
            raise ValueError("invalid prefill-attention configuration")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.out_dtype = out_dtype
        self.shape = (batch, n_queries, q_heads, HEAD_DIM)

    def new_out(self, device="cuda"):
        return torch.empty(self.shape, dtype=self.out_dtype, device=device)

    def run(self, kc: Codec, vc: Codec, q, k: ProdCache, v: MSECache, seq_lens, out, stream=None):
        B.check(B.tq_prefill_attention(self.desc, self.n_queries, self.causal, kc.handle, vc.handle,
                                       q, k.c(), v.c(), seq_lens, out, self.workspace,
                                       self.workspace.numel(), _stream(stream)),
                "tq_prefill_attention")
        return out


class TailStore:
    """A cache in the asymmetric layout: a compressed part (FP16 keys, MSE-coded values) and an
    FP16 tail of the most recent tokens that compacts into the compressed part when it fills
    (tq_store_append); read with DecodePlan.run_asym."""

    def __init__(self, vc: Codec, batch, kv_heads, capacity, tail_capacity=256, device="cuda"):
        cap = _cap(capacity)
        self.vc = vc
        self.batch, self.kv_heads, self.capacity, self.tail_capacity = batch, kv_heads, cap, tail_capacity
        self.k_f16 = torch.zeros(batch, kv_heads, cap, HEAD_DIM, dtype=torch.float16, device=device)
        self.v = MSECache.empty(batch, kv_heads, cap, vc.bits, device=device)
        self.k_tail = torch.zeros(batch, kv_heads, tail_capacity, HEAD_DIM, dtype=torch.float16,
                                  device=device)
        self.v_tail = torch.zeros_like(self.k_tail)
        self.comp_lens = torch.zeros(batch, dtype=torch.int32, device=device)
        self.tail_lens = torch.zeros(batch, dtype=torch.int32, device=device)
        self.workspace = torch.empty(max(B.tq_store_workspace_bytes(batch), 256), dtype=torch.uint8,
                                     device=device)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """k_new, v_new: [batch, kv_heads, 128] contiguous, one dtype."""
        B.check(B.tq_store_append(self.vc.handle, self.batch, self.kv_heads, k_new, v_new,
                                  tq_dtype(k_new.dtype), self.k_f16, self.v.c(), self.capacity,
                                  self.k_tail, self.v_tail, self.tail_capacity, self.comp_lens,
                                  self.tail_lens, self.workspace, self.workspace.numel(),
                                  _stream(stream)), "tq_store_append")

    def plan(self, q_heads, q_dtype=torch.bfloat16, out_dtype=torch.float32, device="cuda"):
        return DecodePlan(self.batch, q_heads, self.kv_heads, self.capacity, self.capacity, q_dtype,
                          out_dtype, tail_capacity=self.tail_capacity, device=device)

    def decode(self, plan: "DecodePlan", q, out, stream=None):
        return plan.run_asym(self.vc, q, self.k_f16, self.v, self.comp_lens, self.k_tail,
                             self.v_tail, self.tail_lens, out, stream=stream)


def device_status():
    """(status, flags) of the device status word (synchronises the device)."""
    return B.tq_device_status()
