"""ctypes binding of libtq.so: the C ABI of include/tq.h under the same names.

Argument marshalling only.  Device buffers are passed as integer addresses (or objects with
``data_ptr()``, e.g. torch tensors); every computation happens in the library.  The binding
raises if the library has not been built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libtq.so")

(TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA, TQ_ERR_TIMEOUT, TQ_ERR_DEVICE_STATUS,
 TQ_ERR_SCRATCH_LIMIT) = range(7)
TQ_F32, TQ_F16, TQ_BF16 = 0, 1, 2
TQ_PROD, TQ_MSE = 0, 1
TQ_HEAD_DIM = 128
TQ_MAX_GROUP = 8
TQ_CAPACITY_ALIGN = 64
TQ_FLAG_POS_OVERFLOW, TQ_FLAG_LEN_OVERFLOW, TQ_FLAG_TIMEOUT, TQ_FLAG_PAGE = 1, 2, 4, 8

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


class tq_pages(ctypes.Structure):
    _fields_ = [("block_table", _vp), ("max_pages", _i32), ("page_tokens", _i32),
                ("num_pages", _i32)]


class tq_prod_cache(ctypes.Structure):
    _fields_ = [("idx", _vp), ("sgn", _vp), ("xnorm", _vp), ("rnorm", _vp),
                ("pages", ctypes.POINTER(tq_pages))]


class tq_mse_cache(ctypes.Structure):
    _fields_ = [("idx", _vp), ("xnorm", _vp), ("pages", ctypes.POINTER(tq_pages))]


class tq_attn_desc(ctypes.Structure):
    _fields_ = [("batch", _i32), ("q_heads", _i32), ("kv_heads", _i32), ("head_dim", _i32),
                ("capacity", _i32), ("max_seq_len", _i32), ("tail_capacity", _i32),
                ("softmax_scale", ctypes.c_float), ("q_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int)]


# name -> (restype, argtypes), mirroring include/tq.h
SIGNATURES = {
    "tq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tq_version": (ctypes.c_char_p, []),
    "tq_lloyd_max_codebook": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _vp]),
    "tq_rotation_from_gaussian": (ctypes.c_int, [ctypes.c_int, _vp, _vp]),
    "tq_codec_create": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp,
                                       ctypes.POINTER(_vp)]),
    "tq_codec_destroy": (ctypes.c_int, [_vp]),
    "tq_code_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int]),
    "tq_quantize_prod": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _i32, _i32, _i32, _i64, _i64,
                                        _i64, _vp, _vp, tq_prod_cache, _i32, _vp]),
    "tq_quantize_mse": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _i32, _i32, _i32, _i64, _i64,
                                       _i64, _vp, _vp, tq_mse_cache, _i32, _vp]),
    "tq_prod_scores": (ctypes.c_int, [_vp, _vp, _i32, _i64, tq_prod_cache, _i32, _i32, _vp,
                                      _i64, _vp]),
    "tq_decode_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(tq_attn_desc)]),
    "tq_decode_attention": (ctypes.c_int, [ctypes.POINTER(tq_attn_desc), _vp, _vp, _vp,
                                           tq_prod_cache, tq_mse_cache, _vp, _vp, _vp,
                                           ctypes.c_size_t, _vp]),
    "tq_prefill_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(tq_attn_desc), _i32]),
    "tq_prefill_attention": (ctypes.c_int, [ctypes.POINTER(tq_attn_desc), _i32, _i32, _vp, _vp,
                                            _vp, tq_prod_cache, tq_mse_cache, _vp, _vp, _vp,
                                            ctypes.c_size_t, _vp]),
    "tq_decode_step": (ctypes.c_int, [ctypes.POINTER(tq_attn_desc), _vp, _vp, _vp, _vp, _vp,
                                      ctypes.c_int, tq_prod_cache, tq_mse_cache, _vp, _vp, _vp,
                                      _vp, ctypes.c_size_t, _vp]),
    "tq_decode_attention_asym": (ctypes.c_int, [ctypes.POINTER(tq_attn_desc), _vp, _vp, _vp,
                                                tq_mse_cache, _vp, _vp, _vp, _vp, _vp, _vp,
                                                ctypes.c_size_t, _vp]),
    "tq_decode_attention_noalloc": (ctypes.c_int, [ctypes.POINTER(tq_attn_desc), _vp, _vp, _vp,
                                                   tq_prod_cache, tq_mse_cache, _vp, _vp, _vp]),
    "tq_decode_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "tq_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "tq_store_workspace_bytes": (ctypes.c_size_t, [_i32]),
    "tq_attention_quality_scratch_bytes": (ctypes.c_size_t, [_i32, _i32]),
    "tq_attention_quality": (ctypes.c_int, [_vp, _vp, _i32, _vp, ctypes.c_int, tq_prod_cache, _i32,
                                            _i32, ctypes.c_float, _vp, ctypes.c_size_t, _vp, _vp,
                                            _vp, _vp]),
    "tq_store_append": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, ctypes.c_int, _vp, tq_mse_cache,
                                       _i32, _vp, _vp, _i32, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "tq_check_bounded_wait": (ctypes.c_int, [ctypes.c_uint32, _vp]),
}

_lib = None


def load():
    """Loads libtq.so (once).  Raises RuntimeError if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m kv_cache_quantization_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def ptr(x) -> int:
    """Address of a buffer: None -> 0, int -> itself, torch tensor -> data_ptr(), numpy array
    -> its host address."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return x.ctypes.data   # numpy array (host)


class TQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tq_status_string(status)}")


def check(status: int, where: str):
    if status != TQ_OK:
        raise TQError(status, where)
    return status


# ------------------------------------------------------------------ same-name wrappers

def tq_status_string(s: int) -> str:
    return load().tq_status_string(s).decode()


def tq_version() -> str:
    return load().tq_version().decode()


def tq_lloyd_max_codebook(d: int, index_bits: int, centroids) -> int:
    return load().tq_lloyd_max_codebook(d, index_bits, ptr(centroids))


def tq_rotation_from_gaussian(d: int, g, pi) -> int:
    return load().tq_rotation_from_gaussian(d, ptr(g), ptr(pi))


def tq_codec_create(d, kind, bits, pi, s, centroids, out: ctypes.c_void_p) -> int:
    return load().tq_codec_create(d, kind, bits, ptr(pi), ptr(s), ptr(centroids), ctypes.byref(out))


def tq_codec_destroy(codec) -> int:
    return load().tq_codec_destroy(codec)


def tq_code_bytes(kind: int, bits: int) -> int:
    return load().tq_code_bytes(kind, bits)


def tq_quantize_prod(kc, x, x_dtype, batch, heads, tokens, stride_b, stride_h, stride_t, pos,
                     count, cache: tq_prod_cache, capacity, stream) -> int:
    return load().tq_quantize_prod(kc, ptr(x), x_dtype, batch, heads, tokens, stride_b, stride_h,
                                   stride_t, ptr(pos), ptr(count), cache, capacity, ptr(stream))


def tq_quantize_mse(vc, x, x_dtype, batch, heads, tokens, stride_b, stride_h, stride_t, pos,
                    count, cache: tq_mse_cache, capacity, stream) -> int:
    return load().tq_quantize_mse(vc, ptr(x), x_dtype, batch, heads, tokens, stride_b, stride_h,
                                  stride_t, ptr(pos), ptr(count), cache, capacity, ptr(stream))


def tq_prod_scores(kc, q, nq, q_stride, keys: tq_prod_cache, capacity, n, scores, scores_stride,
                   stream) -> int:
    return load().tq_prod_scores(kc, ptr(q), nq, q_stride, keys, capacity, n, ptr(scores),
                                 scores_stride, ptr(stream))


def tq_decode_workspace_bytes(desc: tq_attn_desc) -> int:
    return load().tq_decode_workspace_bytes(ctypes.byref(desc))


def tq_decode_attention(desc: tq_attn_desc, kc, vc, q, k: tq_prod_cache, v: tq_mse_cache,
                        seq_lens, out, workspace, workspace_bytes, stream) -> int:
    return load().tq_decode_attention(ctypes.byref(desc), kc, vc, ptr(q), k, v, ptr(seq_lens),
                                      ptr(out), ptr(workspace), workspace_bytes, ptr(stream))


def tq_prefill_workspace_bytes(desc: tq_attn_desc, n_queries: int) -> int:
    return load().tq_prefill_workspace_bytes(ctypes.byref(desc), n_queries)


def tq_prefill_attention(desc: tq_attn_desc, n_queries, causal, kc, vc, q, k: tq_prod_cache,
                         v: tq_mse_cache, seq_lens, out, workspace, workspace_bytes,
                         stream) -> int:
    return load().tq_prefill_attention(ctypes.byref(desc), n_queries, causal, kc, vc, ptr(q), k, v,
                                       ptr(seq_lens), ptr(out), ptr(workspace), workspace_bytes,
                                       ptr(stream))


def tq_decode_step(desc: tq_attn_desc, kc, vc, q, k_new, v_new, kv_dtype, k: tq_prod_cache,
                   v: tq_mse_cache, pos, lens_out, out, workspace, workspace_bytes,
                   stream) -> int:
    return load().tq_decode_step(ctypes.byref(desc), kc, vc, ptr(q), ptr(k_new), ptr(v_new),
                                 kv_dtype, k, v, ptr(pos), ptr(lens_out), ptr(out),
                                 ptr(workspace), workspace_bytes, ptr(stream))


def tq_decode_attention_asym(desc: tq_attn_desc, vc, q, k_f16, v: tq_mse_cache, seq_lens,
                             k_tail, v_tail, tail_lens, out, workspace, workspace_bytes,
                             stream) -> int:
    return load().tq_decode_attention_asym(ctypes.byref(desc), vc, ptr(q), ptr(k_f16), v,
                                           ptr(seq_lens), ptr(k_tail), ptr(v_tail),
                                           ptr(tail_lens), ptr(out), ptr(workspace),
                                           workspace_bytes, ptr(stream))


def tq_decode_attention_noalloc(desc: tq_attn_desc, kc, vc, q, k: tq_prod_cache,
                                v: tq_mse_cache, seq_lens, out, stream) -> int:
    return load().tq_decode_attention_noalloc(ctypes.byref(desc), kc, vc, ptr(q), k, v,
                                              ptr(seq_lens), ptr(out), ptr(stream))


def tq_decode_noalloc_scratch_bytes() -> int:
    return load().tq_decode_noalloc_scratch_bytes()


def tq_check_bounded_wait(limit_us: int, stream) -> int:
    return load().tq_check_bounded_wait(limit_us, ptr(stream))


def tq_attention_quality_scratch_bytes(nq: int, n: int) -> int:
    return load().tq_attention_quality_scratch_bytes(nq, n)


def tq_attention_quality(kc, q, nq, k, k_dtype, codes: tq_prod_cache, capacity, n, softmax_scale,
                         scratch, scratch_bytes, kl, top1_exact, top1_comp, stream) -> int:
    return load().tq_attention_quality(kc, ptr(q), nq, ptr(k), k_dtype, codes, capacity, n,
                                       softmax_scale, ptr(scratch), scratch_bytes, ptr(kl),
                                       ptr(top1_exact), ptr(top1_comp), ptr(stream))


def tq_store_workspace_bytes(batch: int) -> int:
    return load().tq_store_workspace_bytes(batch)


def tq_store_append(vc, batch, kv_heads, k_new, v_new, dtype, k_f16, v: tq_mse_cache, capacity,
                    k_tail, v_tail, tail_capacity, comp_lens, tail_lens, workspace,
                    workspace_bytes, stream) -> int:
    return load().tq_store_append(vc, batch, kv_heads, ptr(k_new), ptr(v_new), dtype, ptr(k_f16),
                                  v, capacity, ptr(k_tail), ptr(v_tail), tail_capacity,
                                  ptr(comp_lens), ptr(tail_lens), ptr(workspace), workspace_bytes,
                                  ptr(stream))


def tq_device_status():
    flags = ctypes.c_uint32(0)
    st = load().tq_device_status(ctypes.byref(flags))
    return st, flags.value
