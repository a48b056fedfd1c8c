// Append path of a KV cache kept as a compressed part plus an FP16 tail of recent tokens.
//
// The pages' store keeps the most recent tokens in full precision and compresses history in
// chunks (QJL deep-dive §六: chunked append into the compressed store, recent tokens in a
// full-precision ring; MLX-port article, quick start: `min_compress_tokens`, 256 by default,
// and the asymmetric mode `key_bits=0`: keys stay FP16, values TurboQuant-MSE).  Here a
// sequence's tail has `tail_capacity` slots; each append writes the new key and value into
// the next slot, and the append that fills the last slot compacts the whole tail: its keys are
// copied into the FP16 key array and its values MSE-quantised into the value cache, both at the
// end of the compressed part, and the tail starts empty again.  Decode attention
// (tq_decode_attention_asym) attends the compressed part and the tail in one softmax.
//
// Per call, all on the caller's stream: the tail append (it also marks which sequences compact),
// the value compaction (the tile quantiser, whose tiles of sequences that do not compact leave
// at once), the key copy, and the length update.
#include <cuda_fp16.h>

#include "tq_internal.h"

TQ_DEFINE_FLAGS(tq_take_flags_store)

namespace {

struct StoreArgs {
  int B, Hkv, cap, T;          // batch, KV heads, compressed capacity, tail slots
  const void* k_new;           // [B][Hkv][128] of dtype
  const void* v_new;
  int dtype;
  __half* k_f16;               // [B][Hkv][cap][128]
  __half* k_tail;              // [B][Hkv][T][128]
  __half* v_tail;
  const int* comp_lens;        // [B]
  const int* tail_lens;        // [B]
  int* count;                  // [B] (workspace): T where the tail compacts this call, else 0
};

__device__ __forceinline__ float load_one(const void* base, int dtype, long long i) {
  if (dtype == TQ_F32) return static_cast<const float*>(base)[i];
  const uint16_t u = static_cast<const uint16_t*>(base)[i];
  if (dtype == TQ_BF16) return __uint_as_float((uint32_t)u << 16);
  return __half2float(__ushort_as_half(u));
}

// Grid (Hkv, B), 128 threads (one per coordinate): the new key and value into tail slot
// tail_lens[b], as FP16; the (b, 0) CTA marks whether b's tail is full after this append.
__global__ void __launch_bounds__(128) tail_append_kernel(const StoreArgs a) {
  const int h = blockIdx.x, b = blockIdx.y, j = threadIdx.x;
  const int slot = a.tail_lens[b];
  const int comp = a.comp_lens[b];
  const bool full = slot + 1 == a.T;
  if (slot < 0 || slot >= a.T || comp < 0 || (full && comp + a.T > a.cap)) {
    // a tail length out of range, or a compaction past the compressed capacity: nothing is
    // written for this sequence
    if (j == 0 && h == 0) {
      a.count[b] = 0;
      atomicOr(&g_tq_flags, TQ_FLAG_LEN_OVERFLOW);
    }
    return;
  }
  const long long bh = (long long)b * a.Hkv + h;
  const long long dst = (bh * a.T + slot) * TQ_D + j;
  a.k_tail[dst] = __float2half_rn(load_one(a.k_new, a.dtype, bh * TQ_D + j));
  a.v_tail[dst] = __float2half_rn(load_one(a.v_new, a.dtype, bh * TQ_D + j));
  if (h == 0 && j == 0) a.count[b] = full ? a.T : 0;
}

// Grid (T / 8, Hkv, B), 128 threads: where b compacts, rows t of its tail keys go to the FP16
// key array at comp_lens[b] + t (16-byte copies; 8 rows a CTA).
__global__ void __launch_bounds__(128) tail_keys_kernel(const StoreArgs a) {
  const int h = blockIdx.y, b = blockIdx.z;
  if (a.count[b] == 0) return;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 4), part = threadIdx.x & 15;
  const long long bh = (long long)b * a.Hkv + h;
  const int dst = a.comp_lens[b] + t;
  const uint4* src = reinterpret_cast<const uint4*>(a.k_tail + (bh * a.T + t) * TQ_D) + part;
  uint4* out = reinterpret_cast<uint4*>(a.k_f16 + (bh * a.cap + dst) * TQ_D) + part;
  *out = *src;
}

// One thread per sequence: the compressed part grows by T where the tail compacted, and the
// tail restarts empty; elsewhere the tail grows by one.
__global__ void tail_lens_kernel(const int* count, int n, int* comp_lens, int* tail_lens,
                                 int T) {
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < n; b += gridDim.x * blockDim.x) {
    const int slot = tail_lens[b];
    if (slot < 0 || slot >= T) continue;   // flagged by the append
    if (count[b] == T) {
      comp_lens[b] += T;
      tail_lens[b] = 0;
    } else if (slot + 1 < T) {
      tail_lens[b] = slot + 1;
    }   // else: a full tail that could not compact (flagged); the token was not stored
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" size_t tq_store_workspace_bytes(int32_t batch) {
  return batch > 0 ? ((size_t)batch * sizeof(int) + 255) / 256 * 256 : 0;
}

extern "C" tq_status tq_store_append(const tq_codec* vc, int32_t batch, int32_t kv_heads,
                                     const void* k_new, const void* v_new, tq_dtype dtype,
                                     uint16_t* k_f16, tq_mse_cache v, int32_t capacity,
                                     uint16_t* k_tail, uint16_t* v_tail, int32_t tail_capacity,
                                     int32_t* comp_lens, int32_t* tail_lens, void* workspace,
                                     size_t workspace_bytes, tq_stream_t stream_) {
  tq_status st = tq_check_codec(vc, TQ_MSE);
  if (st != TQ_OK) return st;
  if (batch < 0 || kv_heads <= 0) return TQ_ERR_INVALID_ARG;
  if (v.pages) return TQ_ERR_UNSUPPORTED;   // the store keeps a flat value cache
  if (capacity <= 0 || capacity % TQ_CAPACITY_ALIGN) return TQ_ERR_INVALID_ARG;
  if (tail_capacity <= 0 || tail_capacity % 8) return TQ_ERR_INVALID_ARG;
  if (dtype != TQ_F32 && dtype != TQ_F16 && dtype != TQ_BF16) return TQ_ERR_UNSUPPORTED;
  if (!k_new || !v_new || !k_f16 || !v.idx || !v.xnorm || !k_tail || !v_tail || !comp_lens ||
      !tail_lens || !workspace)
    return TQ_ERR_INVALID_ARG;
  if (!aligned16(k_f16) || !aligned16(k_tail) || !aligned16(v_tail) || !aligned16(v.idx) ||
      !aligned16(v.xnorm))
    return TQ_ERR_INVALID_ARG;
  if (workspace_bytes < tq_store_workspace_bytes(batch)) return TQ_ERR_INVALID_ARG;
  if (batch == 0) return TQ_OK;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  StoreArgs a{};
  a.B = batch; a.Hkv = kv_heads; a.cap = capacity; a.T = tail_capacity;
  a.k_new = k_new; a.v_new = v_new; a.dtype = dtype;
  a.k_f16 = reinterpret_cast<__half*>(k_f16);
  a.k_tail = reinterpret_cast<__half*>(k_tail);
  a.v_tail = reinterpret_cast<__half*>(v_tail);
  a.comp_lens = comp_lens; a.tail_lens = tail_lens;
  a.count = static_cast<int*>(workspace);
  tail_append_kernel<<<dim3(kv_heads, batch), 128, 0, stream>>>(a);
  if ((st = tq_cuda_status(cudaGetLastError())) != TQ_OK) return st;
  // values of the sequences that compact: the whole tail, MSE-coded at comp_lens[b] + t
  const long long hs = (long long)tail_capacity * TQ_D;
  st = tq_launch_quantize_tiles(vc, false, v_tail, TQ_F16, batch, kv_heads, tail_capacity,
                                kv_heads * hs, hs, TQ_D, comp_lens, a.count, v.idx, nullptr,
                                v.xnorm, nullptr, capacity, stream);
  if (st != TQ_OK) return st;
  tail_keys_kernel<<<dim3(tail_capacity / 8, kv_heads, batch), 128, 0, stream>>>(a);
  tail_lens_kernel<<<(batch + 127) / 128, 128, 0, stream>>>(a.count, batch, comp_lens, tail_lens,
                                                             tail_capacity);
  return tq_cuda_status(cudaGetLastError());
}
