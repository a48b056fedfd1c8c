// Quantisation of one vector by one CTA of 512 threads: the path of a decode step's append
// (one new key or value per sequence and KV head), where a whole tile of the tensor-core
// quantiser would idle.  QJL deep-dive §二 steps 1–3 in the unit-sphere domain: y = Π x/‖x‖,
// idx = #{boundaries ≤ y}, ρ = y − c[idx], sign(M ρ) with M = S Πᵀ, ‖r‖ = ‖x‖·‖ρ‖.
//
// Included by the translation units that launch it; each has its own device status word
// g_tq_flags, defined (TQ_DEFINE_FLAGS) before this header is included.  Internal to the
// library.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "append_args.h"
#include "tq_internal.h"

namespace tq {

constexpr int kAppendThreads = 512;

// One vector to quantise into a cache.
struct AppendArgs {
  const void* x;        // the vector's 128 coordinates (dtype), 16-byte aligned
  int dtype;
  int slot;             // slot in the cache row
  long long row;        // cache row: batch·heads + head, or page·heads + head (paged)
  int rowcap;           // slots per cache row
  uint8_t* idx;         // plane-major index codes, or nibbles (nibbles != 0)
  uint8_t* sgn;         // product code: sign plane (null for MSE codes)
  float* xnorm;
  float* rnorm;
  tq_levels lv;
  int ibits;
  int nibbles;
};

// 8 consecutive elements of x (dtype F32, F16 or BF16) from element `off`, as floats.
__device__ __forceinline__ void append_load8(const void* base, int dtype, long long off,
                                             float* out) {
  if (dtype == TQ_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    float4 a = __ldg(p), b = __ldg(p + 1);
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
  } else {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (dtype == TQ_BF16) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      } else {
        __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
        float2 f = __half22float2(h);
        out[2 * i] = f.x;
        out[2 * i + 1] = f.y;
      }
    }
  }
}

// Thread (k quarter q, output j) of the 512 owns T[32q..32q+31][j] of T = Πᵀ or Mᵀ (row-major
// [128][128]); the values are requested at kernel start, before the programmatic wait.
__device__ __forceinline__ void append_load_t(const float* __restrict__ T, float (&t)[32],
                                              int tid) {
  const int j = tid & 127, q = tid >> 7;
#pragma unroll
  for (int k = 0; k < 32; ++k) t[k] = __ldg(&T[(32 * q + k) * TQ_D + j]);
}

// (T v)_j for j = tid < 128 (other threads get 0): four partial sums over k quarters meet in
// `part` [4][128].  Contains two __syncthreads.
__device__ __forceinline__ float append_matvec(const float (&t)[32], const float* v, float* part,
                                               int tid) {
  const int j = tid & 127, q = tid >> 7;
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < 32; ++k) acc = fmaf(t[k], v[32 * q + k], acc);
  part[q * TQ_D + j] = acc;
  __syncthreads();
  float r = 0.f;
  if (tid < TQ_D) r = (part[j] + part[TQ_D + j]) + (part[2 * TQ_D + j] + part[3 * TQ_D + j]);
  __syncthreads();
  return r;
}

// Shared memory of one append CTA.
struct AppendSmem {
  float xs[TQ_D], rho[TQ_D], part[4 * TQ_D];
  float red[4];
};

// Quantises the vector into the cache: every thread of the CTA calls it (it synchronises the
// CTA); tp (and tm for a product code) were loaded by append_load_t.  The caller has mapped
// the position to a.row and a.slot, inside the cache.
template <bool kProd>
__device__ __forceinline__ void append_quantize(const AppendArgs& a, const float (&tp)[32],
                                                const float (&tm)[32], AppendSmem& sm, int tid) {
  float vals[8];
  if (tid < 16) append_load8(a.x, a.dtype, tid * 8, vals);
  const long long slot = a.row * a.rowcap + a.slot;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid < 16) {
#pragma unroll
    for (int e = 0; e < 8; ++e) sm.xs[tid * 8 + e] = vals[e];
  }
  __syncthreads();
  float x2 = 0.f;
  if (tid < TQ_D) x2 = sm.xs[tid] * sm.xs[tid];
  if (warp < 4) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x2 += __shfl_xor_sync(0xffffffffu, x2, o);
    if (lane == 0) sm.red[warp] = x2;
  }
  __syncthreads();
  const float n = sqrtf((sm.red[0] + sm.red[1]) + (sm.red[2] + sm.red[3]));
  const float acc = append_matvec(tp, sm.xs, sm.part, tid);
  int q = 0;
  float r = 0.f;
  if (tid < TQ_D) {
    const float y = n > 0.f ? acc / n : 0.f;
    for (int bnd = 0; bnd < a.lv.levels - 1; ++bnd) q += (a.lv.b[bnd] <= y) ? 1 : 0;
    r = y - a.lv.c[q];
    sm.rho[tid] = r;
  }
  // index codes: warp w < 4 owns coordinates 32w..32w+31
  if (warp < 4) {
    if (a.nibbles) {
      // byte k = idx(2k) | idx(2k+1) << 4: lane pairs combine through a shuffle
      const int other = __shfl_xor_sync(0xffffffffu, q, 1);
      if ((lane & 1) == 0) a.idx[slot * 64 + (tid >> 1)] = (uint8_t)(q | (other << 4));
    } else {
      for (int p = 0; p < a.ibits; ++p) {
        const unsigned word = __ballot_sync(0xffffffffu, (q >> p) & 1);
        if (lane == 0)
          reinterpret_cast<uint32_t*>(
              a.idx + ((a.row * a.ibits + p) * a.rowcap + a.slot) * 16)[warp] = word;
      }
    }
    if (tid == 0) a.xnorm[slot] = n;
  }
  if constexpr (kProd) {
    float r2 = r * r;
    if (warp < 4) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) r2 += __shfl_xor_sync(0xffffffffu, r2, o);
    }
    __syncthreads();   // rho complete; red reused
    if (warp < 4 && lane == 0) sm.red[warp] = r2;
    const float z = append_matvec(tm, sm.rho, sm.part, tid);   // contains __syncthreads
    if (warp < 4) {
      const unsigned word = n > 0.f ? __ballot_sync(0xffffffffu, z >= 0.f) : 0xffffffffu;
      if (lane == 0) reinterpret_cast<uint32_t*>(a.sgn + slot * 16)[warp] = word;
      if (tid == 0) a.rnorm[slot] = n * sqrtf((sm.red[0] + sm.red[1]) + (sm.red[2] + sm.red[3]));
    }
  }
}

// Appends the key (key = true) or the value of (batch b, KV head kvh) with the constants the
// CTA holds: tp = Πᵀ of that codec, tm = Mᵀ for the key.  Called after the programmatic wait by
// every thread of the CTA.
__device__ __forceinline__ void append_unit(const AppendKV& a, bool key, int kvh, int b,
                                            const float (&tp)[32], const float (&tm)[32],
                                            AppendSmem& sm, int tid) {
  const long long bh = (long long)b * a.Hkv + kvh;
  const int pos = a.pos[b];
  if (key && kvh == 0 && tid == 0 && a.lens_out) a.lens_out[b] = pos + 1;
  if (pos < 0 || pos >= a.cap) {
    if (tid == 0) atomicOr(&g_tq_flags, TQ_FLAG_POS_OVERFLOW);
    return;
  }
  AppendArgs aa;
  const tq_rowmap& map = key ? a.kmap : a.vmap;
  if (!tq_map_slot(map, a.Hkv, b, kvh, pos, aa.row, aa.slot)) {
    if (tid == 0) atomicOr(&g_tq_flags, TQ_FLAG_PAGE);
    return;
  }
  aa.rowcap = tq_row_slots(map, a.cap);
  const long long off = bh * TQ_D;
  aa.x = a.dtype == TQ_F32
             ? static_cast<const void*>(static_cast<const float*>(key ? a.k_new : a.v_new) + off)
             : static_cast<const void*>(static_cast<const uint16_t*>(key ? a.k_new : a.v_new) + off);
  aa.dtype = a.dtype;
  if (key) {
    aa.idx = a.kidx; aa.sgn = a.ksgn; aa.xnorm = a.kxn; aa.rnorm = a.krn;
    aa.lv = a.klv; aa.ibits = a.kbits; aa.nibbles = 0;
    append_quantize<true>(aa, tp, tm, sm, tid);
  } else {
    aa.idx = a.vidx; aa.sgn = nullptr; aa.xnorm = a.vxn; aa.rnorm = nullptr;
    aa.lv = a.vlv; aa.ibits = a.vbits; aa.nibbles = a.v_nibbles;
    append_quantize<false>(aa, tp, tm, sm, tid);
  }
}

// One CTA of 512 threads appends the key (key = true) or the value of (batch b, KV head kvh).
// The codec's constants are requested before the programmatic wait, everything the previous
// kernel in the stream may write (the vectors, the positions, the caches) after it.
__device__ __forceinline__ void append_kv_role(const AppendKV& a, bool key, int kvh, int b) {
  __shared__ AppendSmem sm;
  const int tid = threadIdx.x;
  float tp[32], tm[32];
  append_load_t(key ? a.kpiT : a.vpiT, tp, tid);
  if (key) append_load_t(a.kmT, tm, tid);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  append_unit(a, key, kvh, b, tp, tm, sm, tid);
}

// Shared memory of a CTA that appends a key and a value together.
struct AppendPairSmem {
  float xs[2][TQ_D], rho[TQ_D], part[2][4 * TQ_D];
  float red[8];
  float lb[2][16], lc[2][16];   // boundaries and centroids: [0] key codec, [1] value codec
};

// Fills the codebooks of the two codecs into shared memory (constant indices, so the kernel
// parameters are read in place); the caller synchronises before they are used.
__device__ __forceinline__ void append_pair_levels(const AppendKV& a, AppendPairSmem& sm,
                                                   int tid) {
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      sm.lb[0][i] = a.klv.b[i]; sm.lc[0][i] = a.klv.c[i];
      sm.lb[1][i] = a.vlv.b[i]; sm.lc[1][i] = a.vlv.c[i];
    }
  }
}

// The key and the value of (batch b, KV head kvh) quantised together when the two codecs share
// Π (tp = Πᵀ, tm = Mᵀ of the key codec): one pass over tp rotates both vectors, and the value's
// cells and codes (warps 4–7) proceed beside the key's (warps 0–3).  Each side's arithmetic is,
// operation for operation, that of append_quantize, so the codes and norms are the same bits as
// two single appends.  Every thread of the CTA calls it after the programmatic wait and after
// append_pair_levels; it synchronises the CTA.
__device__ __forceinline__ void append_pair(const AppendKV& a, int kvh, int b,
                                            const float (&tp)[32], const float (&tm)[32],
                                            AppendPairSmem& sm, int tid) {
  const long long bh = (long long)b * a.Hkv + kvh;
  const int pos = a.pos[b];
  if (kvh == 0 && tid == 0 && a.lens_out) a.lens_out[b] = pos + 1;
  if (pos < 0 || pos >= a.cap) {
    if (tid == 0) atomicOr(&g_tq_flags, TQ_FLAG_POS_OVERFLOW);
    return;
  }
  long long krow, vrow;
  int kslot, vslot;
  const bool kok = tq_map_slot(a.kmap, a.Hkv, b, kvh, pos, krow, kslot);
  const bool vok = tq_map_slot(a.vmap, a.Hkv, b, kvh, pos, vrow, vslot);
  if (!kok || !vok) {
    if (tid == 0) atomicOr(&g_tq_flags, TQ_FLAG_PAGE);
    return;
  }
  const int krc = tq_row_slots(a.kmap, a.cap), vrc = tq_row_slots(a.vmap, a.cap);
  const int warp = tid >> 5, lane = tid & 31;
  const int side = warp >> 2;   // for tid < 256: 0 the key's coordinates, 1 the value's
  const long long off = bh * TQ_D;
  const long long kslot_all = krow * krc + kslot, vslot_all = vrow * vrc + vslot;
  if (tid < 32) {
    const void* base = tid < 16 ? a.k_new : a.v_new;
    const void* x = a.dtype == TQ_F32
                        ? static_cast<const void*>(static_cast<const float*>(base) + off)
                        : static_cast<const void*>(static_cast<const uint16_t*>(base) + off);
    float vals[8];
    append_load8(x, a.dtype, (tid & 15) * 8, vals);
#pragma unroll
    for (int e = 0; e < 8; ++e) sm.xs[tid >> 4][(tid & 15) * 8 + e] = vals[e];
  }
  __syncthreads();
  if (warp < 8) {
    const float xv = sm.xs[side][tid & (TQ_D - 1)];
    float x2 = xv * xv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x2 += __shfl_xor_sync(0xffffffffu, x2, o);
    if (lane == 0) sm.red[warp] = x2;
  }
  __syncthreads();
  const int j = tid & (TQ_D - 1), kq = tid >> 7;
  float acc_k = 0.f, acc_v = 0.f;
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    acc_k = fmaf(tp[k], sm.xs[0][32 * kq + k], acc_k);
    acc_v = fmaf(tp[k], sm.xs[1][32 * kq + k], acc_v);
  }
  sm.part[0][kq * TQ_D + j] = acc_k;
  sm.part[1][kq * TQ_D + j] = acc_v;
  __syncthreads();
  int q = 0;
  float r = 0.f, n = 0.f;
  if (warp < 8) {
    const float* red = sm.red + 4 * side;
    n = sqrtf((red[0] + red[1]) + (red[2] + red[3]));
    const float* pt = sm.part[side];
    const float acc = (pt[j] + pt[TQ_D + j]) + (pt[2 * TQ_D + j] + pt[3 * TQ_D + j]);
    const float y = n > 0.f ? acc / n : 0.f;
    const int nb = (side ? a.vlv.levels : a.klv.levels) - 1;
    const float* lb = sm.lb[side];
#pragma unroll
    for (int bnd = 0; bnd < 15; ++bnd) q += (bnd < nb && lb[bnd] <= y) ? 1 : 0;
    r = y - sm.lc[side][q];
    if (side == 0) sm.rho[j] = r;
    // index codes: warp w owns coordinates 32(w mod 4) .. 32(w mod 4) + 31 of its side
    if (side == 1 && a.v_nibbles) {
      const int other = __shfl_xor_sync(0xffffffffu, q, 1);
      if ((lane & 1) == 0) a.vidx[vslot_all * 64 + (j >> 1)] = (uint8_t)(q | (other << 4));
    } else {
      const int ib = side ? a.vbits : a.kbits;
      uint8_t* idx = side ? a.vidx : a.kidx;
      const long long row = side ? vrow : krow;
      const int rc = side ? vrc : krc, sl = side ? vslot : kslot;
      for (int p = 0; p < ib; ++p) {
        const unsigned word = __ballot_sync(0xffffffffu, (q >> p) & 1);
        if (lane == 0)
          reinterpret_cast<uint32_t*>(idx + ((row * ib + p) * rc + sl) * 16)[warp & 3] = word;
      }
    }
    if (j == 0) (side ? a.vxn : a.kxn)[side ? vslot_all : kslot_all] = n;
  }
  // the key's residual: ‖ρ‖² and the signs of M ρ
  float r2 = r * r;
  if (warp < 4) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r2 += __shfl_xor_sync(0xffffffffu, r2, o);
  }
  __syncthreads();   // rho complete; red reused
  if (warp < 4 && lane == 0) sm.red[warp] = r2;
  const float z = append_matvec(tm, sm.rho, sm.part[0], tid);   // contains __syncthreads
  if (warp < 4) {
    const unsigned word = n > 0.f ? __ballot_sync(0xffffffffu, z >= 0.f) : 0xffffffffu;
    if (lane == 0) reinterpret_cast<uint32_t*>(a.ksgn + kslot_all * 16)[warp] = word;
    if (tid == 0) a.krn[kslot_all] = n * sqrtf((sm.red[0] + sm.red[1]) + (sm.red[2] + sm.red[3]));
  }
}

// One CTA of 512 threads appends the key and the value of (batch b, KV head kvh), the codecs
// sharing Π; the constants are requested before the programmatic wait.
__device__ __forceinline__ void append_kv_pair_role(const AppendKV& a, int kvh, int b) {
  __shared__ AppendPairSmem sm;
  const int tid = threadIdx.x;
  float tp[32], tm[32];
  append_load_t(a.kpiT, tp, tid);
  append_load_t(a.kmT, tm, tid);
  append_pair_levels(a, sm, tid);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();
  append_pair(a, kvh, b, tp, tm, sm, tid);
}

// The appends of `units` (batch, KV head) pairs, unit u = b·Hkv + kvh, by a grid of CTAs that
// each take units blockIdx.x, blockIdx.x + gridDim.x, ...  A CTA loads Πᵀ and Mᵀ of the key
// codec once.  When the value codec shares Π it quantises each unit's key and value together;
// otherwise it appends its units' keys, loads the value codec's Πᵀ and appends their values.
__device__ __forceinline__ void append_kv_units(const AppendKV& a, int units) {
  __shared__ union {
    AppendSmem one;
    AppendPairSmem pair;
  } sm;
  const int tid = threadIdx.x;
  float tp[32], tm[32];
  append_load_t(a.kpiT, tp, tid);
  append_load_t(a.kmT, tm, tid);
  if (a.shared_pi) append_pair_levels(a, sm.pair, tid);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (a.shared_pi) {
    __syncthreads();
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      append_pair(a, u % a.Hkv, u / a.Hkv, tp, tm, sm.pair, tid);
      __syncthreads();   // the shared scratch is reused
    }
    return;
  }
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    append_unit(a, true, u % a.Hkv, u / a.Hkv, tp, tm, sm.one, tid);
    __syncthreads();
  }
  append_load_t(a.vpiT, tp, tid);
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    append_unit(a, false, u % a.Hkv, u / a.Hkv, tp, tm, sm.one, tid);
    __syncthreads();
  }
}

}  // namespace tq
