// Quantisation kernels: TurboQuant-prod for keys and TurboQuant-MSE for values.
//
// QJL deep-dive §二: (1) store ‖x‖ and rotate x/‖x‖ by Π; (2) per-coordinate Lloyd-Max
// boundary lookup; (3) sketch the residual with S, keep sign bits and ‖r‖.  The kernel
// keeps everything in the unit-sphere domain: y = Π x / ‖x‖, ρ = y − c[idx],
// ‖r‖ = ‖x‖·‖ρ‖ and sign(S r) = sign(M ρ) with M = S Πᵀ precomputed by the codec.
//
// Layout of one CTA (256 threads) working on a tile of 64 vectors:
//   thread (vg = tid / 16, jg = tid % 16) owns vectors 4vg..4vg+3 and output coordinates
//   8jg..8jg+7, so after each 64×128×128 product it holds exactly one byte of every code
//   plane (coordinates 8jg..8jg+7) of its four vectors and writes codes without a
//   shuffle.  Πᵀ and Mᵀ stay resident in shared memory for the CTA's lifetime
//   (persistent grid over tiles).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <climits>

#include "tq_internal.h"

TQ_DEFINE_FLAGS(tq_take_flags_quantize)

#include "append_small.h"

namespace {

constexpr int kTile = 64;       // vectors per tile
constexpr int kThreads = 256;
constexpr int kXStride = 132;   // padded row stride (floats) of the activation tile

struct QuantArgs {
  const void* x;
  int dtype;
  int batch, heads, tokens;
  long long sb, sh, st;
  const int* pos;
  const int* count;
  uint8_t* idx;
  uint8_t* sgn;
  float* xnorm;
  float* rnorm;
  int capacity;    // slots per sequence
  tq_rowmap map;   // flat, or the pool's block table
  int rowcap;      // slots per cache row: capacity (flat) or page_tokens (paged)
  const float* piT;
  const float* mT;
  tq_levels lv;
  int ibits;
  int nibbles;
  int sparse;      // one tile per CTA; a tile without a vector to write leaves at once
};

__device__ __forceinline__ void load8(const void* base, int dtype, long long off, float* out) {
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

// acc[i][o] = Σ_k X[4vg+i][k] · T[k][8jg+o]   (T = Πᵀ or Mᵀ, both [128][128] in smem)
__device__ __forceinline__ void tile_gemm(const float* __restrict__ X, const float* __restrict__ T,
                                          int vg, int jg, float acc[4][8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int o = 0; o < 8; ++o) acc[i][o] = 0.f;
#pragma unroll 2
  for (int k = 0; k < TQ_D; k += 4) {
    float4 xv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      xv[i] = *reinterpret_cast<const float4*>(&X[(4 * vg + i) * kXStride + k]);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float4 p0 = *reinterpret_cast<const float4*>(&T[(k + kk) * TQ_D + 8 * jg]);
      const float4 p1 = *reinterpret_cast<const float4*>(&T[(k + kk) * TQ_D + 8 * jg + 4]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = kk == 0 ? xv[i].x : kk == 1 ? xv[i].y : kk == 2 ? xv[i].z : xv[i].w;
        acc[i][0] = fmaf(a, p0.x, acc[i][0]);
        acc[i][1] = fmaf(a, p0.y, acc[i][1]);
        acc[i][2] = fmaf(a, p0.z, acc[i][2]);
        acc[i][3] = fmaf(a, p0.w, acc[i][3]);
        acc[i][4] = fmaf(a, p1.x, acc[i][4]);
        acc[i][5] = fmaf(a, p1.y, acc[i][5]);
        acc[i][6] = fmaf(a, p1.z, acc[i][6]);
        acc[i][7] = fmaf(a, p1.w, acc[i][7]);
      }
    }
  }
}

template <bool kProd>
__global__ void __launch_bounds__(kThreads) quantize_kernel(QuantArgs a) {
  extern __shared__ __align__(16) float smem[];
  float* PT = smem;
  float* MT = PT + TQ_D * TQ_D;
  float* X = kProd ? MT + TQ_D * TQ_D : MT;
  __shared__ float s_norm[kTile];
  __shared__ int s_dst[kTile];         // destination slot in its cache row, -1 = skip
  __shared__ long long s_row[kTile];   // destination cache row

  const int tid = threadIdx.x;
  if (a.sparse) {
    // (the caller launches one CTA per tile) most tiles have nothing to write: leave before
    // fetching the codec's constants
    __shared__ int s_any;
    if (tid == 0) s_any = 0;
    __syncthreads();
    if (tid < kTile) {
      const long long i = (long long)blockIdx.x * kTile + tid;
      if (i < (long long)a.batch * a.heads * a.tokens) {
        const int t = (int)(i % a.tokens);
        const int b = (int)(i / a.tokens) / a.heads;
        if (t < (a.count ? a.count[b] : a.tokens)) s_any = 1;
      }
    }
    __syncthreads();
    if (!s_any) return;
  }
  for (int i = tid; i < TQ_D * TQ_D / 4; i += kThreads) {
    reinterpret_cast<float4*>(PT)[i] = __ldg(reinterpret_cast<const float4*>(a.piT) + i);
    if (kProd) reinterpret_cast<float4*>(MT)[i] = __ldg(reinterpret_cast<const float4*>(a.mT) + i);
  }

  const long long total = (long long)a.batch * a.heads * a.tokens;
  const long long ntiles = (total + kTile - 1) / kTile;
  const int vg = tid / 16, jg = tid % 16;

  for (long long tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    __syncthreads();  // previous tile fully consumed (and Πᵀ/Mᵀ loaded on the first pass)
    if (tid < kTile) {
      const long long i = tile * kTile + tid;
      int dst = -1;
      long long row = 0;
      if (i < total) {
        const int t = (int)(i % a.tokens);
        const int bh = (int)(i / a.tokens);
        const int b = bh / a.heads;
        const int cnt = a.count ? a.count[b] : a.tokens;
        if (t < cnt) {
          const int p = (a.pos ? a.pos[b] : 0) + t;
          if (p < 0 || p >= a.capacity) atomicOr(&g_tq_flags, TQ_FLAG_POS_OVERFLOW);
          else if (!tq_map_slot(a.map, a.heads, b, bh - b * a.heads, p, row, dst)) {
            atomicOr(&g_tq_flags, TQ_FLAG_PAGE);
            dst = -1;
          }
        }
      }
      s_dst[tid] = dst;
      s_row[tid] = row;
    }
    // activation tile: 64 vectors × 16 chunks of 8 elements
    for (int c = tid; c < kTile * 16; c += kThreads) {
      const int v = c / 16, part = c % 16;
      const long long i = tile * kTile + v;
      float vals[8];
      if (i < total) {
        const int t = (int)(i % a.tokens);
        const int bh = (int)(i / a.tokens);
        const int b = bh / a.heads, h = bh % a.heads;
        load8(a.x, a.dtype, b * a.sb + h * a.sh + t * a.st + part * 8, vals);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) vals[e] = 0.f;
      }
      float4* dstp = reinterpret_cast<float4*>(&X[v * kXStride + part * 8]);
      dstp[0] = make_float4(vals[0], vals[1], vals[2], vals[3]);
      dstp[1] = make_float4(vals[4], vals[5], vals[6], vals[7]);
    }
    __syncthreads();
    {  // ‖x‖: warp w handles vectors 8w..8w+7
      const int w = tid / 32, lane = tid % 32;
      for (int v = 8 * w; v < 8 * w + 8; ++v) {
        const float4 q = *reinterpret_cast<const float4*>(&X[v * kXStride + 4 * lane]);
        float s = q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) s_norm[v] = sqrtf(s);
      }
    }
    __syncthreads();

    float acc[4][8];
    tile_gemm(X, PT, vg, jg, acc);

    int idx[4][8];
    float ss[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float n = s_norm[4 * vg + i];
      ss[i] = 0.f;
#pragma unroll
      for (int o = 0; o < 8; ++o) {
        const float y = n > 0.f ? acc[i][o] / n : 0.f;
        int q = 0;
        for (int bnd = 0; bnd < a.lv.levels - 1; ++bnd) q += (a.lv.b[bnd] <= y) ? 1 : 0;
        idx[i][o] = q;
        const float r = y - a.lv.c[q];
        acc[i][o] = r;
        ss[i] = fmaf(r, r, ss[i]);
      }
    }
    // write codes of the MSE stage
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v = 4 * vg + i;
      const int dst = s_dst[v];
      if (dst < 0) continue;
      const long long slot = s_row[v] * a.rowcap + dst;
      if (a.nibbles) {
        uint32_t word = 0;
#pragma unroll
        for (int o = 0; o < 8; ++o) word |= (uint32_t)idx[i][o] << (4 * o);
        reinterpret_cast<uint32_t*>(a.idx + slot * 64)[jg] = word;
      } else {
        for (int p = 0; p < a.ibits; ++p) {
          uint32_t byte = 0;
#pragma unroll
          for (int o = 0; o < 8; ++o) byte |= (uint32_t)((idx[i][o] >> p) & 1) << o;
          a.idx[((s_row[v] * a.ibits + p) * a.rowcap + dst) * 16 + jg] = (uint8_t)byte;
        }
      }
      if (jg == 0) a.xnorm[slot] = s_norm[v];
    }
    if constexpr (kProd) {
    // ‖ρ‖ over the 16 threads sharing the vector group (lanes differing in bits 0..3)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], off);
    __syncthreads();  // all threads finished reading X for the rotation product
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4* dstp = reinterpret_cast<float4*>(&X[(4 * vg + i) * kXStride + 8 * jg]);
      dstp[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      dstp[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
    __syncthreads();
    float z[4][8];
    tile_gemm(X, MT, vg, jg, z);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v = 4 * vg + i;
      const int dst = s_dst[v];
      if (dst < 0) continue;
      const float n = s_norm[v];
      uint32_t byte = 0;
#pragma unroll
      for (int o = 0; o < 8; ++o) byte |= (uint32_t)(z[i][o] >= 0.f) << o;
      if (!(n > 0.f)) byte = 0xffu;   // zero vector: zero residual, all signs +1
      const long long slot = s_row[v] * a.rowcap + dst;
      a.sgn[slot * 16 + jg] = (uint8_t)byte;
      if (jg == 0) a.rnorm[slot] = n * sqrtf(ss[i]);
    }
    }  // kProd
  }
}

// Few vectors (a decode step appends one token per sequence and head): one CTA of 512
// threads per vector.  Each 128×128 product is split four ways over k, so every thread
// issues 32 independent coalesced loads of Πᵀ (or Mᵀ) from L2 instead of a 128-long chain;
// codes are assembled with warp ballots.
template <bool kProd>
__global__ void __launch_bounds__(tq::kAppendThreads) quantize_small_kernel(QuantArgs a) {
  __shared__ tq::AppendSmem sm;
  const int tid = threadIdx.x;
  const long long i = blockIdx.x;
  const int t = (int)(i % a.tokens);
  const int bh = (int)(i / a.tokens);
  const int b = bh / a.heads, h = bh % a.heads;
  // Launched as a programmatic-launch secondary of the previous kernel in the stream: the
  // codec's constants (Πᵀ, Mᵀ) are requested at once, everything the previous kernel may
  // produce or read (the vector, the count, the position, the cache) only after it completed.
  float tp[32], tm[32];
  tq::append_load_t(a.piT, tp, tid);
  if constexpr (kProd) tq::append_load_t(a.mT, tm, tid);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int cnt = a.count ? a.count[b] : a.tokens;
  const int pos = a.pos ? a.pos[b] : 0;
  if (t >= cnt) return;
  const int dst = pos + t;
  if (dst < 0 || dst >= a.capacity) {
    if (tid == 0) atomicOr(&g_tq_flags, TQ_FLAG_POS_OVERFLOW);
    return;
  }
  tq::AppendArgs aa;
  if (!tq_map_slot(a.map, a.heads, b, h, dst, aa.row, aa.slot)) {
    if (tid == 0) atomicOr(&g_tq_flags, TQ_FLAG_PAGE);
    return;
  }
  aa.x = a.dtype == TQ_F32
             ? static_cast<const void*>(static_cast<const float*>(a.x) + b * a.sb + h * a.sh + t * a.st)
             : static_cast<const void*>(static_cast<const uint16_t*>(a.x) + b * a.sb + h * a.sh + t * a.st);
  aa.dtype = a.dtype;
  aa.rowcap = a.rowcap;
  aa.idx = a.idx;
  aa.sgn = a.sgn;
  aa.xnorm = a.xnorm;
  aa.rnorm = a.rnorm;
  aa.lv = a.lv;
  aa.ibits = a.ibits;
  aa.nibbles = a.nibbles;
  tq::append_quantize<kProd>(aa, tp, tm, sm, tid);
}

// The appends of a decode step in one launch: at most one CTA per SM, each taking every
// gridDim.x-th (batch, KV head) unit, key and value, with one load of the codecs' constants.
__global__ void __launch_bounds__(tq::kAppendThreads, 1)
    append_kv_kernel(const tq::AppendKV a, int units) {
  tq::append_kv_units(a, units);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tq_status check_x(const void* x, tq_dtype dt, int batch, int heads, int tokens, long long sb,
                  long long sh, long long st, int capacity) {
  if (!x) return TQ_ERR_INVALID_ARG;
  if (dt != TQ_F32 && dt != TQ_F16 && dt != TQ_BF16) return TQ_ERR_UNSUPPORTED;
  if (batch < 0 || heads < 0 || tokens < 0 || sb < 0 || sh < 0 || st < 0) return TQ_ERR_INVALID_ARG;
  if (capacity <= 0 || capacity % TQ_CAPACITY_ALIGN) return TQ_ERR_INVALID_ARG;
  const long long elem_align = dt == TQ_F32 ? 4 : 8;   // 16-byte aligned vector starts
  if (!aligned16(x) || sb % elem_align || sh % elem_align || st % elem_align) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

// Tiles of bf16 / fp16 vectors go to the tensor-core kernel (quantize_tc.cu); fp32 inputs
// and the few vectors of a decode step stay on the kernels above.
bool use_tensor_cores(tq_dtype dt, int batch, int heads, int tokens) {
  const long long total = (long long)batch * heads * tokens;
  const int sms = tq_num_sms();
  return tq_quantize_tc_supported(dt) && total > 2LL * (sms > 0 ? sms : 148);
}

template <bool kProd>
tq_status launch(const QuantArgs& a, cudaStream_t stream) {
  const long long total = (long long)a.batch * a.heads * a.tokens;
  if (total == 0) return TQ_OK;
  const int sms = tq_num_sms();
  if (total <= 2LL * (sms > 0 ? sms : 148)) {
    // programmatic launch: this kernel's start overlaps the end of the previous one
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)total);
    cfg.blockDim = dim3(tq::kAppendThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, quantize_small_kernel<kProd>, a) != cudaSuccess) return TQ_ERR_CUDA;
    return tq_cuda_status(cudaGetLastError());
  }
  const size_t smem = (size_t)(kProd ? 2 : 1) * TQ_D * TQ_D * sizeof(float) +
                      (size_t)kTile * kXStride * sizeof(float);
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return TQ_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(quantize_kernel<kProd>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    configured[dev] = true;
  }
  const long long ntiles = (total + kTile - 1) / kTile;
  const long long per_sm = kProd ? 1 : 2;
  const int grid = (int)(ntiles < sms * per_sm ? ntiles : sms * per_sm);
  quantize_kernel<kProd><<<grid, kThreads, smem, stream>>>(a);
  return tq_cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" tq_status tq_quantize_prod(const tq_codec* kc, const void* x, tq_dtype x_dtype,
                                      int32_t batch, int32_t heads, int32_t tokens,
                                      int64_t stride_b, int64_t stride_h, int64_t stride_t,
                                      const int32_t* pos, const int32_t* count,
                                      tq_prod_cache cache, int32_t capacity, tq_stream_t stream) {
  tq_status st = tq_check_codec(kc, TQ_PROD);
  if (st != TQ_OK) return st;
  st = check_x(x, x_dtype, batch, heads, tokens, stride_b, stride_h, stride_t, capacity);
  if (st != TQ_OK) return st;
  if (!cache.idx || !cache.sgn || !cache.xnorm || !cache.rnorm) return TQ_ERR_INVALID_ARG;
  if (!aligned16(cache.idx) || !aligned16(cache.sgn) || !aligned16(cache.xnorm) ||
      !aligned16(cache.rnorm))
    return TQ_ERR_INVALID_ARG;
  tq_rowmap map;
  if ((st = tq_rowmap_of(cache.pages, capacity, &map)) != TQ_OK) return st;
  if (use_tensor_cores(x_dtype, batch, heads, tokens))
    return tq_launch_quantize_tc(true, x, x_dtype, batch, heads, tokens, stride_b, stride_h,
                                 stride_t, pos, count, cache.idx, cache.sgn, cache.xnorm,
                                 cache.rnorm, capacity, map, kc,
                                 reinterpret_cast<cudaStream_t>(stream));
  QuantArgs a{};
  a.x = x; a.dtype = x_dtype; a.batch = batch; a.heads = heads; a.tokens = tokens;
  a.sb = stride_b; a.sh = stride_h; a.st = stride_t; a.pos = pos; a.count = count;
  a.idx = cache.idx; a.sgn = cache.sgn; a.xnorm = cache.xnorm; a.rnorm = cache.rnorm;
  a.capacity = capacity; a.map = map; a.rowcap = tq_row_slots(map, capacity);
  a.piT = kc->d_piT; a.mT = kc->d_mT; a.lv = tq_make_levels(kc);
  a.ibits = kc->ibits; a.nibbles = 0;
  return launch<true>(a, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" tq_status tq_quantize_mse(const tq_codec* vc, const void* x, tq_dtype x_dtype,
                                     int32_t batch, int32_t heads, int32_t tokens,
                                     int64_t stride_b, int64_t stride_h, int64_t stride_t,
                                     const int32_t* pos, const int32_t* count,
                                     tq_mse_cache cache, int32_t capacity, tq_stream_t stream) {
  tq_status st = tq_check_codec(vc, TQ_MSE);
  if (st != TQ_OK) return st;
  st = check_x(x, x_dtype, batch, heads, tokens, stride_b, stride_h, stride_t, capacity);
  if (st != TQ_OK) return st;
  if (!cache.idx || !cache.xnorm) return TQ_ERR_INVALID_ARG;
  if (!aligned16(cache.idx) || !aligned16(cache.xnorm)) return TQ_ERR_INVALID_ARG;
  tq_rowmap map;
  if ((st = tq_rowmap_of(cache.pages, capacity, &map)) != TQ_OK) return st;
  if (use_tensor_cores(x_dtype, batch, heads, tokens))
    return tq_launch_quantize_tc(false, x, x_dtype, batch, heads, tokens, stride_b, stride_h,
                                 stride_t, pos, count, cache.idx, nullptr, cache.xnorm, nullptr,
                                 capacity, map, vc, reinterpret_cast<cudaStream_t>(stream));
  QuantArgs a{};
  a.x = x; a.dtype = x_dtype; a.batch = batch; a.heads = heads; a.tokens = tokens;
  a.sb = stride_b; a.sh = stride_h; a.st = stride_t; a.pos = pos; a.count = count;
  a.idx = cache.idx; a.sgn = nullptr; a.xnorm = cache.xnorm; a.rnorm = nullptr;
  a.capacity = capacity; a.map = map; a.rowcap = tq_row_slots(map, capacity);
  a.piT = vc->d_piT; a.mT = nullptr; a.lv = tq_make_levels(vc);
  a.ibits = vc->ibits; a.nibbles = vc->ibits == 4;
  return launch<false>(a, reinterpret_cast<cudaStream_t>(stream));
}

// The FFMA tile quantiser with one CTA per tile of 64 vectors, for inputs where few vectors are
// written (count[b] = 0 for most rows): empty tiles cost a CTA start and no more.
tq_status tq_launch_quantize_tiles(const tq_codec* c, bool prod, const void* x, tq_dtype dt,
                                   int batch, int heads, int tokens, long long sb, long long sh,
                                   long long st, const int* pos, const int* count, uint8_t* idx,
                                   uint8_t* sgn, float* xnorm, float* rnorm, int capacity,
                                   cudaStream_t stream) {
  QuantArgs a{};
  a.x = x; a.dtype = dt; a.batch = batch; a.heads = heads; a.tokens = tokens;
  a.sb = sb; a.sh = sh; a.st = st; a.pos = pos; a.count = count;
  a.idx = idx; a.sgn = sgn; a.xnorm = xnorm; a.rnorm = rnorm;
  a.capacity = capacity; a.map = tq_rowmap{nullptr, 0, 0, 0}; a.rowcap = capacity;
  a.piT = c->d_piT; a.mT = prod ? c->d_mT : nullptr;
  a.lv = tq_make_levels(c); a.ibits = c->ibits; a.nibbles = !prod && c->ibits == 4;
  a.sparse = 1;
  const long long total = (long long)batch * heads * tokens;
  if (total == 0) return TQ_OK;
  const long long ntiles = (total + kTile - 1) / kTile;
  if (ntiles > (1LL << 30)) return TQ_ERR_INVALID_ARG;
  const size_t smem = (size_t)(prod ? 2 : 1) * TQ_D * TQ_D * sizeof(float) +
                      (size_t)kTile * kXStride * sizeof(float);
  auto kern = prod ? quantize_kernel<true> : quantize_kernel<false>;
  static bool configured[2][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return TQ_ERR_CUDA;
  if (!configured[prod][dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return TQ_ERR_CUDA;
    configured[prod][dev] = true;
  }
  kern<<<(unsigned)ntiles, kThreads, smem, stream>>>(a);
  return tq_cuda_status(cudaGetLastError());
}

tq_status tq_launch_append_kv(const tq::AppendKV& a, int batch, cudaStream_t stream) {
  const long long units = (long long)batch * a.Hkv;
  if (units <= 0) return TQ_OK;
  if (units > INT_MAX) return TQ_ERR_INVALID_ARG;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<long long>(units, tq_num_sms()));
  cfg.blockDim = dim3(tq::kAppendThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, append_kv_kernel, a, (int)units) != cudaSuccess)
    return TQ_ERR_CUDA;
  return tq_cuda_status(cudaGetLastError());
}

extern "C" tq_status tq_device_status(uint32_t* flags) {
  if (!flags) return TQ_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return TQ_ERR_CUDA;
  const unsigned int a = tq_take_flags_quantize(), b = tq_take_flags_attention();
  const unsigned int d = tq_take_flags_quantize_tc(), e = tq_take_flags_decode_tc();
  const unsigned int f = tq_take_flags_decode_asym(), g = tq_take_flags_store();
  if (a == ~0u || b == ~0u || d == ~0u || e == ~0u || f == ~0u || g == ~0u) return TQ_ERR_CUDA;
  *flags = a | b | d | e | f | g;
  if (*flags & TQ_FLAG_TIMEOUT) return TQ_ERR_TIMEOUT;
  return *flags ? TQ_ERR_DEVICE_STATUS : TQ_OK;
}
