// Asymmetric split decode: keys kept in FP16, values MSE-coded, plus an FP16 tail of recent
// tokens in the same softmax (the MLX-port article, "对称 vs 非对称": K = FP16 / V = turbo for
// dense models; its quick start's min_compress_tokens tail).
//
// One CTA per (batch, KV head, split); splits past the compressed part cover the FP16 tail.
// A producer warp streams 128-token tiles into a 4-stage ring: the FP16 key rows by TMA tensor
// copies (two boxes of 64 columns per tile, 128-byte swizzle: 16-byte chunk c of row t at
// chunk c ^ (t & 7) of its 128-byte row, so that ldmatrix reads 8 rows without bank
// conflicts), the value codes and norms by bulk copies.  Eight softmax warps in two groups of four take alternate tiles; a warp scores its 32
// tokens with mma.sync m16n8k16 against the query held as an fp16 pair (value and rounding
// residue, per-head power-of-two scale), then runs the online softmax and the value products
// shared with the packed-key kernel.  Tail tiles take FP16 values through ldmatrix.trans.
// Each CTA writes one (m, l, acc) record per head in the layout of the CUDA-core path, whose
// merge kernel combines them (rotating back the compressed part only).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <string.h>

#include "decode_args.h"
#include "tc_ptx.h"
#include "tile_mma.h"

TQ_DEFINE_FLAGS(tq_take_flags_decode_asym)

namespace {
using namespace tq;

constexpr int kTile = 128;                    // tokens per tile and ring stage
constexpr int kStages = 4;
constexpr int kSWarps = 8;                    // softmax warps: two groups of four
constexpr int kThreads = (kSWarps + 1) * 32;  // + producer warp
constexpr int kRec = TQ_REC;
constexpr int kAccPitch = 140;
constexpr int kBarS = 1;

__host__ __device__ constexpr int accidx(int col, int j) { return col * kAccPitch + j + (j >> 4); }

__device__ __forceinline__ float load_elem_any(const void* base, int dtype, long long i) {
  if (dtype == TQ_F32) return static_cast<const float*>(base)[i];
  const uint16_t u = static_cast<const uint16_t*>(base)[i];
  if (dtype == TQ_BF16) return __uint_as_float((uint32_t)u << 16);
  return __half2float(__ushort_as_half(u));
}

// shared memory: the ring (per stage: swizzled key rows, value codes, value norms), then the
// 4-bit pair table
template <int VB>
struct AL {
  static constexpr int krows = 0;                      // two 64-column halves of 128 × 128 B
  static constexpr int vcodes = kTile * 256;
  static constexpr int vcode_bytes = VB == 4 ? kTile * 64 : VB * kTile * 16;
  static constexpr int vxn = vcodes + 8192;                              // room for 4-bit codes
  static constexpr int stage = vxn + 1024;             // a multiple of 1024 (swizzle atoms)
  static constexpr int ring = kStages * stage;
  static constexpr int lut = ring;
  static constexpr int lut_bytes = VB == 4 ? 256 * 32 * 4 : 0;
  static constexpr int total = lut + lut_bytes + 1024;  // + alignment of the base to 1024
  static_assert(stage % 1024 == 0, "stage alignment");
  // after the main loop the ring holds the softmax warps' accumulators and statistics
  static constexpr int comb_stats = kSWarps * 8 * kAccPitch * 4;
  static_assert(vcode_bytes <= 8192, "value codes");
  static_assert(comb_stats + (kSWarps * 4 + 3) * 8 * 4 <= ring, "combine scratch");
};

// TMA tensor copy of the box at (column x, row y) into shared memory, completing on `bar`
__device__ __forceinline__ void tma_rows(uint32_t dst, const CUtensorMap* map, int x, int y,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(s32(bar))
      : "memory");
}
// byte offset of 16-byte chunk `ch` (0..15) of row `t` in a tile of two swizzled 64-column
// halves (128 rows × 128 B each)
__device__ __forceinline__ uint32_t swz(int t, int ch) {
  return (uint32_t)(ch >> 3) * 16384u + (uint32_t)t * 128u + ((uint32_t)((ch & 7) ^ (t & 7)) << 4);
}

template <int VB, bool HILO>
__global__ void __launch_bounds__(kThreads, 1) decode_asym_tc_kernel(const __grid_constant__ tq_asym_launch a) {
  using L = AL<VB>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (s32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t lut_bar;
  __shared__ __align__(16) uint2 qb[8][2][32];   // query B fragments: [16-dim block][hi, lo][lane]
  __shared__ float s_qmax[8];

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long bh = (long long)b * a.Hkv + kvh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool tail = split >= a.nsplit_main;
  const int cap = tail ? a.tail_cap : a.cap;
  int len = tail ? a.tail_lens[b] : a.seq_lens[b];
  if (len > cap) {
    if (tid == 0 && (split == 0 || split == a.nsplit_main) && kvh == 0)
      atomicOr(&g_tq_flags, TQ_FLAG_LEN_OVERFLOW);
    len = cap;
  }
  const int span = tail ? a.tail_split : a.split_len;
  const int t_begin = (tail ? split - a.nsplit_main : split) * span;
  const int t_end = min(t_begin + span, len);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;
  // the tail's values are FP16 rows: a tile takes two stages (keys, values)
  const int depth = tail ? kStages / 2 : kStages;
  const CUtensorMap* kmap = tail ? &a.ktmap : &a.kmap;

  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full_bar[st], 1);
      mbar_init(&empty_bar[st], kSWarps / 2);
    }
    mbar_init(&lut_bar, 1);
    mbar_init_fence();
  }
  __syncthreads();

  // ============================================================ producer warp
  if (warp == kSWarps) {
    if (!tail && VB == 4 && ntiles > 0 && lane == 0) {
      mbar_expect_tx(&lut_bar, L::lut_bytes);
      bulk_g2s(smem + L::lut, a.lut, L::lut_bytes, &lut_bar);
    }
    int i = 0;
    for (; i < ntiles; ++i) {
      const int slot = i % depth;
      if (i >= depth && !mbar_wait(&empty_bar[slot], ((i / depth) - 1) & 1)) {
        if (lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
        break;
      }
      const int t0 = t_begin + i * kTile;
      unsigned char* kst = smem + (tail ? 2 * slot : slot) * L::stage;
      if (lane == 0) {
        // key rows (and the tail's value rows) by TMA; rows past the tensor read as zeros
        const int y = (int)(bh * cap + t0);
        unsigned bytes = 2u * 16384u;
        if (tail) {
          bytes += 2u * 16384u;
        } else {
          const int n = min(kTile, a.cap - t0);   // a multiple of 64 (the capacity is)
          bytes += (unsigned)n * ((VB == 4 ? 64 : VB * 16) + 4);
        }
        mbar_expect_tx(&full_bar[slot], bytes);
        tma_rows(s32(kst + L::krows), kmap, 0, y, &full_bar[slot]);
        tma_rows(s32(kst + L::krows + 16384), kmap, 64, y, &full_bar[slot]);
        if (tail) {
          tma_rows(s32(kst + L::stage), &a.vtmap, 0, y, &full_bar[slot]);
          tma_rows(s32(kst + L::stage + 16384), &a.vtmap, 64, y, &full_bar[slot]);
        } else {
          const int n = min(kTile, a.cap - t0);
          if (VB == 4) {
            bulk_g2s(kst + L::vcodes, a.vidx + (bh * a.cap + t0) * 64, n * 64, &full_bar[slot]);
          } else {
            for (int p = 0; p < VB; ++p)
              bulk_g2s(kst + L::vcodes + p * kTile * 16, a.vidx + ((bh * VB + p) * a.cap + t0) * 16,
                       n * 16, &full_bar[slot]);
          }
          bulk_g2s(kst + L::vxn, a.vxn + bh * a.cap + t0, n * 4, &full_bar[slot]);
        }
      }
      __syncwarp();
    }
    // every copy issued lands before the CTA may finish
    for (int k = i - depth > 0 ? i - depth : 0; k < i; ++k)
      mbar_wait(&full_bar[k % depth], (k / depth) & 1);
    if (!tail && VB == 4 && ntiles > 0) mbar_wait(&lut_bar, 0);
    return;
  }

  // ============================================================ softmax warps
  const int q = warp & 3, grp = warp >> 2;
  const int g = lane >> 2, c = lane & 3;
  // query B fragments: column n is head n (G > 4) or head n / 2 (G ≤ 4), scaled by a power of
  // two per head so that its largest |value| lies in [2^14, 2^15); hi + lo carry ~22 bits
  if (warp < a.G) {
    float mx = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const long long e = ((long long)b * a.Hq + kvh * a.G + warp) * TQ_D + lane + 32 * k;
      mx = fmaxf(mx, fabsf(load_elem_any(a.q, a.q_dtype, e)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_qmax[warp] = mx;
  }
  named_sync(kBarS, kSWarps * 32);
  auto qscale = [&](int head) {
    const float mx = s_qmax[head];
    if (!(mx > 0.f) || !isfinite(mx)) return 1.f;
    int e;
    frexpf(mx, &e);                   // mx = f·2^e, f in [0.5, 1)
    return ldexpf(1.f, 15 - e);
  };
  {
    const int kk = tid >> 5, ln = lane;   // 256 threads: (16-dim block, lane)
    const int gg = ln >> 2, cc = ln & 3;
    const int head = HILO ? gg >> 1 : gg;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (head < a.G) {
      const float sg = qscale(head);
      const long long e0 = ((long long)b * a.Hq + kvh * a.G + head) * TQ_D + 16 * kk;
      const int ks[4] = {2 * cc, 2 * cc + 1, 2 * cc + 8, 2 * cc + 9};
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] = sg * load_elem_any(a.q, a.q_dtype, e0 + ks[u]);
    }
    float hi[4], lo[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      hi[u] = __half2float(__float2half_rn(x[u]));
      lo[u] = x[u] - hi[u];
    }
    qb[kk][0][ln] = make_uint2(pack_half2(hi[0], hi[1]), pack_half2(hi[2], hi[3]));
    qb[kk][1][ln] = make_uint2(pack_half2(lo[0], lo[1]), pack_half2(lo[2], lo[3]));
  }
  // per-column logit scale: softmax scale · log2(e) / the column's query scale
  float cs[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int col = 2 * c + h, head = HILO ? col >> 1 : col;
    cs[h] = head < a.G ? a.scale_log2 / qscale(head) : 0.f;
  }
  named_sync(kBarS, kSWarps * 32);
  bool okp = tail || VB != 4 || ntiles == 0 || mbar_wait(&lut_bar, 0);
  if (!okp && lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);

  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f}, lw_run[2] = {0.f, 0.f};
  const uint32_t* lut_lane = reinterpret_cast<const uint32_t*>(smem + L::lut) + lane;

  for (int i = grp; i < ntiles && okp; i += 2) {
    const int slot = i % depth;
    const bool okw = mbar_wait(&full_bar[slot], (i / depth) & 1);
    if (!__all_sync(0xffffffffu, okw)) {   // ldmatrix and mma.sync below are warp-collective
      if (lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
      break;
    }
    const unsigned char* kst = smem + (tail ? 2 * slot : slot) * L::stage;
    const uint32_t kbase = s32(kst + L::krows);
    const int t_tile = t_begin + i * kTile;
    // ---- scores: D[token][column] = Σ_k K[token][k]·Q[column][k], query as hi + lo
    float d[2][4];
#pragma unroll
    for (int T = 0; T < 2; ++T) {
      d[T][0] = d[T][1] = d[T][2] = d[T][3] = 0.f;
      const int mi = lane >> 3, r = lane & 7;
      const int tok = 32 * q + 16 * T + r + 8 * (mi & 1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + swz(tok, 2 * kk + (mi >> 1)), a0, a1, a2, a3);
        const uint2 bh_ = qb[kk][0][lane], bl_ = qb[kk][1][lane];
        mma16816(d[T], a0, a1, a2, a3, bh_.x, bh_.y);
        mma16816(d[T], a0, a1, a2, a3, bl_.x, bl_.y);
      }
    }
    float lg[2][2][2];
    bool okt[2][2];
#pragma unroll
    for (int T = 0; T < 2; ++T)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        okt[T][k] = t_tile + 32 * q + 16 * T + g + 8 * k < t_end;
#pragma unroll
        for (int h = 0; h < 2; ++h) lg[T][k][h] = okt[T][k] ? d[T][2 * k + h] * cs[h] : -INFINITY;
      }
    if (!tail) {
      const float* vxn = reinterpret_cast<const float*>(kst + L::vxn) + 32 * q;
      softmax_values_step<VB, HILO>(lg, okt, vxn, kst + L::vcodes + 32 * q * (VB == 4 ? 64 : 16),
                                    kTile * 16, lut_lane, a.vd.coef, acc, m_run, l_run, lw_run,
                                    lane);
    } else {
      // FP16 values: A = Vᵀ fragments (coordinates × tokens) by ldmatrix.trans of the rows
      float w[2][2][2];
      online_softmax<HILO ? 1 : 2>(lg, okt, nullptr, acc, m_run, l_run, lw_run, w, lane);
      const uint32_t vbase = s32(kst + L::stage);
#pragma unroll
      for (int T = 0; T < 2; ++T) {
        uint32_t bw0, bw1;
        weight_fragments<HILO>(w, T, bw0, bw1);
        const int mi = lane >> 3, r = lane & 7;
        const int tok = 32 * q + 16 * T + r + 8 * (mi >> 1);
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(vbase + swz(tok, 2 * k8 + (mi & 1)), a0, a1, a2, a3);
          mma16816(acc[k8], a0, a1, a2, a3, bw0, bw1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);
  }

  // ============================================================ combine the softmax warps
  mirror_stats<HILO ? 1 : 2>(m_run, l_run, lw_run);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], o);
      lw_run[h] += __shfl_xor_sync(0xffffffffu, lw_run[h], o);
    }
  }
  named_sync(kBarS, kSWarps * 32);   // every softmax warp is done with the ring: reuse it
  float* cacc = reinterpret_cast<float*>(smem);                   // [warp][col][140]
  float* cstat = reinterpret_cast<float*>(smem + L::comb_stats);  // [warp][3][8]
  float* fac = cstat + kSWarps * 3 * 8;                           // [warp][8]
  float* cML = fac + kSWarps * 8;                                 // M, L, LW [3][8]
#pragma unroll
  for (int k8 = 0; k8 < 8; ++k8) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int hi_row = k >> 1;                    // 0: row g, 1: row g + 8
      const int col = 2 * c + (k & 1);
      int coord;
      float v = acc[k8][k];
      if (tail) {
        coord = 16 * k8 + g + 8 * hi_row;
      } else if (VB == 4) {
        coord = 16 * g + 2 * k8 + hi_row;
        v *= a.vc_unscale;
      } else {
        const int e = 2 * k8 + hi_row;
        coord = 16 * g + pair_lo(e);
        v *= exp2f((float)-pos_exp(pair_pos(e)));
      }
      cacc[accidx(warp * 8 + col, coord)] = v;
    }
  }
  if (g == 0) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int col = 2 * c + k;
      cstat[(warp * 3 + 0) * 8 + col] = m_run[k];
      cstat[(warp * 3 + 1) * 8 + col] = l_run[k];
      cstat[(warp * 3 + 2) * 8 + col] = lw_run[k];
    }
  }
  named_sync(kBarS, kSWarps * 32);
  if (tid < 8) {
    const int col = tid;
    float M = -INFINITY;
    for (int wp = 0; wp < kSWarps; ++wp) M = fmaxf(M, cstat[(wp * 3) * 8 + col]);
    float Lsum = 0.f, lw = 0.f;
    for (int wp = 0; wp < kSWarps; ++wp) {
      const float mw_ = cstat[(wp * 3) * 8 + col];
      const float f = (M == -INFINITY || mw_ == -INFINITY) ? 0.f : exp2f(mw_ - M);
      fac[wp * 8 + col] = f;
      Lsum += f * cstat[(wp * 3 + 1) * 8 + col];
      lw += f * cstat[(wp * 3 + 2) * 8 + col];
    }
    cML[col] = M;
    cML[8 + col] = Lsum;
    cML[16 + col] = lw;
  }
  named_sync(kBarS, kSWarps * 32);
  // the record: m in natural-log units (the merge kernel's), l, acc (rotated domain for codes)
  float* rec = a.part + ((bh * a.nsplit + split) * a.G) * kRec;
  for (int it = tid; it < a.G * TQ_D; it += kSWarps * 32) {
    const int head = it >> 7, j = it & 127;
    const int col = HILO ? 2 * head : head;
    float acc_j = 0.f;
#pragma unroll
    for (int wp = 0; wp < kSWarps; ++wp) {
      float av = cacc[accidx(wp * 8 + col, j)];
      if (HILO) av += cacc[accidx(wp * 8 + col + 1, j)];
      acc_j = fmaf(fac[wp * 8 + col], av, acc_j);
    }
    if (!tail && VB != 4) acc_j -= a.vd.cst * cML[16 + col];
    rec[head * kRec + 2 + j] = acc_j;
    if (j == 0) {
      rec[head * kRec] = cML[col] * 0.6931471805599453f;
      rec[head * kRec + 1] = cML[8 + col];
    }
  }
}

template <int VB, bool HILO>
tq_status launch_one(const tq_asym_launch& a, cudaStream_t stream) {
  constexpr int smem = AL<VB>::total;
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return TQ_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(decode_asym_tc_kernel<VB, HILO>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    configured[dev] = true;
  }
  decode_asym_tc_kernel<VB, HILO><<<dim3(a.nsplit, a.Hkv, a.B), kThreads, smem, stream>>>(a);
  return tq_cuda_status(cudaGetLastError());
}

template <int VB>
tq_status launch_v(const tq_asym_launch& a, cudaStream_t stream) {
  return a.G <= 4 ? launch_one<VB, true>(a, stream) : launch_one<VB, false>(a, stream);
}

}  // namespace

tq_status tq_asym_encode_rows(CUtensorMap* map, const void* base, long long rows) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);
  static Encode encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return TQ_ERR_CUDA;
    encode = reinterpret_cast<Encode>(fn);
  }
  if (rows <= 0 || !base) {   // unused (no tail): never read by the kernel
    memset(map, 0, sizeof(*map));
    return TQ_OK;
  }
  const cuuint64_t dims[2] = {(cuuint64_t)TQ_D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)TQ_D * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kTile};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TQ_OK : TQ_ERR_CUDA;
}

bool tq_asym_tc_supported(int vbits, int G, int split_len, int tail_split) {
  return vbits >= 1 && vbits <= 4 && G >= 1 && G <= 8 && split_len % kTile == 0 &&
         tail_split % kTile == 0;
}

tq_status tq_launch_decode_asym_tc(const tq_asym_launch& a, cudaStream_t stream) {
  if (!tq_asym_tc_supported(a.vbits, a.G, a.split_len, a.tail_split)) return TQ_ERR_UNSUPPORTED;
  switch (a.vbits) {
    case 1: return launch_v<1>(a, stream);
    case 2: return launch_v<2>(a, stream);
    case 3: return launch_v<3>(a, stream);
    case 4: return launch_v<4>(a, stream);
  }
  return TQ_ERR_UNSUPPORTED;
}
