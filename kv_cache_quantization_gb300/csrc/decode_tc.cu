// Split-context decode attention on packed codes, key scores on the fifth-generation tensor
// cores (tcgen05, kind::f8f6f4, operands and accumulators in TMEM).
//
// The estimator of the QJL deep-dive (§五, §六) for key t and query head h is
//   s = ‖x_t‖·⟨Π q_h, c[idx_t]⟩ + ‖r_t‖·√(π/2)/d·⟨S q_h, 2·sign_t − 1⟩,
// and the value side accumulates Σ_t p_t·‖v_t‖·c_v[idx_t] in the rotated domain, rotated
// back once per head at the end (out = Πᵀ·acc / L).
//
// Key scores.  The Lloyd-Max levels are expanded into odd Walsh monomials, so a key index
// becomes NKV "virtual" 0/1 bit planes (XORs of its index bits); with the sign plane that
// is NP planes, and each score is a sum over planes of ⟨0/1 bits, query vector⟩.  For a tile
// of 128 tokens (one token per TMEM lane) the expander warps turn every plane into an e4m3
// A operand in TMEM: a byte is 0x40 (= 2.0) where the bit is set, else 0, produced four
// coordinates at a time by one shift and one AND.  The query operand B (shared memory)
// carries each query value as four e4m3 "pieces" at their true scale (x ≈ p0 + p1 + p2 + p3,
// about 15 significant bits), one B row per (piece, column), so D column (piece, column)
// sums to the exact fp32 contraction of that piece and the softmax warps add the four.
// Each plane is a 128 × 32 × 128 product: 4 MMAs of K = 32, issued by one thread per plane.
//
// Softmax and values.  Two groups of four softmax warps take alternate tiles.  A warp reads
// its 32 tokens' accumulators with the 16x256b TMEM load (register layout of the mma.sync
// accumulator fragment), keeps an online softmax per column and accumulates values with
// mma.sync m16n8k16 (4-bit codes through a pair table of fp16 levels, 1–3-bit codes as planes).
//
// Data path.  A producer warp streams 128-token stages of packed K/V through an 8-deep
// shared-memory ring with bulk copies (TMA engine).  The query operand of each (batch, KV
// head) is built by a small kernel that runs as this kernel's programmatic-launch primary:
// the split CTAs start streaming the cache at once and wait for that kernel only before
// their first MMA.  Each CTA writes one (m, l, acc) record per head; the last CTA of a
// (batch, KV head) to finish (a ticket counter in the workspace) merges the records with
// log-sum-exp weights and rotates the result back.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "decode_mma.h"
#include "tc_ptx.h"

TQ_DEFINE_FLAGS(tq_take_flags_decode_tc)

namespace {
using namespace tq;

constexpr int kTile = 128;                    // tokens per tile = TMEM lanes
constexpr int kStageTok = 256;                // tokens per ring stage (two tiles)
constexpr int kStages = 4;
constexpr int kEWarps = 4;                    // expand planes into TMEM
constexpr int kSWarps = 8;                    // softmax + values (two groups of four)
constexpr int kIWarps = 3;                    // issue MMAs (one thread each)
constexpr int kCompute = (kEWarps + kSWarps + kIWarps) * 32;
constexpr int kThreads = kCompute + 32;       // + producer warp
constexpr int kPieces = 4;                    // e4m3 pieces per query value
constexpr int kN = kPieces * 8;               // MMA N: 4 pieces × 8 columns
constexpr int kBImg = kN * 128;               // one plane's query operand (4 KB of e4m3)
constexpr int kBSbo = 8 * 128;                // 8-row groups of the operand image
constexpr int kCstBytes = 8 * 4 * 4;          // 8 columns × {A, Cm, B, Cq}
constexpr int kRec = TQ_REC;
constexpr int kMaxSplits = 256;
constexpr int kAccPitch = 140;
constexpr int kPrepThreads = 256;
// named barriers
constexpr int kBarS = 2, kBarAll = 3;

__host__ __device__ constexpr int accidx(int col, int j) { return col * kAccPitch + j + (j >> 4); }

// Virtual planes of a KB-bit index: the odd subsets of its bit positions, as bit masks.
__host__ __device__ constexpr int num_vplanes(int kb) { return kb == 1 ? 1 : kb == 2 ? 2 : 4; }
__host__ __device__ constexpr int vplane_mask(int kb, int v) {
  return kb == 1 ? 1 : kb == 2 ? (v == 0 ? 1 : 2) : (v == 0 ? 1 : v == 1 ? 2 : v == 2 ? 4 : 7);
}
template <int KB>
__device__ __forceinline__ uint32_t vplane_word(const uint32_t* w, int v) {
  const int m = vplane_mask(KB, v);
  uint32_t x = 0;
#pragma unroll
  for (int i = 0; i < KB; ++i)
    if (m & (1 << i)) x ^= w[i];
  return x;
}
// Bytes of the operand images per (batch, KV head): NP planes + score constants.
__host__ __device__ constexpr int frag_block(int np) { return np * kBImg + kCstBytes; }
constexpr int kMaxFragBlock = frag_block(5);

// Operand K position k of plane word i (coordinates 32i..32i+31): column c = k / 4 =
// 8i + r holds coordinates 32i + 8b + r in its bytes b = 0..3.
__host__ __device__ constexpr int coord_of_k(int k) {
  return 32 * (k >> 5) + 8 * (k & 3) + ((k >> 2) & 7);
}
// canonical K-major offset of byte (row n < 32, k < 128) in one plane's e4m3 operand
__host__ __device__ constexpr int bimg_off(int n, int k) {
  return (n >> 3) * kBSbo + (k >> 4) * 128 + (n & 7) * 16 + (k & 15);
}

// ---------------------------------------------------------------- bit-pair expansion (values)
// 1–3-bit value planes in the PV product: pair e of a word holds bit lo(e) in its low fp16
// half and bit lo(e)+16 in its high half, as 0 or 2^exp(e) (see pair_at).
__host__ __device__ constexpr int pair_lo(int e) {
  return e < 5 ? 10 + e : e < 10 ? e : e < 15 ? e - 10 : 15;
}
__host__ __device__ constexpr int pair_pos(int e) { return e < 15 ? 10 + e % 5 : 14; }
__host__ __device__ constexpr int pos_exp(int pos) {
  return pos == 10 ? -14 : pos == 11 ? -13 : pos == 12 ? -11 : pos == 13 ? -7 : 1;
}
struct Shifted {
  uint32_t w, w5, w10, w1;
};
__device__ __forceinline__ Shifted shifted(uint32_t w) { return Shifted{w, w << 5, w << 10, w >> 1}; }
__device__ __forceinline__ uint32_t pair_at(const Shifted& x, int e) {
  const int pos = pair_pos(e);
  const uint32_t mask = (1u << pos) | (1u << (pos + 16));
  return (e < 5 ? x.w : e < 10 ? x.w5 : e < 15 ? x.w10 : x.w1) & mask;
}

// ---------------------------------------------------------------- warp-level matrix ops
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// D (TMEM) (+)= A (TMEM, e4m3) · Bᵀ (shared, e4m3), fp32 accumulation
__device__ __forceinline__ void mma_f8(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc));
}
// 16 TMEM lanes × 32 columns in the accumulator-fragment layout (repetition k = columns
// 8k..8k+7 in registers 4k..4k+3: (row g, cols 2c, 2c+1), (row g+8, same columns))
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ float e4m3_value(__nv_fp8_storage_t x) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(x, __NV_E4M3)));
}

// ---------------------------------------------------------------- query operand kernel
// Grid (4 slices, KV heads, batch).  The CTA for slice s computes (Π q_h)_j and (S q_h)_j
// for the group's heads h and coordinates j = 32s..32s+31 (plane word s), and writes the
// operand bytes of K positions 32s..32s+31 of every plane: row (piece p, column n) holds
// piece p of 0.5·coef_v·(Π q)_j/‖q‖·s_idx (index plane v) or 0.5·2·(S q)_j/(‖q‖·smax)·s_sgn
// (sign plane), column n = head n (G > 4) or head n/2 (G ≤ 4).  ‖q‖ and the column sums
// (Πᵀ1)·q, (Sᵀ1)·q come straight from q, so no slice needs another slice's results.
template <int KB, bool HILO>
__global__ void __launch_bounds__(kPrepThreads) query_prep_tc_kernel(const tq_mma_launch a) {
  constexpr int NKV = num_vplanes(KB);
  constexpr int NP = NKV + 1;
  __shared__ float qf[8][TQ_D];
  __shared__ float part[2][4][8][32];     // [Π|S][k quarter][head][j in slice]
  __shared__ float qs[2][8][32];
  __shared__ float s_nq[8], s_uq[8], s_wq[8];
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long bh = (long long)b * a.Hkv + kvh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the decode grid may start now; it waits for this grid before its first MMA
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = tid; i < 8 * TQ_D; i += kPrepThreads) {
    const int h = i >> 7, j = i & 127;
    float v = 0.f;
    if (h < a.G) {
      const long long e = ((long long)b * a.Hq + kvh * a.G + h) * TQ_D + j;
      if (a.q_dtype == TQ_F32) v = static_cast<const float*>(a.q)[e];
      else if (a.q_dtype == TQ_BF16)
        v = __uint_as_float((uint32_t)static_cast<const uint16_t*>(a.q)[e] << 16);
      else v = __half2float(__ushort_as_half(static_cast<const uint16_t*>(a.q)[e]));
    }
    qf[h][j] = v;
  }
  // thread (which, k quarter, j): 32 coalesced loads of Πᵀ or Sᵀ, issued together
  const int which = tid >> 7, kq = (tid >> 5) & 3, jl = lane;
  const float* T = which ? a.sT : a.piT;
  float t[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) t[k] = __ldg(&T[(32 * kq + k) * TQ_D + 32 * s + jl]);
  __syncthreads();
  if (warp < a.G) {
    // ‖q‖, (Πᵀ1)·q and (Sᵀ1)·q of head `warp`
    float n2 = 0.f, uq = 0.f, wq = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = lane + 32 * k;
      const float x = qf[warp][j];
      n2 = fmaf(x, x, n2);
      uq = fmaf(__ldg(&a.u[j]), x, uq);
      wq = fmaf(__ldg(&a.w[j]), x, wq);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n2 += __shfl_xor_sync(0xffffffffu, n2, o);
      uq += __shfl_xor_sync(0xffffffffu, uq, o);
      wq += __shfl_xor_sync(0xffffffffu, wq, o);
    }
    if (lane == 0) {
      s_nq[warp] = sqrtf(n2);
      s_uq[warp] = uq;
      s_wq[warp] = wq;
    }
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    float acc = 0.f;
    if (h < a.G) {
#pragma unroll
      for (int k = 0; k < 32; ++k) acc = fmaf(t[k], qf[h][32 * kq + k], acc);
    }
    part[which][kq][h][jl] = acc;
  }
  __syncthreads();
  for (int i = tid; i < 2 * 8 * 32; i += kPrepThreads) {
    const int wh = i >> 8, h = (i >> 5) & 7, j = i & 31;
    qs[wh][h][j] = (part[wh][0][h][j] + part[wh][1][h][j]) + (part[wh][2][h][j] + part[wh][3][h][j]);
  }
  __syncthreads();
  unsigned char* out = static_cast<unsigned char*>(a.qfrag) + bh * (long long)frag_block(NP);
  // item (plane v, column n, K position k within the slice): four piece bytes
  for (int i = tid; i < NP * 8 * 32; i += kPrepThreads) {
    const int v = i >> 8, n = (i >> 5) & 7, kl = i & 31;
    const int k = 32 * s + kl;
    const int jl2 = coord_of_k(k) - 32 * s;
    const int head = HILO ? n >> 1 : n;
    float x = 0.f;
    if (head < a.G && s_nq[head] > 0.f) {
      const float nq = s_nq[head];
      x = v < NKV ? 0.5f * a.kd.coef[v] * qs[0][head][jl2] / nq * a.s_idx
                  : qs[1][head][jl2] / (nq * a.smax) * a.s_sgn;
    }
#pragma unroll
    for (int p = 0; p < kPieces; ++p) {
      const __nv_fp8_storage_t y = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
      x -= e4m3_value(y);
      out[v * kBImg + bimg_off(p * 8 + n, k)] = y;
    }
  }
  if (s == 0 && tid < 8) {
    // score constants of column n: A, Cm, B, Cq (see the softmax warps)
    const int n = tid, head = HILO ? n >> 1 : n;
    float* cst = reinterpret_cast<float*>(out + NP * kBImg);
    const float nq = head < a.G ? s_nq[head] : 0.f;
    const bool ok = nq > 0.f;
    cst[n * 4 + 0] = nq * a.scale_log2 / a.s_idx;
    cst[n * 4 + 1] = ok ? a.s_idx * a.kd.cst * s_uq[head] / nq : 0.f;
    cst[n * 4 + 2] = nq * a.smax * a.scale_log2 * (1.2533141373155003f / TQ_D) / a.s_sgn;
    cst[n * 4 + 3] = ok ? a.s_sgn * s_wq[head] / (nq * a.smax) : 0.f;
  }
}

// ---------------------------------------------------------------- shared memory and TMEM
template <int KB, int VB>
struct TL {
  static constexpr int NP = num_vplanes(KB) + 1;             // planes incl. the sign plane
  // one ring stage (256 tokens)
  static constexpr int kplanes = 0;
  static constexpr int ksgn = kplanes + KB * kStageTok * 16;
  static constexpr int kxn = ksgn + kStageTok * 16;
  static constexpr int krn = kxn + kStageTok * 4;
  static constexpr int vcodes = krn + kStageTok * 4;
  static constexpr int vcode_bytes = VB == 4 ? kStageTok * 64 : VB * kStageTok * 16;
  static constexpr int vxn = vcodes + vcode_bytes;
  static constexpr int stage = vxn + kStageTok * 4;
  static constexpr int ring = kStages * stage;
  static constexpr int lut = ring;                           // VB == 4: 256 keys × 32 copies
  static constexpr int lut_bytes = VB == 4 ? 256 * 32 * 4 : 0;
  static constexpr int frag = lut + lut_bytes;               // operand images + constants
  static constexpr int used = frag + frag_block(NP);
  // the last-CTA merge stages Π (64 KB) and the split records in shared memory, with its
  // accumulators and weights (12 KB) at the end; make room for 36 split records of 8 heads
  static constexpr int merge_min = 65536 + 36 * 8 * kRec * 4 + 12288;
  static constexpr int total = used > merge_min ? used : merge_min;
  static constexpr int mrg_acc = total - 12288;              // float [8][128]
  static constexpr int mrg_w = mrg_acc + 4096;               // float [8][kMaxSplits]
  // after the main loop the ring is reused: softmax-warp accumulators and statistics
  static constexpr int comb_acc = 0;
  static constexpr int comb_stats = kSWarps * 8 * kAccPitch * 4;
  static_assert(comb_stats + (kSWarps * 4 + 3) * 8 * 4 <= ring, "combine scratch");
  // TMEM: A (one tile: NP planes × 32 columns of e4m3), D (NP planes × 32 columns)
  static constexpr int a_cols = NP * 32;
  static constexpr int d_cols = NP * kN;
  static constexpr int abufs = (2 * a_cols + 2 * d_cols <= 512) ? 2 : 1;
  static constexpr int d_col = abufs * a_cols;
  static_assert(d_col + 2 * d_cols <= 512, "TMEM columns");
};

// ---------------------------------------------------------------- the split kernel
template <int KB, int VB, bool HILO>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const tq_mma_launch a) {
  using L = TL<KB, VB>;
  constexpr int NKV = num_vplanes(KB);
  constexpr int NP = NKV + 1;
  constexpr int NVV = VB == 4 ? 0 : num_vplanes(VB);
  constexpr int NI = NP < kIWarps ? NP : kIWarps;             // active issuer warps
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t mma_done[2];
  __shared__ __align__(8) uint64_t d_free[2];
  __shared__ __align__(8) uint64_t a_full[2];
  __shared__ __align__(8) uint64_t prol_bar;
  __shared__ __align__(8) uint64_t mrg_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_ticket;

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long bh = (long long)b * a.Hkv + kvh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int len = a.seq_lens[b];
  if (len > a.cap) {
    if (tid == 0 && split == 0 && kvh == 0) atomicOr(&g_tq_flags, TQ_FLAG_LEN_OVERFLOW);
    len = a.cap;
  }
  const int t_begin = split * a.split_len;
  const int t_end = min(t_begin + a.split_len, len);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;
  const int nstages = (ntiles + 1) / 2;

  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full_bar[st], 1);
      mbar_init(&empty_bar[st], 2 * (kEWarps + kSWarps / 2));   // two tiles per stage
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&mma_done[i], NI);
      mbar_init(&d_free[i], kSWarps / 2);
      mbar_init(&a_full[i], kEWarps);
    }
    mbar_init(&prol_bar, 1);
    mbar_init(&mrg_bar, 1);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(&s_tmem, 512);
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = s_tmem;

  // ============================================================ producer warp
  if (warp == kEWarps + kSWarps + kIWarps) {
    if (lane == 0) {
      auto issue = [&](int c) {
        const int st = c % kStages;
        const int t0 = t_begin + c * kStageTok;
        const int n = min(kStageTok, a.cap - t0);   // a multiple of 64 (the capacity is)
        unsigned char* base = smem + st * L::stage;
        const unsigned bytes =
            (unsigned)n * (KB * 16 + 16 + 4 + 4 + (VB == 4 ? 64 : VB * 16) + 4);
        mbar_expect_tx(&full_bar[st], bytes);
        for (int p = 0; p < KB; ++p)
          bulk_g2s(base + L::kplanes + p * kStageTok * 16,
                   a.kidx + ((bh * KB + p) * a.cap + t0) * 16, n * 16, &full_bar[st]);
        bulk_g2s(base + L::ksgn, a.ksgn + (bh * a.cap + t0) * 16, n * 16, &full_bar[st]);
        bulk_g2s(base + L::kxn, a.kxn + bh * a.cap + t0, n * 4, &full_bar[st]);
        bulk_g2s(base + L::krn, a.krn + bh * a.cap + t0, n * 4, &full_bar[st]);
        if (VB == 4) {
          bulk_g2s(base + L::vcodes, a.vidx + (bh * a.cap + t0) * 64, n * 64, &full_bar[st]);
        } else {
          for (int p = 0; p < VB; ++p)
            bulk_g2s(base + L::vcodes + p * kStageTok * 16,
                     a.vidx + ((bh * VB + p) * a.cap + t0) * 16, n * 16, &full_bar[st]);
        }
        bulk_g2s(base + L::vxn, a.vxn + bh * a.cap + t0, n * 4, &full_bar[st]);
      };
      int c = 0;
      for (; c < nstages && c < kStages; ++c) issue(c);
      // the operand images are the primary kernel's output
      asm volatile("griddepcontrol.wait;" ::: "memory");
      mbar_expect_tx(&prol_bar, frag_block(NP) + L::lut_bytes);
      bulk_g2s(smem + L::frag, static_cast<const unsigned char*>(a.qfrag) + bh * (long long)frag_block(NP),
               frag_block(NP), &prol_bar);
      if (VB == 4) bulk_g2s(smem + L::lut, a.lut, L::lut_bytes, &prol_bar);
      for (; c < nstages; ++c) {
        const int st = c % kStages;
        if (!mbar_wait(&empty_bar[st], ((c / kStages) - 1) & 1)) {
          atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
          break;
        }
        issue(c);
      }
      // every copy issued lands before the CTA may finish
      for (int k = c - kStages > 0 ? c - kStages : 0; k < c; ++k)
        mbar_wait(&full_bar[k % kStages], (k / kStages) & 1);
      mbar_wait(&prol_bar, 0);
    }
    return;
  }

  if (warp < kEWarps) {
    // ========================================================== expander warps
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    for (int i = 0; i < ntiles; ++i) {
      const int c = i >> 1, h = i & 1;
      const int st = c % kStages;
      const int ab = L::abufs == 2 ? (i & 1) : 0;
      bool okl = mbar_wait(&full_bar[st], (c / kStages) & 1);
      uint32_t pw[KB][4], sw[4];
      {
        const unsigned char* base = smem + st * L::stage;
        const int row = h * kTile + tid;
#pragma unroll
        for (int p = 0; p < KB; ++p) {
          const uint4 u = *reinterpret_cast<const uint4*>(base + L::kplanes + p * kStageTok * 16 + row * 16);
          pw[p][0] = u.x; pw[p][1] = u.y; pw[p][2] = u.z; pw[p][3] = u.w;
        }
        const uint4 u = *reinterpret_cast<const uint4*>(base + L::ksgn + row * 16);
        sw[0] = u.x; sw[1] = u.y; sw[2] = u.z; sw[3] = u.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);
      // the A buffer is free once the MMAs of the tile that used it last have completed
      const int prev = i - L::abufs;
      if (okl && prev >= 0) okl = mbar_wait(&mma_done[prev & 1], (prev >> 1) & 1);
      if (!__all_sync(0xffffffffu, okl)) {   // the TMEM stores below are warp-collective
        if (lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
        break;
      }
      tc_after();
      const uint32_t abase = tmem + lane_base + ab * L::a_cols;
#pragma unroll
      for (int v = 0; v < NP; ++v) {
        uint32_t col[32];
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) {
          uint32_t pv[KB];
#pragma unroll
          for (int p = 0; p < KB; ++p) pv[p] = pw[p][w4];
          const uint32_t x = v < NKV ? vplane_word<KB>(pv, v) : sw[w4];
          // column 8·w4 + r: byte b = bit 8b + r of the word, moved to bit 6 (e4m3 2.0)
#pragma unroll
          for (int r = 0; r < 8; ++r)
            col[8 * w4 + r] = (r < 7 ? x << (6 - r) : x >> 1) & 0x40404040u;
        }
        tmem_st_32x32b_x32(abase + 32 * v, col);
      }
      tmem_wait_st();
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[ab]);
    }
  } else if (warp >= kEWarps + kSWarps) {
    // ========================================================== MMA-issue warps
    // Issuer iw owns planes iw, iw + kIWarps, ...: 4 MMAs of K = 32 per plane and tile,
    // D[i & 1] column block (plane, piece, column).
    const int iw = warp - kEWarps - kSWarps;
    if (lane == 0 && iw < NI && ntiles > 0) {
      const uint32_t idesc = idesc_f16(128, kN);   // e4m3 × e4m3 → f32 has the same fields
      const uint32_t frag_s = s32(smem + L::frag);
      bool ok = mbar_wait(&prol_bar, 0);
      for (int i = 0; i < ntiles && ok; ++i) {
        const int ab = L::abufs == 2 ? (i & 1) : 0;
        const int db = i & 1;
        ok = mbar_wait(&a_full[ab], (i / L::abufs) & 1) &&
             (i < 2 || mbar_wait(&d_free[db], ((i - 2) >> 1) & 1));
        if (!ok) break;
        tc_after();
        for (int v = iw; v < NP; v += kIWarps) {
          const uint32_t d = tmem + L::d_col + db * L::d_cols + v * kN;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t acol = tmem + ab * L::a_cols + 32 * v + 8 * ks;
            const uint64_t bd = smem_desc(frag_s + v * kBImg + ks * 256, 128, kBSbo);
            mma_f8(d, acol, bd, idesc, ks > 0 ? 1u : 0u);
          }
        }
        mma_commit(&mma_done[db]);
      }
      if (!ok) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ========================================================== softmax / value warps
    const int sw_ = warp - kEWarps;                       // 0..7
    const int q = warp & 3;                               // TMEM lane quadrant
    const int grp = sw_ >> 2;                             // tiles i ≡ grp (mod 2)
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const int g = lane >> 2, c = lane & 3;
    bool okp = ntiles == 0 || mbar_wait(&prol_bar, 0);
    if (!okp) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    float hA[2], hCm[2], hB[2], hCq[2];
    {
      const float* cst = reinterpret_cast<const float*>(smem + L::frag + NP * kBImg);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int col = 2 * c + k;
        hA[k] = cst[col * 4 + 0];
        hCm[k] = cst[col * 4 + 1];
        hB[k] = cst[col * 4 + 2];
        hCq[k] = cst[col * 4 + 3];
      }
    }
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f}, lw_run[2] = {0.f, 0.f};
    const uint32_t* lut_lane = reinterpret_cast<const uint32_t*>(smem + L::lut) + lane;

    for (int i = grp; i < ntiles && okp; i += 2) {
      const int st = (i >> 1) % kStages;
      const int hrow = (i & 1) * kTile;                   // the tile's first row in the stage
      const int db = i & 1;
      const bool okw = mbar_wait(&mma_done[db], (i >> 1) & 1) &&
                       mbar_wait(&full_bar[st], ((i >> 1) / kStages) & 1);
      if (!__all_sync(0xffffffffu, okw)) {   // the TMEM loads below are warp-collective
        if (lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
        break;
      }
      tc_after();
      // ---- accumulators → per-fragment sums: dm (index planes), dq (sign plane)
      float dm[2][4], dq[2][4];
#pragma unroll
      for (int T = 0; T < 2; ++T) {
#pragma unroll
        for (int e = 0; e < 4; ++e) dm[T][e] = dq[T][e] = 0.f;
        const uint32_t taddr = tmem + L::d_col + db * L::d_cols + lane_base +
                               ((uint32_t)(16 * T) << 16);
#pragma unroll
        for (int v = 0; v < NP; ++v) {
          uint32_t r[16];
          tmem_ld_16x256b_x4(taddr + v * kN, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float sum = (__uint_as_float(r[e]) + __uint_as_float(r[4 + e])) +
                              (__uint_as_float(r[8 + e]) + __uint_as_float(r[12 + e]));
            if (v < NKV) dm[T][e] += sum;
            else dq[T][e] = sum;
          }
        }
      }
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_free[db]);

      const unsigned char* base = smem + st * L::stage;
      const float* kxn = reinterpret_cast<const float*>(base + L::kxn) + hrow;
      const float* krn = reinterpret_cast<const float*>(base + L::krn) + hrow;
      const float* vxn = reinterpret_cast<const float*>(base + L::vxn) + hrow;
      const int t_tile = t_begin + i * kTile;
      const int r8 = lane & 7, m8 = (lane >> 3) & 1;
      // ---- scores → base-2 logits; rows: token g (k = 0) and g + 8 (k = 1) of each fragment
      float lg[2][2][2];
#pragma unroll
      for (int T = 0; T < 2; ++T)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int tl = 32 * q + 16 * T + g + 8 * k;
          const bool valid = t_tile + tl < t_end;
          const float xn = kxn[tl], rn = krn[tl];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float sc = xn * hA[h] * (dm[T][2 * k + h] - hCm[h]) +
                             rn * hB[h] * (dq[T][2 * k + h] - hCq[h]);
            lg[T][k][h] = valid ? sc : -INFINITY;
          }
        }
      // ---- online softmax over the warp's 32 tokens (per column pair)
      float mt[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float m = fmaxf(fmaxf(lg[0][0][h], lg[0][1][h]), fmaxf(lg[1][0][h], lg[1][1][h]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        mt[h] = fmaxf(m_run[h], m);
      }
      if (__any_sync(0xffffffffu, mt[0] > m_run[0] || mt[1] > m_run[1])) {
        float corr[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          corr[h] = m_run[h] == -INFINITY ? 0.f : exp2f(m_run[h] - mt[h]);
          l_run[h] *= corr[h];
          lw_run[h] *= corr[h];
          m_run[h] = mt[h];
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          acc[k][0] *= corr[0];
          acc[k][1] *= corr[1];
          acc[k][2] *= corr[0];
          acc[k][3] *= corr[1];
        }
      }
      float w[2][2][2];
#pragma unroll
      for (int T = 0; T < 2; ++T)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          // tokens past the sequence (or past the capacity in a short last tile) may hold
          // stale bytes: their weight is exactly zero, never 0 × (stale norm)
          const int tl = 32 * q + 16 * T + g + 8 * k;
          const bool valid = t_tile + tl < t_end;
          const float vn = vxn[tl];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float pr = valid ? exp2f(lg[T][k][h] - m_run[h]) : 0.f;
            l_run[h] += pr;
            w[T][k][h] = valid ? pr * vn : 0.f;
            lw_run[h] += w[T][k][h];
          }
        }
      // ---- value accumulation: acc[coord][column] += Σ_t A[coord][t] · B[t][column]
#pragma unroll
      for (int T = 0; T < 2; ++T) {
        const int trow0 = hrow + 32 * q + 16 * T;        // fragment's first token in the stage
        if constexpr (VB == 4) {
          uint32_t bw0, bw1;
          if (HILO) {
            const float h0 = __half2float(__float2half_rn(w[T][0][0]));
            const float h1 = __half2float(__float2half_rn(w[T][1][0]));
            bw0 = movm_t(pack_half2(h0, w[T][0][0] - h0));
            bw1 = movm_t(pack_half2(h1, w[T][1][0] - h1));
          } else {
            bw0 = movm_t(pack_half2(w[T][0][0], w[T][0][1]));
            bw1 = movm_t(pack_half2(w[T][1][0], w[T][1][1]));
          }
          // 8 code bytes (coordinates 16g..16g+15) of tokens 2c, 2c+1, 2c+8, 2c+9
          const unsigned char* vb = base + L::vcodes + (trow0 + 2 * c) * 64 + 8 * g;
          const uint2 u0 = *reinterpret_cast<const uint2*>(vb);
          const uint2 u1 = *reinterpret_cast<const uint2*>(vb + 64);
          const uint2 u2 = *reinterpret_cast<const uint2*>(vb + 8 * 64);
          const uint2 u3 = *reinterpret_cast<const uint2*>(vb + 9 * 64);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t A = half ? u0.y : u0.x, Bw = half ? u1.y : u1.x;
            const uint32_t C = half ? u2.y : u2.x, D = half ? u3.y : u3.x;
            // key byte i: low nibble = code of the first token, high nibble = second token
            const uint32_t klo01 = (A & 0x0f0f0f0fu) | ((Bw << 4) & 0xf0f0f0f0u);
            const uint32_t khi01 = ((A >> 4) & 0x0f0f0f0fu) | (Bw & 0xf0f0f0f0u);
            const uint32_t klo23 = (C & 0x0f0f0f0fu) | ((D << 4) & 0xf0f0f0f0u);
            const uint32_t khi23 = ((C >> 4) & 0x0f0f0f0fu) | (D & 0xf0f0f0f0u);
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const uint32_t a0 = lut_lane[((klo01 >> (8 * i4)) & 0xffu) << 5];
              const uint32_t a1 = lut_lane[((khi01 >> (8 * i4)) & 0xffu) << 5];
              const uint32_t a2 = lut_lane[((klo23 >> (8 * i4)) & 0xffu) << 5];
              const uint32_t a3 = lut_lane[((khi23 >> (8 * i4)) & 0xffu) << 5];
              mma16816(acc[4 * half + i4], a0, a1, a2, a3, bw0, bw1);
            }
          }
        } else {
          // planes transposed on load: pair word = {chunk g of token 2c, chunk g of token 2c+1}
          uint32_t mw[3][2] = {};
#pragma unroll
          for (int p = 0; p < VB; ++p)
            ldsm_x2_t(s32(base + L::vcodes + p * kStageTok * 16 + (trow0 + r8 + 8 * m8) * 16),
                      mw[p][0], mw[p][1]);
#pragma unroll
          for (int v = 0; v < NVV; ++v) {
            const float coef = a.vd.coef[v];
            uint32_t bw0, bw1;
            if (HILO) {
              const float x0 = coef * w[T][0][0], x1 = coef * w[T][1][0];
              const float h0 = __half2float(__float2half_rn(x0)), h1 = __half2float(__float2half_rn(x1));
              bw0 = movm_t(pack_half2(h0, x0 - h0));
              bw1 = movm_t(pack_half2(h1, x1 - h1));
            } else {
              bw0 = movm_t(pack_half2(coef * w[T][0][0], coef * w[T][0][1]));
              bw1 = movm_t(pack_half2(coef * w[T][1][0], coef * w[T][1][1]));
            }
            const uint32_t w0[3] = {mw[0][0], mw[1][0], mw[2][0]};
            const uint32_t w1[3] = {mw[0][1], mw[1][1], mw[2][1]};
            const Shifted e0 = shifted(vplane_word<VB < 4 ? VB : 1>(w0, v));
            const Shifted e1 = shifted(vplane_word<VB < 4 ? VB : 1>(w1, v));
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma16816(acc[k], pair_at(e0, 2 * k), pair_at(e0, 2 * k + 1), pair_at(e1, 2 * k),
                       pair_at(e1, 2 * k + 1), bw0, bw1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);
    }

    // ---------------------------------------------------------- combine the softmax warps
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], o);
        lw_run[h] += __shfl_xor_sync(0xffffffffu, lw_run[h], o);
      }
    }
    named_sync(kBarS, kSWarps * 32);   // every softmax warp is done with the ring: reuse it
    const int stid = tid - kEWarps * 32;
    float* cacc = reinterpret_cast<float*>(smem + L::comb_acc);     // [warp][col][140]
    float* cstat = reinterpret_cast<float*>(smem + L::comb_stats);  // [warp][3][8]
    float* fac = cstat + kSWarps * 3 * 8;                           // [warp][8]
    float* cML = fac + kSWarps * 8;                                 // M, L, LW [3][8]
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int hi_row = k >> 1;                  // 0: row g, 1: row g + 8
        const int col = 2 * c + (k & 1);
        int coord;
        float v = acc[k8][k];
        if (VB == 4) {
          coord = 16 * g + 2 * k8 + hi_row;
          v *= a.vc_unscale;
        } else {
          const int e = 2 * k8 + hi_row;
          coord = 16 * g + pair_lo(e);
          v *= exp2f((float)-pos_exp(pair_pos(e)));
        }
        cacc[accidx(sw_ * 8 + col, coord)] = v;
      }
    }
    if (g == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int col = 2 * c + k;
        cstat[(sw_ * 3 + 0) * 8 + col] = m_run[k];
        cstat[(sw_ * 3 + 1) * 8 + col] = l_run[k];
        cstat[(sw_ * 3 + 2) * 8 + col] = lw_run[k];
      }
    }
    named_sync(kBarS, kSWarps * 32);
    if (stid < 8) {
      const int col = stid;
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
    float* rec_base = a.part + ((bh * a.nsplit + split) * a.G) * kRec;
    for (int i = stid; i < a.G * TQ_D; i += kSWarps * 32) {
      const int head = i >> 7, j = i & 127;
      const int col = HILO ? 2 * head : head;
      float acc_j = 0.f;
#pragma unroll
      for (int wp = 0; wp < kSWarps; ++wp) {
        float av = cacc[accidx(wp * 8 + col, j)];
        if (HILO) av += cacc[accidx(wp * 8 + col + 1, j)];
        acc_j = fmaf(fac[wp * 8 + col], av, acc_j);
      }
      if (VB != 4) acc_j -= a.vd.cst * cML[16 + col];
      float* rec = rec_base + head * kRec;
      if (j == 0) {
        rec[0] = cML[col];        // base-2 maximum
        rec[1] = cML[8 + col];
      }
      rec[2 + j] = acc_j;
    }
    __threadfence();
    named_sync(kBarS, kSWarps * 32);
    if (stid == 0) s_ticket = atomicAdd(&a.counters[bh], 1);
  }

  // ============================================================ end of the split; last CTA merges
  tc_before();
  fence_async_smem();   // the merge's bulk copies overwrite shared memory written above
  named_sync(kBarAll, kCompute);
  tc_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
  if (s_ticket != a.nsplit - 1) return;
  __threadfence();
  // Stage Π (fp32) and as many split records as fit in shared memory with bulk copies; the
  // records of one (batch, KV head) are contiguous: [split][head][kRec]
  float* s_pi = reinterpret_cast<float*>(smem);                       // [128][128]
  float* s_rec = reinterpret_cast<float*>(smem + 65536);              // up to L::mrg_acc
  float* s_acc = reinterpret_cast<float*>(smem + L::mrg_acc);         // [8][128]
  float* s_w = reinterpret_cast<float*>(smem + L::mrg_w);             // [8][kMaxSplits]
  __shared__ float s_M[8], s_L[8];
  const long long rec_floats = (long long)a.nsplit * a.G * kRec;
  const int chunk_splits = (int)((L::mrg_acc - 65536) / (a.G * kRec * 4));
  const float* recs = a.part + bh * rec_floats;
  const bool one_chunk = a.nsplit <= chunk_splits;
  if (tid == 0) {
    // Π and the first (usually the only) chunk of records, in flight while the weights are
    // prepared
    const int ns = min(chunk_splits, a.nsplit);
    const unsigned bytes = (unsigned)(ns * a.G * kRec * 4);
    mbar_expect_tx(&mrg_bar, bytes + 65536u);
    bulk_g2s(s_pi, a.pi, 65536, &mrg_bar);
    bulk_g2s(s_rec, recs, bytes, &mrg_bar);
  }
  // warp h: maximum and weights of head h over the splits, from the staged records when
  // they all fit, else with plain loads (2 per split)
  auto weights = [&](const float* src, bool staged) {
    float mx = -INFINITY;
    for (int s = lane; s < a.nsplit; s += 32) {
      const long long o = ((long long)s * a.G + warp) * kRec;
      const float m = staged ? src[o] : __ldcg(&src[o]);
      const float l = staged ? src[o + 1] : __ldcg(&src[o + 1]);
      const float mm = l > 0.f ? m : -INFINITY;
      s_w[warp * kMaxSplits + s] = mm;
      mx = fmaxf(mx, mm);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float Ls = 0.f;
    for (int s = lane; s < a.nsplit; s += 32) {
      const long long o = ((long long)s * a.G + warp) * kRec + 1;
      const float mm = s_w[warp * kMaxSplits + s];
      const float wgt = (mx == -INFINITY || mm == -INFINITY) ? 0.f : exp2f(mm - mx);
      s_w[warp * kMaxSplits + s] = wgt;
      Ls += wgt * (staged ? src[o] : __ldcg(&src[o]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (lane == 0) {
      s_M[warp] = mx;
      s_L[warp] = Ls;
    }
  };
  if (!one_chunk && warp < a.G) weights(recs, false);
  float accv[3] = {0.f, 0.f, 0.f};   // thread's (head, j) items: tid, tid + kCompute, ...
  uint32_t mphase = 0;
  for (int s0 = 0; s0 < a.nsplit; s0 += chunk_splits) {
    const int ns = min(chunk_splits, a.nsplit - s0);
    if (tid == 0 && s0 > 0) {
      const unsigned bytes = (unsigned)(ns * a.G * kRec * 4);
      mbar_expect_tx(&mrg_bar, bytes);
      bulk_g2s(s_rec, recs + (long long)s0 * a.G * kRec, bytes, &mrg_bar);
    }
    if (!mbar_wait(&mrg_bar, mphase) && tid == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    mphase ^= 1;
    if (one_chunk) {
      if (warp < a.G) weights(s_rec, true);
    }
    named_sync(kBarAll, kCompute);   // weights ready and staged records visible
#pragma unroll
    for (int it = 0; it < 3; ++it) {
      const int item = tid + it * kCompute;
      if (item < a.G * TQ_D) {
        const int head = item >> 7, j = item & 127;
        const float* wv = s_w + head * kMaxSplits + s0;
        const float* rv = s_rec + head * kRec + 2 + j;
        const int step = a.G * kRec;
        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
        int sp = 0;
        for (; sp + 4 <= ns; sp += 4) {
          x0 = fmaf(wv[sp], rv[sp * step], x0);
          x1 = fmaf(wv[sp + 1], rv[(sp + 1) * step], x1);
          x2 = fmaf(wv[sp + 2], rv[(sp + 2) * step], x2);
          x3 = fmaf(wv[sp + 3], rv[(sp + 3) * step], x3);
        }
        for (; sp < ns; ++sp) x0 = fmaf(wv[sp], rv[sp * step], x0);
        accv[it] += (x0 + x1) + (x2 + x3);
      }
    }
    named_sync(kBarAll, kCompute);   // the staging buffer is free for the next chunk
  }
#pragma unroll
  for (int it = 0; it < 3; ++it) {
    const int item = tid + it * kCompute;
    if (item < a.G * TQ_D) s_acc[item] = accv[it];
  }
  named_sync(kBarAll, kCompute);
  // out_h = Πᵀ·acc_h / L_h: thread item (head, i)
#pragma unroll
  for (int it = 0; it < 3; ++it) {
    const int item = tid + it * kCompute;
    if (item < a.G * TQ_D) {
      const int head = item >> 7, i = item & 127;
      float o0 = 0.f, o1 = 0.f;
#pragma unroll 8
      for (int j = 0; j < TQ_D; j += 2) {
        o0 = fmaf(s_pi[j * TQ_D + i], s_acc[head * TQ_D + j], o0);
        o1 = fmaf(s_pi[(j + 1) * TQ_D + i], s_acc[head * TQ_D + j + 1], o1);
      }
      const float Lh = s_L[head];
      const float v = Lh > 0.f ? (o0 + o1) / Lh : 0.f;
      const long long e = ((long long)b * a.Hq + kvh * a.G + head) * TQ_D + i;
      if (a.out_dtype == TQ_F32) static_cast<float*>(a.out)[e] = v;
      else if (a.out_dtype == TQ_BF16) static_cast<__nv_bfloat16*>(a.out)[e] = __float2bfloat16_rn(v);
      else static_cast<__half*>(a.out)[e] = __float2half_rn(v);
    }
  }
  if (tid == 0) a.counters[bh] = 0;   // ready for the next call
}

template <int KB, int VB, bool HILO>
tq_status launch_one(const tq_mma_launch& a, cudaStream_t stream) {
  constexpr int smem = TL<KB, VB>::total;
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return TQ_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(decode_tc_kernel<KB, VB, HILO>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    configured[dev] = true;
  }
  query_prep_tc_kernel<KB, HILO><<<dim3(4, a.Hkv, a.B), kPrepThreads, 0, stream>>>(a);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nsplit, a.Hkv, a.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_tc_kernel<KB, VB, HILO>, a) != cudaSuccess)
    return TQ_ERR_CUDA;
  return tq_cuda_status(cudaGetLastError());
}

template <int KB, int VB>
tq_status launch_kv(const tq_mma_launch& a, cudaStream_t stream) {
  return a.G <= 4 ? launch_one<KB, VB, true>(a, stream) : launch_one<KB, VB, false>(a, stream);
}

template <int KB>
tq_status launch_k(const tq_mma_launch& a, cudaStream_t stream) {
  switch (a.vbits) {
    case 1: return launch_kv<KB, 1>(a, stream);
    case 2: return launch_kv<KB, 2>(a, stream);
    case 3: return launch_kv<KB, 3>(a, stream);
    case 4: return launch_kv<KB, 4>(a, stream);
  }
  return TQ_ERR_UNSUPPORTED;
}

}  // namespace

bool tq_tc_decode_supported(int kbits, int vbits, int G, int nsplit) {
  return kbits >= 1 && kbits <= 3 && vbits >= 1 && vbits <= 4 && G >= 1 && G <= 8 &&
         nsplit >= 1 && nsplit <= kMaxSplits;
}

size_t tq_tc_frag_bytes_max() { return (size_t)kMaxFragBlock; }

// Power-of-two scales of the query operand: the largest index-plane value is at most
// 0.5·max|coef| (|(Π q)_j| ≤ ‖q‖), the largest sign-plane value at most 1 (|(S q)_j| ≤
// smax·‖q‖); each scale puts that bound in [224, 448), inside the e4m3 range.
void tq_tc_operand_scales(const tq_plane_decomp& kd, float* s_idx, float* s_sgn) {
  float m = 0.f;
  for (int v = 0; v < kd.n; ++v) m = fmaxf(m, 0.5f * fabsf(kd.coef[v]));
  int e = 0;
  frexpf(448.f / (m > 0.f ? m : 1.f), &e);   // 448/m = f·2^e, f in [0.5, 1)
  *s_idx = ldexpf(1.f, e - 1);
  *s_sgn = 256.f;
}

tq_status tq_launch_decode_tc(const tq_mma_launch& a, cudaStream_t stream) {
  if (!tq_tc_decode_supported(a.kbits, a.vbits, a.G, a.nsplit)) return TQ_ERR_UNSUPPORTED;
  if (!a.counters || !a.qfrag) return TQ_ERR_INVALID_ARG;
  switch (a.kbits) {
    case 1: return launch_k<1>(a, stream);
    case 2: return launch_k<2>(a, stream);
    case 3: return launch_k<3>(a, stream);
  }
  return TQ_ERR_UNSUPPORTED;
}
