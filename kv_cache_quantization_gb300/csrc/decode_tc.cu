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
// A operand in TMEM with one AND/OR per four coordinates: bit r of every byte of a plane word
// becomes the byte a_r + b_r·bit (the bit set into the mantissa, exponent or sign of a constant,
// see expand_c).  The query operand B (shared memory) carries each query value divided by the
// b_r of its K position as four e4m3 "pieces" at their true scale (y ≈ p0 + p1 + p2 + p3,
// about 15 significant bits), one B row per (piece, column), so D column (piece, column) sums
// to the exact fp32 contraction of that piece plus a known constant (Σ a_r·y), and the softmax
// warps add the pieces and take the constant off.  Each plane is a 128 × N × 128 product: 4 MMAs
// of K = 32, issued by one thread per D block (N = 32: 8 head columns, or N = 16 for groups of
// at most 4 heads, each head's four pieces in two column pairs).
//
// Softmax and values.  Two groups of four softmax warps take alternate tiles.  A warp reads
// its 32 tokens' accumulators with the 16x256b TMEM load (register layout of the mma.sync
// accumulator fragment), keeps an online softmax per column and accumulates values with
// mma.sync m16n8k16 (4-bit codes through a pair table of fp16 levels, 1–3-bit codes as planes).
//
// Data path.  A producer warp streams 256-token stages of packed K/V through a 4-deep
// shared-memory ring with bulk copies (TMA engine).  The splits of one (batch, KV head) run as
// thread-block clusters of up to 4 CTAs, which build the query operand together at the start
// (each computes a quarter of Π q and S q and stores its bytes into every CTA of the cluster
// through distributed shared memory) while the ring fills.  At the end each CTA sends its
// (m, l, acc) per head to every CTA of its cluster; every CTA merges the cluster's results and
// rotates back its quarter of the output coordinates into the cluster's record.  The last CTA
// of a (batch, KV head) to finish (a ticket counter in the workspace) adds up the records with
// log-sum-exp weights.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "decode_args.h"
#include "tc_ptx.h"
#include "tile_mma.h"

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
// MMA N: 4 pieces × 8 head columns, or (group of at most 4 heads) 4 pieces × 4 heads
__host__ __device__ constexpr int kNof(bool hilo) { return hilo ? 16 : kPieces * 8; }
// one plane's query operand (4 KB or 2 KB of e4m3)
__host__ __device__ constexpr int kBImgOf(bool hilo) { return kNof(hilo) * 128; }
constexpr int kBSbo = 8 * 128;                // 8-row groups of the operand image
// score constants: 8 columns × {A, Cm, B, Cq}, then the operand offsets of the 4 slices
// ([slice][index planes | sign plane][8 columns], see query_prep_tc_kernel)
constexpr int kCstFloats = 8 * 4;
constexpr int kCstBytes = (kCstFloats + 4 * 2 * 8) * 4;
constexpr int kRec = TQ_REC;
constexpr int kPrepThreads = 256;
constexpr int kMaxSplits = 256;
constexpr int kAccPitch = 140;
// named barriers
constexpr int kBarS = 2, kBarAll = 3;

__host__ __device__ constexpr int accidx(int col, int j) { return col * kAccPitch + j + (j >> 4); }

// Bytes of the operand images per (batch, KV head): NP planes + score constants.
__host__ __device__ constexpr int frag_block(int np, bool hilo) {
  return np * kBImgOf(hilo) + kCstBytes;
}
constexpr int kMaxFragBlock = frag_block(5, false);

// The expander turns bit r of every byte of a plane word into one e4m3 byte by a single
// AND/OR: (word & (0x01 << r)) | C_r per byte.  The byte's value is a_r + b_r·bit: the bit
// lands in the mantissa (r < 3) or the exponent (3 ≤ r < 7) of the constant C_r, or (r = 7)
// in its sign.  The query operand at such a K position carries (intended value)/b_r, and the
// constant part Σ a_r·(operand) is taken off with the score constants.
__host__ __device__ constexpr uint32_t expand_c(int r) {
  return r == 0 ? 0x48484848u : r == 1 ? 0x40404040u : r == 2 ? 0x38383838u
       : r == 3 ? 0x30303030u : r == 4 ? 0x28282828u : r == 5 ? 0x18181818u
       : r == 6 ? 0u : 0x38383838u;
}
// a_r and 1/b_r of the expanded byte a_r + b_r·bit
__host__ __device__ constexpr float expand_a(int r) {
  return r == 0 ? 4.f : r == 1 ? 2.f : r == 2 ? 1.f : r == 3 ? 0.5f : r == 4 ? 0.25f
       : r == 5 ? 0.0625f : r == 6 ? 0.f : 1.f;
}
__host__ __device__ constexpr float expand_inv_b(int r) {
  return r <= 3 ? 2.f : r == 4 ? 4.f / 3.f : r == 5 ? 16.f / 15.f : r == 6 ? 0.5f : -0.5f;
}

// Operand K position k of plane word i (coordinates 32i..32i+31): column c = k / 4 =
// 8i + r holds coordinates 32i + 8b + r in its bytes b = 0..3.
__host__ __device__ constexpr int coord_of_k(int k) {
  return 32 * (k >> 5) + 8 * (k & 3) + ((k >> 2) & 7);
}
// canonical K-major offset of byte (row n < 32, k < 128) in one plane's e4m3 operand
__host__ __device__ constexpr int bimg_off(int n, int k) {
  return (n >> 3) * kBSbo + (k >> 4) * 128 + (n & 7) * 16 + (k & 15);
}
// operand row of piece p of column n: p·8 + n, or (4-head layout) rows 2n, 2n + 1, 8 + 2n,
// 9 + 2n, so that the accumulator-fragment load gives lane (g, c) the four pieces of head c
__host__ __device__ constexpr int bimg_row(bool hilo, int p, int n) {
  return hilo ? (p >> 1) * 8 + 2 * n + (p & 1) : p * 8 + n;
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

__device__ __forceinline__ void tmem_ld_16x256b_x2(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

// true in exactly one lane of the (converged) warp
__device__ __forceinline__ bool elect_one() {
  uint32_t p;
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n selp.u32 %0, 1, 0, e;\n}\n"
      : "=r"(p));
  return p != 0;
}

__device__ __forceinline__ float e4m3_value(__nv_fp8_storage_t x) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(x, __NV_E4M3)));
}

// ---------------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_ctas() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// the shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void fence_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
// arrive on the mbarrier at `saddr` in CTA `rank`, ordering this thread's earlier writes
__device__ __forceinline__ void arrive_remote(uint32_t saddr, uint32_t rank) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   map_rank(saddr, rank))
               : "memory");
}
// bounded wait with cluster-scope acquire (the phase was completed by arrivals of peers)
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, unsigned parity) {
  auto try1 = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(s32(bar)), "r"(parity), "r"(10000000u)
        : "memory");
    return ok != 0;
  };
  if (try1()) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (try1()) return true;
    if (global_ns() - t0 > 20000000ull) return false;
  }
}
// cluster-wide barrier in two halves: every thread of every CTA arrives once (at kernel
// start, after its mbarriers are initialised) and waits before its first remote mbarrier
// access, so the barrier's latency hides behind the work in between
__device__ __forceinline__ void cluster_arrive_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_all() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- query operand kernel
// Grid (4 slices, KV heads, batch).  The CTA for slice s computes (Π q_h)_j and (S q_h)_j
// for the group's heads h and coordinates j = 32s..32s+31 (plane word s), and writes the
// operand bytes of K positions 32s..32s+31 of every plane: row (piece p, column n) holds
// piece p of coef_v·(Π q)_j/‖q‖·s_idx (index plane v) or 2·(S q)_j/(‖q‖·smax)·s_sgn (sign
// plane), divided by the b_r of the K position's expanded A byte; column n = head n.  ‖q‖ and
// the column sums (Πᵀ1)·q, (Sᵀ1)·q come straight from q, so no slice needs another slice's
// results; each slice writes its share of the operand offsets Σ a_r·(operand).
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
  float uk[4], wk[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uk[k] = __ldg(&a.u[lane + 32 * k]);
    wk[k] = __ldg(&a.w[lane + 32 * k]);
  }
  __syncthreads();
  if (warp < a.G) {
    // ‖q‖, (Πᵀ1)·q and (Sᵀ1)·q of head `warp`
    float n2 = 0.f, uq = 0.f, wq = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = lane + 32 * k;
      const float x = qf[warp][j];
      n2 = fmaf(x, x, n2);
      uq = fmaf(uk[k], x, uq);
      wq = fmaf(wk[k], x, wq);
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
  constexpr int kBImg = kBImgOf(HILO);
  unsigned char* out = static_cast<unsigned char*>(a.qfrag) + bh * (long long)frag_block(NP, HILO);
  float* cst = reinterpret_cast<float*>(out + NP * kBImg);
  {
    // Warp n: column n (head n); lane: K position 32s + lane; plane after plane.  A set bit
    // must contribute 2x (x: the half-scaled operand value below), and the expanded A byte at
    // this K position is a_r + b_r·bit, so the operand is y = 2x/b_r, stored as four e4m3
    // pieces; the warp adds up a_r·(sum of the pieces) over its K positions: the constant the
    // MMAs add to the column, which the softmax warps take off.
    const int n = warp, kl = lane;
    const int k = 32 * s + kl;
    const int jl2 = coord_of_k(k) - 32 * s;
    const int r = (k >> 2) & 7;
    const float ar = expand_a(r), ib = expand_inv_b(r);
    const bool col_ok = !HILO || n < 4;
    float off_idx = 0.f, off_sgn = 0.f;
    for (int v = 0; v < NP && col_ok; ++v) {
      float x = 0.f;
      if (n < a.G && s_nq[n] > 0.f) {
        const float nq = s_nq[n];
        x = v < NKV ? 0.5f * a.kd.coef[v] * qs[0][n][jl2] / nq * a.s_idx
                    : qs[1][n][jl2] / (nq * a.smax) * a.s_sgn;
      }
      float y = 2.f * x * ib, yhat = 0.f;
#pragma unroll
      for (int p = 0; p < kPieces; ++p) {
        const __nv_fp8_storage_t e = __nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
        const float pv = e4m3_value(e);
        y -= pv;
        yhat += pv;
        out[v * kBImg + bimg_off(bimg_row(HILO, p, n), k)] = e;
      }
      if (v < NKV) off_idx = fmaf(ar, yhat, off_idx);
      else off_sgn = fmaf(ar, yhat, off_sgn);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      off_idx += __shfl_xor_sync(0xffffffffu, off_idx, o);
      off_sgn += __shfl_xor_sync(0xffffffffu, off_sgn, o);
    }
    if (lane == 0 && col_ok) {
      float* offp = cst + kCstFloats + s * 16;   // [index planes | sign plane][8 columns]
      const int c0 = HILO ? 2 * n : n;
      offp[c0] = off_idx;
      offp[8 + c0] = off_sgn;
      if (HILO) {
        offp[c0 + 1] = off_idx;
        offp[8 + c0 + 1] = off_sgn;
      }
    }
  }
  if (s == 0 && tid < 8) {
    // score constants of column n: A, Cm, B, Cq (see the softmax warps)
    const int n = tid, head = HILO ? n >> 1 : n;
    const float nq = head < a.G ? s_nq[head] : 0.f;
    const bool ok = nq > 0.f;
    cst[n * 4 + 0] = nq * a.scale_log2 / a.s_idx;
    cst[n * 4 + 1] = ok ? a.s_idx * a.kd.cst * s_uq[head] / nq : 0.f;
    cst[n * 4 + 2] = nq * a.smax * a.scale_log2 * (1.2533141373155003f / TQ_D) / a.s_sgn;
    cst[n * 4 + 3] = ok ? a.s_sgn * s_wq[head] / (nq * a.smax) : 0.f;
  }
}

// ---------------------------------------------------------------- shared memory and TMEM
template <int KB, int VB, bool HILO>
struct TL {
  static constexpr int NP = num_vplanes(KB) + 1;             // planes incl. the sign plane
  static constexpr int kN = kNof(HILO);                      // MMA N (D columns per block)
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
  static constexpr int used = frag + frag_block(NP, HILO);
  // the slots for the per-CTA results of the cluster (up to 4 × (16 + 8·128) floats)
  static constexpr int slots = used;
  static constexpr int total = slots + 4 * (16 + 8 * 128) * 4;
  // after the main loop the ring is reused: softmax-warp accumulators and statistics (later
  // the merged accumulators [8][128]), then rows of Πᵀ (512 bytes each) for the rotation back;
  // the last CTA's merge keeps its weights [2][8][kMaxSplits] at the start
  static constexpr int comb_acc = 0;
  static constexpr int comb_stats = kSWarps * 8 * kAccPitch * 4;
  static constexpr int pi_off = (comb_stats + (kSWarps * 4 + 3 + 4) * 8 * 4 + 127) / 128 * 128;
  static constexpr int pi_rows = (ring - pi_off) / 512 / 32 * 32;   // rows per chunk
  static_assert(pi_rows >= 32, "rotation rows");
  static_assert(2 * 8 * kMaxSplits * 4 <= ring, "merge weights");
  // TMEM: A (one tile: NP planes × 32 columns of e4m3), D (NP planes × 32 columns)
  static constexpr int a_cols = NP * 32;
  // D: index planes summed in pairs by the MMAs (block j = planes 2j, 2j + 1), then the sign
  // plane's block
  static constexpr int d_blocks = (NP - 1 + 1) / 2 + 1;
  static constexpr int d_cols = d_blocks * kN;
  static constexpr int abufs = (2 * a_cols + 2 * d_cols <= 512) ? 2 : 1;
  static constexpr int d_col = abufs * a_cols;
  static_assert(d_col + 2 * d_cols <= 512, "TMEM columns");
};

// ---------------------------------------------------------------- the split kernel
template <int KB, int VB, bool HILO>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const tq_mma_launch a) {
  using L = TL<KB, VB, HILO>;
  constexpr int kN = L::kN;
  constexpr int kBImg = kBImgOf(HILO);
  constexpr int NKV = num_vplanes(KB);
  constexpr int NP = NKV + 1;
  constexpr int NVV = VB == 4 ? 0 : num_vplanes(VB);
  constexpr int NI = L::d_blocks;                              // issuer warps: one per D block
  static_assert(L::d_blocks <= kIWarps, "issuer warps");
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t mma_done[2];
  __shared__ __align__(8) uint64_t d_free[2];
  __shared__ __align__(8) uint64_t a_full[2];
  __shared__ __align__(8) uint64_t prol_bar;   // query operand (and value pair table) landed
  __shared__ __align__(8) uint64_t comb_bar;   // every CTA's result is in this CTA's slots
  __shared__ __align__(8) uint64_t pi_bar;     // rows of Πᵀ landed
  __shared__ __align__(8) uint64_t rec_bar;    // (leader) every CTA of the cluster wrote its record part
  __shared__ __align__(8) uint64_t last_bar;   // the leader's verdict (s_last) arrived
  __shared__ __align__(8) uint64_t mrg_bar;    // a chunk of record slices landed
  __shared__ float s_hM[8], s_hL[8];
  __shared__ int s_last;
  __shared__ uint32_t s_tmem;
  __shared__ int s_ticket;

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long bh = (long long)b * a.Hkv + kvh;
  // the warp index through a shuffle: the compiler then knows it is warp-uniform and keeps
  // the TMEM addresses derived from it in uniform registers
  const int tid = threadIdx.x, warp = __shfl_sync(0xffffffffu, tid >> 5, 0), lane = tid & 31;
  const uint32_t rank = cluster_rank(), C = cluster_ctas();
  int len = a.seq_lens[b];
  if (len > a.cap) {
    if (tid == 0 && split == 0 && kvh == 0) atomicOr(&g_tq_flags, TQ_FLAG_LEN_OVERFLOW);
    len = a.cap;
  }
  const int t_begin = split * a.split_len;
  const int t_end = min(t_begin + a.split_len, len);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;
  const int nstages = (ntiles + 1) / 2;
  // Without clusters only the splits that hold tokens take part (ragged batches launch many
  // empty ones): an empty split leaves at once, and a sequence without tokens gets its zero
  // output from split 0.
  const int used = C == 1 ? (len + a.split_len - 1) / a.split_len : a.nsplit;
  if (C == 1 && ntiles == 0) {
    if (len == 0 && split == 0)
      for (int i = tid; i < a.G * TQ_D; i += kThreads) {
        const long long e = ((long long)b * a.Hq + kvh * a.G) * TQ_D + i;
        if (a.out_dtype == TQ_F32) static_cast<float*>(a.out)[e] = 0.f;
        else if (a.out_dtype == TQ_BF16) static_cast<__nv_bfloat16*>(a.out)[e] = __float2bfloat16_rn(0.f);
        else static_cast<__half*>(a.out)[e] = __float2half_rn(0.f);
      }
    return;
  }
  const int cid = split / (int)C, nclus = used / (int)C;

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
    mbar_init(&comb_bar, C);
    mbar_init(&pi_bar, 1);
    mbar_init(&rec_bar, C);
    mbar_init(&last_bar, 1);
    mbar_init(&mrg_bar, 1);
    mbar_init_fence();
    s_ticket = -1;
  }
  if (warp == 0) tmem_alloc(&s_tmem, 512);
  tc_before();
  __syncthreads();
  tc_after();
  // every CTA of the cluster initialises its barriers before any remote access (the wait half
  // comes just before the first remote store, at the end of the split)
  if (C > 1) cluster_arrive_all();
  const uint32_t tmem = s_tmem;

  // output coordinates i0..i0+R of this CTA (the rotation back and the final merge), and the
  // chunks of prow rows of Πᵀ that the rotation back stages in the ring
  const int R = TQ_D / (int)C, i0 = (int)rank * R;
  const int prow = R < L::pi_rows ? R : L::pi_rows;

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
      // the ring fills while the query-operand kernel (this grid's programmatic-launch
      // primary) runs; its output is copied in as soon as that grid has completed
      int c = 0;
      for (; c < nstages && c < kStages; ++c) issue(c);
      asm volatile("griddepcontrol.wait;" ::: "memory");
      mbar_expect_tx(&prol_bar, frag_block(NP, HILO) + L::lut_bytes);
      bulk_g2s(smem + L::frag,
               static_cast<const unsigned char*>(a.qfrag) + bh * (long long)frag_block(NP, HILO),
               frag_block(NP, HILO), &prol_bar);
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
    if (C > 1) cluster_wait_all();
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
          // column 8·w4 + r: byte b = bit 8b + r of the word as the e4m3 byte a_r + b_r·bit
          // (one AND/OR per four coordinates)
#pragma unroll
          for (int r = 0; r < 8; ++r) col[8 * w4 + r] = (x & (0x01010101u << r)) | expand_c(r);
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
    // Issuer iw owns D block iw: index planes 2iw and 2iw + 1 accumulated into one block, or
    // (last block) the sign plane; 4 MMAs of K = 32 per plane and tile, D[i & 1].  The whole
    // warp waits and forms the (warp-uniform) descriptors; one elected lane issues the MMAs
    // and their commit.
    const int iw = warp - kEWarps - kSWarps;
    if (iw < NI && ntiles > 0) {
      const uint32_t idesc = idesc_f16(128, kN);   // e4m3 × e4m3 → f32 has the same fields
      const uint32_t frag_s = s32(smem + L::frag);
      const bool sign_blk = iw == NI - 1;
      const int v0 = sign_blk ? NKV : 2 * iw;
      const int nv = sign_blk ? 1 : (2 * iw + 1 < NKV ? 2 : 1);
      uint64_t bdesc[2][4];
#pragma unroll
      for (int o = 0; o < 2; ++o)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          bdesc[o][ks] = smem_desc(frag_s + (v0 + (o < nv ? o : 0)) * kBImg + ks * 256, 128, kBSbo);
      bool ok = mbar_wait(&prol_bar, 0);
      for (int i = 0; i < ntiles && ok; ++i) {
        const int ab = L::abufs == 2 ? (i & 1) : 0;
        const int db = i & 1;
        ok = mbar_wait(&a_full[ab], (i / L::abufs) & 1) &&
             (i < 2 || mbar_wait(&d_free[db], ((i - 2) >> 1) & 1));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_after();
        if (elect_one()) {
          const uint32_t d = tmem + L::d_col + db * L::d_cols + iw * kN;
#pragma unroll
          for (int o = 0; o < 2; ++o) {
            if (o < nv) {
              const uint32_t a0 = tmem + ab * L::a_cols + 32 * (v0 + o);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_f8(d, a0 + 8 * ks, bdesc[o][ks], idesc, (o > 0 || ks > 0) ? 1u : 0u);
            }
          }
          mma_commit(&mma_done[db]);
        }
        __syncwarp();
      }
      if (!ok && lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ========================================================== softmax / value warps
    const int sw_ = warp - kEWarps;                       // 0..7
    const int q = warp & 3;                               // TMEM lane quadrant
    const int grp = sw_ >> 2;                             // tiles i ≡ grp (mod 2)
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const int g = lane >> 2, c = lane & 3;
    // the operand constants (and the cluster's stores into this CTA) are complete
    bool okp = mbar_wait(&prol_bar, 0);
    if (!okp) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    float hA[2], hCm[2], hB[2], hCq[2];
    {
      const float* cst = reinterpret_cast<const float*>(smem + L::frag + NP * kBImg);
      const float* offp = cst + kCstFloats;   // [slice][index planes | sign plane][column]
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int col = 2 * c + k;
        hA[k] = cst[col * 4 + 0];
        hCm[k] = cst[col * 4 + 1] + ((offp[col] + offp[16 + col]) + (offp[32 + col] + offp[48 + col]));
        hB[k] = cst[col * 4 + 2];
        hCq[k] = cst[col * 4 + 3] +
                 ((offp[8 + col] + offp[24 + col]) + (offp[40 + col] + offp[56 + col]));
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
      // ---- accumulators → per-fragment sums: dm (index planes), dq (sign plane).  A block
      // is kN columns: 4 pieces × 8 head columns (rows g, g + 8 and columns 2c, 2c + 1 in
      // registers e = 2·row + h), or 4 pieces × 4 heads (head c's pieces in columns 2c, 2c + 1
      // of the block's two repetitions; sums in e = 0 and 2).
      constexpr int NH = HILO ? 1 : 2;
      constexpr int NB = L::d_blocks;
      constexpr int RPB = kN / 8;              // 16x256b repetitions per block
      constexpr int NREP = NB * RPB;
      float dm[2][4], dq[2][4];
#pragma unroll
      for (int T = 0; T < 2; ++T) {
#pragma unroll
        for (int e = 0; e < 4; ++e) dm[T][e] = dq[T][e] = 0.f;
        const uint32_t taddr = tmem + L::d_col + db * L::d_cols + lane_base +
                               ((uint32_t)(16 * T) << 16);
#pragma unroll
        for (int r0 = 0; r0 < NREP; r0 += 8) {
          uint32_t r[32];
          const int nr = NREP - r0 < 8 ? NREP - r0 : 8;
          if (nr == 8) {
            tmem_ld_16x256b_x8(taddr + 8 * r0, r);
          } else {
            if (nr >= 4) tmem_ld_16x256b_x4(taddr + 8 * r0, r);
            if (nr == 2 || nr == 6) tmem_ld_16x256b_x2(taddr + 8 * (r0 + nr - 2), r + 4 * (nr - 2));
          }
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (u < nr) {
              const int R = r0 + u, j = R / RPB;
              float* tgt = j < NB - 1 ? dm[T] : dq[T];
              const uint32_t* rr = r + 4 * u;
              if (HILO) {
                tgt[0] += __uint_as_float(rr[0]) + __uint_as_float(rr[1]);
                tgt[2] += __uint_as_float(rr[2]) + __uint_as_float(rr[3]);
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) tgt[e] += __uint_as_float(rr[e]);
              }
            }
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
          for (int h = 0; h < NH; ++h) {
            const float sc = xn * hA[h] * (dm[T][2 * k + h] - hCm[h]) +
                             rn * hB[h] * (dq[T][2 * k + h] - hCq[h]);
            lg[T][k][h] = valid ? sc : -INFINITY;
          }
          if (NH == 1) lg[T][k][1] = lg[T][k][0];
        }
      bool okt[2][2];
#pragma unroll
      for (int T = 0; T < 2; ++T)
#pragma unroll
        for (int k = 0; k < 2; ++k) okt[T][k] = t_tile + 32 * q + 16 * T + g + 8 * k < t_end;
      softmax_values_step<VB, HILO>(lg, okt, vxn + 32 * q,
                                    base + L::vcodes + (hrow + 32 * q) * (VB == 4 ? 64 : 16),
                                    kStageTok * 16, lut_lane, a.vd.coef, acc, m_run, l_run,
                                    lw_run, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);
    }

    // ---------------------------------------------------------- combine the softmax warps
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
    const int stid = tid - kEWarps * 32;
    // the first chunk of Πᵀ rows is in flight during the combine
    if (stid == 0) {
      mbar_expect_tx(&pi_bar, (unsigned)prow * 512u);
      bulk_g2s(smem + L::pi_off, a.vpiT + (long long)i0 * TQ_D, (unsigned)prow * 512u, &pi_bar);
    }
    float* cacc = reinterpret_cast<float*>(smem + L::comb_acc);     // [warp][col][140]
    float* cstat = reinterpret_cast<float*>(smem + L::comb_stats);  // [warp][3][8]
    float* fac = cstat + kSWarps * 3 * 8;                           // [warp][8]
    float* cML = fac + kSWarps * 8;                                 // M, L, LW [3][8], then [8][4]
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
    // ---- this CTA's per-head result (M, L, acc[128]) into slot `rank` of every CTA of the
    // cluster
    constexpr int kSlot = 16 + 8 * TQ_D;
    float* slots = reinterpret_cast<float*>(smem + L::slots);  // [C][M[8], L[8], acc[8][128]]
    const uint32_t slots_s = s32(slots);
    if (C > 1) cluster_wait_all();   // every peer's barriers are initialised
    // item (head, 4 coordinates): the combined values, stored as one 16-byte word per CTA
    for (int it = stid; it < a.G * (TQ_D / 4); it += kSWarps * 32) {
      const int head = it >> 5, j0 = 4 * (it & 31);
      const int col = HILO ? 2 * head : head;
      float v4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = j0 + e;
        float acc_j = 0.f;
#pragma unroll
        for (int wp = 0; wp < kSWarps; ++wp) {
          float av = cacc[accidx(wp * 8 + col, j)];
          if (HILO) av += cacc[accidx(wp * 8 + col + 1, j)];
          acc_j = fmaf(fac[wp * 8 + col], av, acc_j);
        }
        if (VB != 4) acc_j -= a.vd.cst * cML[16 + col];
        v4[e] = acc_j;
      }
      const uint4 u = make_uint4(__float_as_uint(v4[0]), __float_as_uint(v4[1]),
                                 __float_as_uint(v4[2]), __float_as_uint(v4[3]));
      const int off = (int)rank * kSlot + 16 + head * TQ_D + j0;
      for (uint32_t d = 0; d < C; ++d) {
        if (d == rank) *reinterpret_cast<uint4*>(slots + off) = u;
        else st_cluster_v4(map_rank(slots_s + 4u * off, d), u);
      }
      if (j0 == 0) {
        const int o = (int)rank * kSlot + head;
        for (uint32_t d = 0; d < C; ++d) {
          if (d == rank) {
            slots[o] = cML[col];                       // base-2 maximum
            slots[o + 8] = cML[8 + col];
          } else {
            st_cluster_f32(map_rank(slots_s + 4u * o, d), cML[col]);
            st_cluster_f32(map_rank(slots_s + 4u * (o + 8), d), cML[8 + col]);
          }
        }
      }
    }
    if (C > 1) fence_cluster();
    named_sync(kBarS, kSWarps * 32);
    if (stid < (int)C) {
      if (stid == (int)rank) mbar_arrive(&comb_bar);
      else arrive_remote(s32(&comb_bar), (uint32_t)stid);
    }
    // ---- merge the cluster's C results (every CTA does it; they agree bit for bit): weights
    // per head first, then 4 coordinates per item
    bool okc = C == 1 ? mbar_wait(&comb_bar, 0) : mbar_wait_cluster(&comb_bar, 0);
    if (!okc && stid == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    float* cw = cML + 24;                                         // [8][4] slot weights
    if (stid < a.G) {
      const int head = stid;
      float M = -INFINITY;
      for (uint32_t r = 0; r < C; ++r)
        if (slots[r * kSlot + 8 + head] > 0.f) M = fmaxf(M, slots[r * kSlot + head]);
      float Ls = 0.f;
      for (uint32_t r = 0; r < C; ++r) {
        const float l = slots[r * kSlot + 8 + head];
        const float wr = (M == -INFINITY || !(l > 0.f)) ? 0.f : exp2f(slots[r * kSlot + head] - M);
        cw[head * 4 + r] = wr;
        Ls = fmaf(wr, l, Ls);
      }
      s_hM[head] = M;
      s_hL[head] = Ls;
    }
    named_sync(kBarS, kSWarps * 32);
    float* mrg = reinterpret_cast<float*>(smem + L::comb_acc);   // [8][128], after cacc is read
    for (int it = stid; it < a.G * (TQ_D / 4); it += kSWarps * 32) {
      const int head = it >> 5, j0 = 4 * (it & 31);
      float4 m4 = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t r = 0; r < C; ++r) {
        const float wr = cw[head * 4 + r];
        const float4 v = *reinterpret_cast<const float4*>(slots + r * kSlot + 16 + head * TQ_D + j0);
        m4.x = fmaf(wr, v.x, m4.x);
        m4.y = fmaf(wr, v.y, m4.y);
        m4.z = fmaf(wr, v.z, m4.z);
        m4.w = fmaf(wr, v.w, m4.w);
      }
      *reinterpret_cast<float4*>(mrg + head * TQ_D + j0) = m4;
    }
  }

  // ============================================================ end of the split
  // every compute warp: rotate back this CTA's output rows of the merged accumulators into the
  // cluster's record, then the ticket
  tc_before();
  named_sync(kBarAll, kCompute);
  tc_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
  {
    const float* mrg = reinterpret_cast<const float*>(smem + L::comb_acc);   // [8][128]
    float* rec_base = a.part + ((bh * (a.nsplit / (int)C) + cid) * a.G) * kRec;
    const float4* pis = reinterpret_cast<const float4*>(smem + L::pi_off);  // [prow][32]
    for (int c0 = 0, ph = 0; c0 < R; c0 += prow, ph ^= 1) {
      if (c0 > 0) {
        named_sync(kBarAll, kCompute);   // the previous chunk is consumed
        if (tid == 0) {
          mbar_expect_tx(&pi_bar, (unsigned)prow * 512u);
          bulk_g2s(smem + L::pi_off, a.vpiT + (long long)(i0 + c0) * TQ_D, (unsigned)prow * 512u,
                   &pi_bar);
        }
      }
      const bool okp2 = mbar_wait(&pi_bar, (unsigned)ph);
      if (!okp2 && lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
      // task (head, 32-row group) per warp; lane = output row; the j loop starts at a
      // lane-dependent offset so that the float4 reads of both operands are free of bank
      // conflicts
      const int ngrp = prow / 32;
      for (int task = warp; okp2 && task < a.G * ngrp; task += kCompute / 32) {
        const int h = task / ngrp, r = (task - h * ngrp) * 32 + lane;
        const float4* mh = reinterpret_cast<const float4*>(mrg + h * TQ_D);
        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll 8
        for (int jj = 0; jj < 32; ++jj) {
          const int jq = (jj + lane) & 31;
          const float4 pv = pis[r * 32 + jq];
          const float4 mv = mh[jq];
          o0 = fmaf(pv.x, mv.x, o0);
          o1 = fmaf(pv.y, mv.y, o1);
          o2 = fmaf(pv.z, mv.z, o2);
          o3 = fmaf(pv.w, mv.w, o3);
        }
        rec_base[h * kRec + 4 + i0 + c0 + r] = (o0 + o1) + (o2 + o3);
      }
    }
    if (rank == 0 && tid < a.G) {
      rec_base[tid * kRec] = s_hM[tid];
      rec_base[tid * kRec + 1] = s_hL[tid];
    }
  }
  named_sync(kBarAll, kCompute);
  if (tid == 0) {
    // this CTA's part of the record is released at device scope; the leader, once every CTA
    // of the cluster has reported, takes the cluster's ticket and tells the cluster whether
    // it was the last one of the (batch, KV head)
    fence_gpu();
    if (rank == 0) mbar_arrive(&rec_bar);
    else arrive_remote(s32(&rec_bar), 0);
    bool okt = true;
    if (rank == 0) {
      okt = C == 1 ? mbar_wait(&rec_bar, 0) : mbar_wait_cluster(&rec_bar, 0);
      fence_gpu();
      const int last = atomicAdd(&a.counters[bh], 1) == nclus - 1 ? 1 : 0;
      for (uint32_t d = 0; d < C; ++d) {
        if (d == 0) {
          s_last = last;
          mbar_arrive(&last_bar);
        } else {
          st_cluster_s32(map_rank(s32(&s_last), d), last);
          arrive_remote(s32(&last_bar), d);
        }
      }
    }
    okt = (C == 1 ? mbar_wait(&last_bar, 0) : mbar_wait_cluster(&last_bar, 0)) && okt;
    if (!okt) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    s_ticket = okt ? s_last : 0;
  }
  named_sync(kBarAll, kCompute);
  if (s_ticket != 1) return;
  // Every record (one per cluster) is rotated back already: out_h = Σ_r w_r·rec_r / Σ_r w_r·L_r
  // with w_r = 2^(M_r − max M).  CTA `rank` of the last cluster produces output coordinates
  // i0..i0+R.  Without clusters the records are contiguous and arrive by bulk copy, in chunks
  // that fit in shared memory; in a cluster each CTA loads its 128-byte slices directly (few
  // small bulk copies would cost more than they save).  Warp h computes the weights of head h.
  if (tid == 0) {
    fence_gpu();
    fence_proxy_async_global();
  }
  named_sync(kBarAll, kCompute);
  const float* recs = a.part + bh * (long long)(a.nsplit / (int)C) * a.G * kRec;
  float* sa = reinterpret_cast<float*>(smem);                          // C == 1: [chunk][G][kRec]
  float* s_w = reinterpret_cast<float*>(smem + L::slots);              // [2][8][kMaxSplits]
  const int chunk = C == 1 ? min(nclus, (int)(L::slots / (a.G * kRec * 4))) : nclus;
  auto issue_chunk = [&](int r0) {
    const int n = min(chunk, nclus - r0);
    const unsigned bytes = (unsigned)(n * a.G * kRec * 4);
    mbar_expect_tx(&mrg_bar, bytes);
    bulk_g2s(sa, recs + (long long)r0 * a.G * kRec, bytes, &mrg_bar);
  };
  if (C == 1 && tid == 0) issue_chunk(0);
  constexpr int kPre = 16;
  float pv[kPre];
  const bool slice_item = C > 1 && tid < a.G * R;   // R ≤ 64 here: one item per thread
  const int sh = slice_item ? tid / R : 0, si = slice_item ? tid - sh * R : 0;
#pragma unroll
  for (int r = 0; r < kPre; ++r)
    pv[r] = (slice_item && r < nclus)
                ? __ldcg(&recs[((long long)r * a.G + sh) * kRec + 4 + i0 + si]) : 0.f;
  if (warp < a.G) {
    float mx = -INFINITY;
#pragma unroll 4
    for (int r = lane; r < nclus; r += 32) {
      const long long o = ((long long)r * a.G + warp) * kRec;
      const float m = __ldcg(&recs[o]), l = __ldcg(&recs[o + 1]);
      const float mm = l > 0.f ? m : -INFINITY;
      s_w[warp * kMaxSplits + r] = mm;
      mx = fmaxf(mx, mm);
      s_w[(8 + warp) * kMaxSplits + r] = l;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float Ls = 0.f;
    for (int r = lane; r < nclus; r += 32) {
      const float mm = s_w[warp * kMaxSplits + r];
      const float wgt = (mx == -INFINITY || mm == -INFINITY) ? 0.f : exp2f(mm - mx);
      s_w[warp * kMaxSplits + r] = wgt;
      Ls += wgt * s_w[(8 + warp) * kMaxSplits + r];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (lane == 0) s_hL[warp] = Ls;
  }
  named_sync(kBarAll, kCompute);   // weights ready
  constexpr int kItems = (8 * TQ_D + kCompute - 1) / kCompute;
  float x[kItems] = {};
  if (C > 1) {
    if (slice_item) {
      const float* wv = s_w + sh * kMaxSplits;
      float x0 = 0.f, x1 = 0.f;
#pragma unroll
      for (int r = 0; r < kPre; r += 2) {
        if (r < nclus) x0 = fmaf(wv[r], pv[r], x0);
        if (r + 1 < nclus) x1 = fmaf(wv[r + 1], pv[r + 1], x1);
      }
      for (int r0 = kPre; r0 < nclus; r0 += kPre) {   // beyond the prefetched records
#pragma unroll
        for (int r = 0; r < kPre; ++r)
          pv[r] = r0 + r < nclus ? __ldcg(&recs[((long long)(r0 + r) * a.G + sh) * kRec + 4 + i0 + si]) : 0.f;
#pragma unroll
        for (int r = 0; r < kPre; ++r)
          if (r0 + r < nclus) x0 = fmaf(wv[r0 + r], pv[r], x0);
      }
      x[0] = x0 + x1;
    }
  } else {
    uint32_t mphase = 0;
    for (int r0 = 0; r0 < nclus; r0 += chunk) {
      const bool okm = mbar_wait(&mrg_bar, mphase);
      if (!okm && tid == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
      mphase ^= 1;
      const int n = min(chunk, nclus - r0);
#pragma unroll
      for (int it = 0; it < kItems; ++it) {
        const int item = tid + it * kCompute;
        if (item < a.G * TQ_D) {
          const int h = item >> 7, i = item & 127;
          const float* wv = s_w + h * kMaxSplits + r0;
          const float* av = sa + h * kRec + 4 + i;
          const int step = a.G * kRec;
          float x0 = 0.f, x1 = 0.f;
          int r = 0;
          for (; r + 2 <= n; r += 2) {
            x0 = fmaf(wv[r], av[r * step], x0);
            x1 = fmaf(wv[r + 1], av[(r + 1) * step], x1);
          }
          if (r < n) x0 = fmaf(wv[r], av[r * step], x0);
          x[it] += x0 + x1;
        }
      }
      if (r0 + chunk < nclus) {
        named_sync(kBarAll, kCompute);   // the chunk buffer is consumed
        if (tid == 0) {
          fence_async_smem();
          issue_chunk(r0 + chunk);
        }
      }
    }
  }
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int item = C > 1 ? (it == 0 && slice_item ? tid : -1) : tid + it * kCompute;
    if (item >= 0 && item < a.G * R) {
      const int h = item / R, i = item - h * R;
      const float Lh = s_hL[h];
      const float v = Lh > 0.f ? x[it] / Lh : 0.f;
      const long long e = ((long long)b * a.Hq + kvh * a.G + h) * TQ_D + i0 + i;
      if (a.out_dtype == TQ_F32) static_cast<float*>(a.out)[e] = v;
      else if (a.out_dtype == TQ_BF16) static_cast<__nv_bfloat16*>(a.out)[e] = __float2bfloat16_rn(v);
      else static_cast<__half*>(a.out)[e] = __float2half_rn(v);
    }
  }
  if (rank == 0 && tid == 0) a.counters[bh] = 0;   // ready for the next call
}

// Cluster size and split count: as many CTAs as can be co-resident (one per SM), in clusters
// of 4, 2 or 1 consecutive splits of one (batch, KV head).
template <int KB, int VB, bool HILO>
tq_status launch_one(const tq_mma_launch& a0, cudaStream_t stream) {
  constexpr int smem = TL<KB, VB, HILO>::total;
  auto kern = decode_tc_kernel<KB, VB, HILO>;
  static bool configured[64] = {};
  static int max_ctas[64][3] = {};   // co-resident CTAs with clusters of 1, 2, 4
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return TQ_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    max_ctas[dev][0] = per_sm * tq_num_sms();
    for (int k = 1; k < 3; ++k) {
      const int csz = 1 << k;
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(csz, 1, 1);
      q.blockDim = dim3(kThreads);
      q.dynamicSmemBytes = smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = csz;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      q.attrs = at;
      q.numAttrs = 1;
      int nclusters = 0;
      if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &q) != cudaSuccess) nclusters = 0;
      max_ctas[dev][k] = nclusters * csz;
    }
    cudaGetLastError();
    configured[dev] = true;
  }
  // the choice with the shortest estimated critical path: tiles per CTA plus the end of the
  // split, which costs about three tiles more without clusters and one and a half more with
  // clusters of two than with clusters of four (each CTA rotates back a smaller share); on a
  // tie the larger cluster
  const int units = a0.B * a0.Hkv;
  const long long len = a0.max_len > 0 ? a0.max_len : 1;
  int best_c = 1, best_n = 1;
  long long best_cost = -1;
  for (int k = 0; k < 3; ++k) {
    const int csz = 1 << k;
    int ns = max_ctas[dev][k] / units;
    if (ns > a0.nsplit) ns = a0.nsplit;
    ns -= ns % csz;
    if (ns < csz) {
      if (csz > 1) continue;
      ns = 1;
    }
    const long long tiles = ((len + ns - 1) / ns + kTile - 1) / kTile;
    const long long cost = 2 * tiles + (csz == 1 ? 6 : csz == 2 ? 3 : 0);
    if (best_cost < 0 || cost <= best_cost) {
      best_cost = cost;
      best_c = csz;
      best_n = ns;
    }
  }
  if (max_ctas[dev][0] / units < 2 && a0.nsplit > 1) {
    // fewer SMs than two splits per unit: the plan's splits, in several waves
    best_c = 1;
    best_n = a0.nsplit;
  }
  tq_mma_launch a = a0;
  long long sl = a.max_len > 0 ? (a.max_len + best_n - 1) / best_n : 1;
  sl = (sl + kTile - 1) / kTile * kTile;
  // splits rounded to whole tiles may cover the context with fewer of them: launch only those
  // (whole clusters), which leaves SMs to the query-operand kernel running alongside
  if (a.max_len > 0) {
    int used = (int)((a.max_len + sl - 1) / sl);
    used = (used + best_c - 1) / best_c * best_c;
    if (used < best_n) best_n = used;
  }
  a.nsplit = best_n;
  a.split_len = (int)sl;
  query_prep_tc_kernel<KB, HILO><<<dim3(4, a.Hkv, a.B), kPrepThreads, 0, stream>>>(a);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nsplit, a.Hkv, a.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = best_c;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = best_c > 1 ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return TQ_ERR_CUDA;
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
// smax·‖q‖); the operand holds twice them divided by b_r (|1/b_r| ≤ 2, see expand_inv_b), so
// each scale puts four times the bound in [224, 448), inside the e4m3 range.
void tq_tc_operand_scales(const tq_plane_decomp& kd, float* s_idx, float* s_sgn) {
  float m = 0.f;
  for (int v = 0; v < kd.n; ++v) m = fmaxf(m, 0.5f * fabsf(kd.coef[v]));
  int e = 0;
  frexpf(448.f / (m > 0.f ? m : 1.f), &e);   // 448/m = f·2^e, f in [0.5, 1)
  *s_idx = ldexpf(1.f, e - 3);
  *s_sgn = 64.f;
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
