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
// shared-memory ring with bulk copies (TMA engine).  The query operand comes from a small
// kernel that runs first (this grid's programmatic-launch primary) while the ring fills.
// At the end each split writes its record (m, l, acc[128] per head, still in the rotated
// domain) to the workspace and takes a ticket; the last split of a (batch, KV head) copies the
// records and Π into shared memory, adds up the records with log-sum-exp weights and rotates
// the sum back once (out = Πᵀ·acc / L).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "decode_args.h"
#include "tc_ptx.h"
#include "tile_mma.h"

TQ_DEFINE_FLAGS(tq_take_flags_decode_tc)

#include "append_small.h"

namespace {
using namespace tq;

constexpr int kTile = 128;                    // tokens per tile = TMEM lanes
constexpr int kStageTok = 256;                // tokens per ring stage (two tiles)
constexpr int kStages = 4;
constexpr int kEWarps = 4;                    // expand planes into TMEM
// Warp roles of a split CTA with NG softmax groups: 4 expander warps, NG groups of four
// softmax + value warps (group g takes the tiles i ≡ g mod NG), one MMA-issue warp, and the
// producer warp last.
template <int NG>
struct Roles {
  static constexpr int S = 4 * NG;                           // softmax + value warps
  static constexpr int issuer = kEWarps + S;                 // the MMA-issue warp
  static constexpr int compute = (kEWarps + S + 1) * 32;    // every warp but the producer
  static constexpr int threads = compute + 32;
};
constexpr int kPieces = 4;                    // e4m3 pieces per query value
// MMA N: 4 pieces × 8 head columns, or (group of at most 4 heads) 4 pieces × 4 heads
__host__ __device__ constexpr int kNof(bool hilo) { return hilo ? 16 : kPieces * 8; }
// one plane's query operand (4 KB or 2 KB of e4m3)
__host__ __device__ constexpr int kBImgOf(bool hilo) { return kNof(hilo) * 128; }
constexpr int kBSbo = 8 * 128;                // 8-row groups of the operand image
// score constants: 8 columns × {A, Cm, B, Cq}, then the operand offsets
// ([16 slices][index planes | sign plane][8 columns], see query_prep_tc_kernel)
constexpr int kCstFloats = 8 * 4;
constexpr int kCstBytes = (kCstFloats + 16 * 2 * 8) * 4;
constexpr int kRec = TQ_REC;
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


// ---------------------------------------------------------------- query operand kernel
// Grid (kSlices / SPC, KV heads, batch), the split kernel's programmatic-launch primary.  The
// work for slice s (SPC slices a CTA) computes (Π q_h)_j and (S q_h)_j for the group's heads h
// and the 8 coordinates j = 8s..8s+7, and writes the operand bytes of their K positions k
// (coord_of_k(k) = j) in every plane: row (piece p, column n) holds piece p of
// coef_v·(Π q)_j/‖q‖·s_idx (index plane v) or 2·(S q)_j/(‖q‖·smax)·s_sgn (sign plane), divided
// by the b_r of the K position's expanded A byte; column n = head n.  It also writes the
// slice's share of the operand offsets Σ a_r·(operand) (the constant the MMAs add to each
// column) and, slice 0, the score constants.  ‖q‖ and the column sums (Πᵀ1)·q, (Sᵀ1)·q come
// straight from q, so no slice needs another slice's results.
constexpr int kSlices = 16;
constexpr int kPrepThreads = 256;
// SPC slices per CTA (grid kSlices / SPC × KV heads × batch): one slice a CTA while the grid
// stays small; large batches take 2 or 4, so that the operand kernel runs in one short wave
// and frees the SMs for the split grid.
// The operand work of CTA `bx` for slices SPC·bx .. SPC·bx + SPC − 1, by the first kPrepThreads
// threads of the CTA; any further threads only take part in the CTA barriers.
template <int KB, bool HILO, int SPC>
__device__ __forceinline__ void query_prep_role(const tq_mma_launch& a, int bx) {
  constexpr int NKV = num_vplanes(KB);
  constexpr int NP = NKV + 1;
  constexpr int kBImg = kBImgOf(HILO);
  constexpr int kN = kNof(HILO);
  constexpr int NCOL = HILO ? 4 : 8;
  // SPC = 4: the CTA holds K positions 32·bx .. +31 of every operand row whole, so
  // they are gathered here and leave as 16-byte stores
  __shared__ __align__(16) unsigned char stage[SPC == 4 ? NP * kN * 32 : 16];
  __shared__ __align__(16) float qf[8][TQ_D];
  // [slice][Π|S][head][k chunk · 8 + j in slice], rows padded to 136 floats: a warp's stores
  // (8 j × 4 k chunks) and the sums' reads (8 j × 4 heads) fall in 32 distinct banks
  constexpr int kRedPitch = 16 * 8 + 8;
  __shared__ __align__(16) float red[SPC][2][8][kRedPitch];
  __shared__ float prod[SPC][2][8][8];      // [slice][Π|S][j in slice][head]
  __shared__ float s_nq[8], s_inq[8], s_uq[8], s_wq[8];
  __shared__ float s_off[SPC][2][8];        // [slice][index planes | sign plane][column]
  const int kvh = blockIdx.y, b = blockIdx.z;
  const long long bh = (long long)b * a.Hkv + kvh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool act = tid < kPrepThreads;
  // thread (which, k chunk kq, jl): 8 entries of rows j of M (M = Π or S, read from Mᵀ: the
  // codec's constants), requested at once.  SPC < 4: row j = 8(SPC·bx + u) + jl of each slice u
  // (t[u]).  SPC = 4: the CTA's 32 rows are consecutive and the thread takes rows
  // 32bx + 4jl + e (t[e]: slice jl / 2, j in slice 4(jl mod 2) + e) by 16-byte loads.
  const int which = (tid >> 7) & 1, kq = (tid >> 3) & 15, jl = tid & 7;
  const float* T = which ? a.sT : a.piT;
  float t[SPC][8];
  if constexpr (SPC == 4) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(&T[(8 * kq + k) * TQ_D + 32 * bx + 4 * jl]));
      t[0][k] = v.x; t[1][k] = v.y; t[2][k] = v.z; t[3][k] = v.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < SPC; ++u) {
      const int j = 8 * (SPC * bx + u) + jl;
#pragma unroll
      for (int k = 0; k < 8; ++k) t[u][k] = __ldg(&T[(8 * kq + k) * TQ_D + j]);
    }
  }
  // the column sums Πᵀ1 and Sᵀ1 at the lane's coordinates (for the norm warps)
  float cu[4], cw[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    cu[k] = __ldg(&a.u[lane + 32 * k]);
    cw[k] = __ldg(&a.w[lane + 32 * k]);
  }
  // This grid is a programmatic-launch secondary of the previous kernel in the stream: the
  // queries (and the cache that the split grid streams before it waits for this grid) may be
  // that kernel's output, so the split grid may start only once every CTA is past this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The split tickets of this (batch, KV head) start the call at zero whatever the workspace
  // held before (another descriptor's records, an asymmetric call, a call that gave up on a
  // wait): the split grid takes tickets only after this grid has completed.
  if (bx == 0 && tid == 0) a.counters[bh] = 0;
  for (int i = tid; act && i < 8 * TQ_D; i += kPrepThreads) {
    const int h = i >> 7, jq = i & 127;
    float v = 0.f;
    if (h < a.G) {
      const long long e = ((long long)b * a.Hq + kvh * a.G + h) * TQ_D + jq;
      if (a.q_dtype == TQ_F32) v = __ldg(static_cast<const float*>(a.q) + e);
      else if (a.q_dtype == TQ_BF16)
        v = __uint_as_float((uint32_t)__ldg(static_cast<const unsigned short*>(a.q) + e) << 16);
      else v = __half2float(__ushort_as_half(__ldg(static_cast<const unsigned short*>(a.q) + e)));
    }
    qf[h][jq] = v;
  }
  if (tid < 8) s_inq[tid] = 0.f;
  __syncthreads();
  if (warp < a.G) {
    // ‖q‖, (Πᵀ1)·q and (Sᵀ1)·q of head `warp`
    float n2 = 0.f, uq = 0.f, wq = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int jq = lane + 32 * k;
      const float x = qf[warp][jq];
      n2 = fmaf(x, x, n2);
      uq = fmaf(cu[k], x, uq);
      wq = fmaf(cw[k], x, wq);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n2 += __shfl_xor_sync(0xffffffffu, n2, o);
      uq += __shfl_xor_sync(0xffffffffu, uq, o);
      wq += __shfl_xor_sync(0xffffffffu, wq, o);
    }
    if (lane == 0) {
      const float nq = sqrtf(n2);
      s_nq[warp] = nq;
      s_inq[warp] = nq > 0.f ? 1.f / nq : 0.f;
      s_uq[warp] = uq;
      s_wq[warp] = wq;
    }
  }
#pragma unroll
  // head h's 8 query values of the lane's k chunk are read once for all SPC slices; heads past
  // the group have q = 0, so their sums are exactly 0 without the products
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    float x[SPC];
#pragma unroll
    for (int u = 0; u < SPC; ++u) x[u] = 0.f;
    if (h < NCOL && h < a.G && act) {
      const float4 qa = *reinterpret_cast<const float4*>(&qf[h][8 * kq]);
      const float4 qb = *reinterpret_cast<const float4*>(&qf[h][8 * kq + 4]);
      const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
      for (int u = 0; u < SPC; ++u)
#pragma unroll
        for (int k = 0; k < 8; ++k) x[u] = fmaf(t[u][k], qv[k], x[u]);
    }
    if (act) {
      if constexpr (SPC == 4) {
        *reinterpret_cast<float4*>(&red[jl >> 1][which][h][kq * 8 + 4 * (jl & 1)]) =
            make_float4(x[0], x[1], x[2], x[3]);
      } else {
#pragma unroll
        for (int u = 0; u < SPC; ++u) red[u][which][h][kq * 8 + jl] = x[u];
      }
    }
  }
  __syncthreads();
  for (int it = tid; act && it < SPC * 2 * 8 * 8; it += kPrepThreads) {
    const int u = it >> 7, wh = (it >> 6) & 1, h = (it >> 3) & 7, jj = it & 7;
    float x = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) x += red[u][wh][h][k * 8 + jj];
    prod[u][wh][jj][h] = x;
  }
  __syncthreads();
  unsigned char* out = static_cast<unsigned char*>(a.qfrag) + bh * (long long)frag_block(NP, HILO);
  float* cst = reinterpret_cast<float*>(out + NP * kBImg);
  // item (slice u, column n, j in slice jj), every plane: the four piece bytes of K position k;
  // the 8 items of a (slice, column) are adjacent lanes and add up its offsets by shuffles
  // (item counts are multiples of 32: whole warps take part)
  const float sgn_scale = a.s_sgn / a.smax;
  for (int it = tid; act && it < SPC * NCOL * 8; it += kPrepThreads) {
    const int u = it / (NCOL * 8), n = (it >> 3) % NCOL, jj = it & 7;
    const int s = SPC * bx + u;
    const int k = 32 * (s >> 2) + 4 * jj + (s & 3);   // coord_of_k(k) = 8s + jj
    const int r = jj;                                  // (k >> 2) & 7
    const float inq = s_inq[n];                        // 1/‖q‖; 0 for a zero or absent head
    const float xi = 0.5f * a.s_idx * inq * prod[u][0][jj][n];
    const float xs = sgn_scale * inq * prod[u][1][jj][n];
    const float ib2 = 2.f * expand_inv_b(r), ar = expand_a(r);
    float oi = 0.f, os = 0.f;
#pragma unroll
    for (int v = 0; v < NP; ++v) {
      float y = ib2 * (v < NKV ? a.kd.coef[v] * xi : xs), yhat = 0.f;
      uint32_t e4 = 0u;
#pragma unroll
      for (int pc = 0; pc < kPieces; ++pc) {
        const __nv_fp8_storage_t e = __nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
        const float pv = e4m3_value(e);
        y -= pv;
        yhat += pv;
        e4 |= (uint32_t)e << (8 * pc);
      }
#pragma unroll
      for (int pc = 0; pc < kPieces; ++pc) {
        const unsigned char byte = (unsigned char)(e4 >> (8 * pc));
        if constexpr (SPC == 4) stage[(v * kN + bimg_row(HILO, pc, n)) * 32 + 4 * jj + u] = byte;
        else out[v * kBImg + bimg_off(bimg_row(HILO, pc, n), k)] = byte;
      }
      if (v < NKV) oi = fmaf(ar, yhat, oi);
      else os = fmaf(ar, yhat, os);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      oi += __shfl_xor_sync(0xffffffffu, oi, o);
      os += __shfl_xor_sync(0xffffffffu, os, o);
    }
    if (jj == 0) {
      s_off[u][0][n] = oi;
      s_off[u][1][n] = os;
    }
  }
  __syncthreads();
  if constexpr (SPC == 4) {
    for (int c = tid; act && c < NP * kN * 2; c += kPrepThreads) {
      const int v = c / (kN * 2), row = (c >> 1) % kN, hf = c & 1;
      *reinterpret_cast<uint4*>(out + v * kBImg + bimg_off(row, 32 * bx + 16 * hf)) =
          *reinterpret_cast<const uint4*>(stage + (v * kN + row) * 32 + 16 * hf);
    }
  }
  if (tid < SPC * 2 * NCOL) {
    // the slices' operand offsets: [slice][index planes | sign plane][column]
    const int u = tid / (2 * NCOL), kind = (tid / NCOL) & 1, n = tid % NCOL;
    const int s = SPC * bx + u;
    float* offp = cst + kCstFloats + s * 16 + kind * 8;
    if (HILO) {
      offp[2 * n] = s_off[u][kind][n];
      offp[2 * n + 1] = s_off[u][kind][n];
    } else {
      offp[n] = s_off[u][kind][n];
    }
  }
  if (bx == 0 && tid < 8) {
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

template <int KB, bool HILO, int SPC>
__global__ void __launch_bounds__(kPrepThreads, SPC == 4 ? 4 : 1)
    query_prep_tc_kernel(const tq_mma_launch a) {
  query_prep_role<KB, HILO, SPC>(a, blockIdx.x);
}

// Prologue of a decode step, the split kernel's programmatic-launch primary in place of the
// operand kernel.  Grid (kSlices / SPC + appends, KV heads, batch): the first kSlices / SPC CTAs
// of a (batch, KV head) build its query operand; the rest quantise the step's new key (product
// code) and value (MSE code) into the caches at position seq_lens[b]: one CTA for both when
// the two codecs share Π, else one CTA each.  One launch does the work of the appends and the
// operand kernel, which would otherwise run one after the other.
template <int KB, bool HILO, int SPC>
__global__ void __launch_bounds__(kAppendThreads, 1) step_prologue_kernel(const tq_mma_launch a) {
  constexpr int nsl = kSlices / SPC;
  if ((int)blockIdx.x < nsl) query_prep_role<KB, HILO, SPC>(a, blockIdx.x);
  else if (a.app.shared_pi) append_kv_pair_role(a.app, blockIdx.y, blockIdx.z);
  else append_kv_role(a.app, (int)blockIdx.x == nsl, blockIdx.y, blockIdx.z);
}

// Tokens that query row b attends: its sequence's length (+ len_add for a decode step), plus,
// for row i of a causal prefill chunk, the chunk's own first i + 1 tokens.
__device__ __forceinline__ int row_len(const tq_mma_launch& a, int b) {
  const int s = b / a.qps;
  return a.seq_lens[s] + a.len_add + (a.causal ? b - s * a.qps + 1 : 0);
}

// A sequence of len tokens is cut into ceil(len / split_len) splits of equal size in whole tiles
// (at most split_len, a multiple of the tile): every one of them holds tokens, and a ragged
// batch's splits are as even as its lengths allow.
__device__ __forceinline__ int seq_split_len(int len, int split_len) {
  const int ns = len > 0 ? (len + split_len - 1) / split_len : 1;
  return ((len + ns - 1) / ns + kTile - 1) / kTile * kTile;
}

// ---------------------------------------------------------------- shared memory and TMEM
template <int KB, int VB, bool HILO, int NG>
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
  // after the main loop everything is reused: first the softmax warps' accumulators and
  // statistics; then, in the split that merges, the merged accumulators [128][8], merge
  // weights and sums [2][8][kMaxSplits], the merge's partial sums [at most 15][128], Π (64 KB)
  // and the records, copied in chunks of whole splits into [rec_off, total) (then the rotation's
  // 15 partial sums [15][8][128]); the dynamic shared memory is sized so that one chunk holds
  // the records of every split at the usual split counts
  static constexpr int comb_acc = 0;
  static constexpr int comb_stats = Roles<NG>::S * 8 * kAccPitch * 4;
  static constexpr int mrg_acc = 0;
  static constexpr int mrg_w = 8 * TQ_D * 4;
  static constexpr int mrg_part = mrg_w + 2 * 8 * kMaxSplits * 4;
  static constexpr int pi_off = mrg_part + (Roles<NG>::compute / 32) * (TQ_D + 4) * 4;
  static constexpr int rec_off = pi_off + TQ_D * TQ_D * 4;
  static constexpr int total = 226 * 1024;
  static_assert(used <= total && rec_off + 16 * 8 * TQ_REC * 4 <= total, "shared memory");
  static_assert(rec_off + (Roles<NG>::compute / 32) * 8 * TQ_D * 4 <= total,
                "rotation partial sums");
  // TMEM: A (one tile: NP planes × 32 columns of e4m3), D (NP planes × 32 columns)
  static constexpr int a_cols = NP * 32;
  // D: index planes summed in pairs by the MMAs (block j = planes 2j, 2j + 1), then the sign
  // plane's block
  static constexpr int d_blocks = (NP - 1 + 1) / 2 + 1;
  static constexpr int d_cols = d_blocks * kN;
  // one D buffer per softmax group
  static constexpr int abufs = (2 * a_cols + NG * d_cols <= 512) ? 2 : 1;
  static constexpr int d_col = abufs * a_cols;
  static_assert(d_col + NG * d_cols <= 512, "TMEM columns");
};

// ---------------------------------------------------------------- paged stage copies
// One ring stage of a page pool's cache (include/tq.h, tq_pages): tokens [t0, t1) of sequence
// `seq`, KV head kvh, as runs within one page each, up to the end of the page of the row's last
// attended token (len; pages past it are not read).  A run whose table entry lies outside the
// pool is left out and raises TQ_FLAG_PAGE (its rows keep stale data).  A cache without a
// table (the other of the pair may have one) is read as one run of row ch.  Run bounds are
// multiples of 64 tokens, so every copy is 16-byte aligned.  Called by the producer's lane.
template <int KB, int VB>
__device__ __noinline__ void paged_stage(const tq_mma_launch& a, int o_kplanes, int o_ksgn,
                                         int o_kxn, int o_krn, int o_vcodes, int o_vxn,
                                         unsigned char* base, uint64_t* bar, long long ch, int seq,
                                         int kvh, int len, int t0, int t1) {
  constexpr unsigned kTokK = KB * 16 + 16 + 4 + 4;              // key bytes per token
  constexpr unsigned kTokV = (VB == 4 ? 64 : VB * 16) + 4;      // value bytes per token
  // n tokens from slot `slot` of cache row `row` (rc slots a row) to stage token `off`
  auto copy_k = [&](long long row, int rc, int slot, int n, int off) {
    for (int p = 0; p < KB; ++p)
      bulk_g2s(base + o_kplanes + (p * kStageTok + off) * 16,
               a.kidx + ((row * KB + p) * rc + slot) * 16, n * 16, bar);
    bulk_g2s(base + o_ksgn + off * 16, a.ksgn + (row * rc + slot) * 16, n * 16, bar);
    bulk_g2s(base + o_kxn + off * 4, a.kxn + row * rc + slot, n * 4, bar);
    bulk_g2s(base + o_krn + off * 4, a.krn + row * rc + slot, n * 4, bar);
  };
  auto copy_v = [&](long long row, int rc, int slot, int n, int off) {
    if (VB == 4) {
      bulk_g2s(base + o_vcodes + off * 64, a.vidx + (row * rc + slot) * 64, n * 64, bar);
    } else {
      for (int p = 0; p < VB; ++p)
        bulk_g2s(base + o_vcodes + (p * kStageTok + off) * 16,
                 a.vidx + ((row * VB + p) * rc + slot) * 16, n * 16, bar);
    }
    bulk_g2s(base + o_vxn + off * 4, a.vxn + row * rc + slot, n * 4, bar);
  };
  // f(row, slot, n, offset from t0) for each run of map m; bytes only (copy = false) or copies
  auto runs = [&](const tq_rowmap& m, bool copy, auto&& f) {
    if (!m.table) {
      f(ch, a.cap, t0, t1 - t0, 0);
      return;
    }
    const int P = m.page_tokens;
    const int te_all = min(t1, ((len - 1) / P + 1) * P);
    for (int t = t0; t < te_all;) {
      const int q = t / P, te = min(te_all, (q + 1) * P);
      const int pg = __ldg(m.table + (long long)seq * m.max_pages + q);
      if (pg >= 0 && pg < m.num_pages) f((long long)pg * a.Hkv + kvh, P, t - q * P, te - t, t - t0);
      else if (copy) atomicOr(&g_tq_flags, TQ_FLAG_PAGE);
      t = te;
    }
  };
  // the bytes of every run first: the barrier expects them before the copies land
  unsigned bytes = 0;
  runs(a.kmap, false, [&](long long, int, int, int n, int) { bytes += (unsigned)n * kTokK; });
  runs(a.vmap, false, [&](long long, int, int, int n, int) { bytes += (unsigned)n * kTokV; });
  mbar_expect_tx(bar, bytes);
  runs(a.kmap, true, copy_k);
  runs(a.vmap, true, copy_v);
}

// ---------------------------------------------------------------- the split kernel
template <int KB, int VB, bool HILO, int NG, bool kPaged>
__global__ void __launch_bounds__(Roles<NG>::threads, 1) decode_tc_kernel(const tq_mma_launch a) {
  using L = TL<KB, VB, HILO, NG>;
  using R = Roles<NG>;
  constexpr int kThreads = R::threads;
  constexpr int kCompute = R::compute;
  constexpr int kSWarps = R::S;
  constexpr int kN = L::kN;
  constexpr int kBImg = kBImgOf(HILO);
  constexpr int NKV = num_vplanes(KB);
  constexpr int NP = NKV + 1;
  constexpr int NVV = VB == 4 ? 0 : num_vplanes(VB);
  constexpr int NB = L::d_blocks;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t mma_done[NG];   // key scores of group g's tile in D[g]
  __shared__ __align__(8) uint64_t d_free[NG];
  __shared__ __align__(8) uint64_t a_full[2];
  __shared__ __align__(8) uint64_t op_bar;     // query operand and constants landed
  __shared__ __align__(8) uint64_t prol_bar;   // value pair table landed (4-bit values)
  __shared__ __align__(8) uint64_t pi_bar;     // Π landed (rotation back)
  __shared__ __align__(8) uint64_t rec_bar;    // a chunk of records landed (last split)
  __shared__ float s_hL[8];
  __shared__ uint32_t s_tmem;
  __shared__ int s_ticket;
  __shared__ int s_item;

  // the warp index through a shuffle: the compiler then knows it is warp-uniform and keeps
  // the TMEM addresses derived from it in uniform registers
  const int tid = threadIdx.x, warp = __shfl_sync(0xffffffffu, tid >> 5, 0), lane = tid & 31;
  // CTAs are dispatched in blockIdx order.  For a batch, the work items (sequence, split) are
  // taken largest first (ties by index), the KV heads of an item side by side: the long splits
  // start in the first wave and the short ones fill in behind them (longest-processing-time-
  // first list scheduling).  The ranking uses the dynamic shared memory, not yet in use.
  int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int nitems = a.B * (int)gridDim.x;
  if (a.B > 1 && nitems <= kThreads) {
    int* sc_len = reinterpret_cast<int*>(smem);
    int* sc_work = sc_len + kThreads;
    if (tid < a.B) sc_len[tid] = min(row_len(a, tid), a.cap);
    __syncthreads();
    if (tid < nitems) {
      const int ib = tid / (int)gridDim.x, is = tid - ib * (int)gridDim.x;
      const int lb = sc_len[ib], slb = seq_split_len(lb, a.split_len);
      sc_work[tid] = max(0, min(slb, lb - is * slb));
    }
    __syncthreads();
    const int pos = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    if (tid < nitems) {
      const int wt = sc_work[tid];
      int rank = 0;
      for (int o = 0; o < nitems; ++o) {
        const int wo = sc_work[o];
        rank += (wo > wt || (wo == wt && o < tid)) ? 1 : 0;
      }
      if (rank == pos / a.Hkv) s_item = tid;
    }
    fence_async_smem();   // the scratch is the ring: bulk copies write it next
    __syncthreads();
    b = s_item / (int)gridDim.x;
    split = s_item - b * (int)gridDim.x;
    kvh = pos % a.Hkv;
  }
  int len = row_len(a, b);   // in flight during the setup
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full_bar[st], 1);
      mbar_init(&empty_bar[st], 2 * (kEWarps + 4));   // two tiles per stage
    }
    for (int i = 0; i < NG; ++i) {
      mbar_init(&mma_done[i], 1);
      mbar_init(&d_free[i], 4);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&a_full[i], kEWarps);
    mbar_init(&op_bar, 1);
    mbar_init(&prol_bar, 1);
    mbar_init(&pi_bar, 1);
    mbar_init(&rec_bar, 1);
    mbar_init_fence();
    s_ticket = 0;
  }
  if (warp == 0) tmem_alloc(&s_tmem, 512);
  tc_before();
  __syncthreads();
  tc_after();
  const long long bh = (long long)b * a.Hkv + kvh;   // query row: operand, records, tickets
  const long long ch = (long long)(b / a.qps) * a.Hkv + kvh;   // the cache row it attends
  if (len > a.cap) {
    if (tid == 0 && split == 0 && kvh == 0) atomicOr(&g_tq_flags, TQ_FLAG_LEN_OVERFLOW);
    len = a.cap;
  }
  const int slb = seq_split_len(len, a.split_len);
  const int t_begin = split * slb;
  const int t_end = min(t_begin + slb, len);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;
  const int nstages = (ntiles + 1) / 2;
  // Only the splits that hold tokens take part (ragged batches launch many empty ones): an
  // empty split leaves right after the setup, and a sequence without tokens gets its zero
  // output from split 0.
  const int used = (len + a.split_len - 1) / a.split_len;   // the splits with tokens
  if (ntiles == 0) {
    if (len == 0 && split == 0)
      for (int i = tid; i < a.G * TQ_D; i += kThreads) {
        const long long e = ((long long)b * a.Hq + kvh * a.G) * TQ_D + i;
        if (a.out_dtype == TQ_F32) static_cast<float*>(a.out)[e] = 0.f;
        else if (a.out_dtype == TQ_BF16) static_cast<__nv_bfloat16*>(a.out)[e] = __float2bfloat16_rn(0.f);
        else static_cast<__half*>(a.out)[e] = __float2half_rn(0.f);
      }
    if (warp == 0) tmem_dealloc(s_tmem, 512);
    return;
  }

  const uint32_t tmem = s_tmem;

  // ============================================================ producer warp
  if (warp == R::issuer + 1) {
    if (lane == 0) {
      // the stage's tokens [t0, t0 + 256) (not past the capacity); the flat layout's rows are
      // contiguous, a page pool's are runs within pages (kPaged)
      auto issue = [&](int c) {
        const int st = c % kStages;
        const int t0 = t_begin + c * kStageTok;
        if constexpr (!kPaged) {
          const int n = min(kStageTok, a.cap - t0);   // a multiple of 64 (the capacity is)
          unsigned char* base = smem + st * L::stage;
          const unsigned bytes =
              (unsigned)n * (KB * 16 + 16 + 4 + 4 + (VB == 4 ? 64 : VB * 16) + 4);
          mbar_expect_tx(&full_bar[st], bytes);
          for (int p = 0; p < KB; ++p)
            bulk_g2s(base + L::kplanes + p * kStageTok * 16,
                     a.kidx + ((ch * KB + p) * a.cap + t0) * 16, n * 16, &full_bar[st]);
          bulk_g2s(base + L::ksgn, a.ksgn + (ch * a.cap + t0) * 16, n * 16, &full_bar[st]);
          bulk_g2s(base + L::kxn, a.kxn + ch * a.cap + t0, n * 4, &full_bar[st]);
          bulk_g2s(base + L::krn, a.krn + ch * a.cap + t0, n * 4, &full_bar[st]);
          if (VB == 4) {
            bulk_g2s(base + L::vcodes, a.vidx + (ch * a.cap + t0) * 64, n * 64, &full_bar[st]);
          } else {
            for (int p = 0; p < VB; ++p)
              bulk_g2s(base + L::vcodes + p * kStageTok * 16,
                       a.vidx + ((ch * VB + p) * a.cap + t0) * 16, n * 16, &full_bar[st]);
          }
          bulk_g2s(base + L::vxn, a.vxn + ch * a.cap + t0, n * 4, &full_bar[st]);
        } else {
          paged_stage<KB, VB>(a, L::kplanes, L::ksgn, L::kxn, L::krn, L::vcodes, L::vxn,
                              smem + st * L::stage, &full_bar[st], ch, b / a.qps, kvh, len, t0,
                              min(t0 + kStageTok, a.cap));
        }
      };
      // Π is read again only by the split that merges: have it in L2 by then
      if (split == 0) bulk_prefetch_l2(a.pi, TQ_D * TQ_D * 4);
      // The ring's first stages and the value pair table come in while this grid's programmatic-
      // launch primary (the operand kernel, or a decode step's prologue) runs: the cache is final
      // by then, except for the last `fresh` tokens that a step's prologue appends, whose stages
      // are requested after the wait.  The operand is copied in as soon as the primary grid has
      // completed, ahead of the remaining stages.
      int c = 0;
      for (; c < nstages && c < kStages; ++c) {
        const int t0 = t_begin + c * kStageTok;
        if (a.fresh > 0 && t0 + min(kStageTok, a.cap - t0) > len - a.fresh) break;
        issue(c);
      }
      if (VB == 4) {
        mbar_expect_tx(&prol_bar, L::lut_bytes);
        bulk_g2s(smem + L::lut, a.lut, L::lut_bytes, &prol_bar);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      mbar_expect_tx(&op_bar, frag_block(NP, HILO));
      bulk_g2s(smem + L::frag,
               static_cast<const unsigned char*>(a.qfrag) + bh * (long long)frag_block(NP, HILO),
               frag_block(NP, HILO), &op_bar);
      for (; c < nstages && c < kStages; ++c) issue(c);
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
      if (VB == 4) mbar_wait(&prol_bar, 0);
      mbar_wait(&op_bar, 0);
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
      if (okl && prev >= 0) okl = mbar_wait(&mma_done[prev % NG], (prev / NG) & 1);
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
  } else if (warp == R::issuer) {
    // ========================================================== MMA-issue warp
    // D block j accumulates index planes 2j and 2j + 1, the last block the sign plane; 4 MMAs
    // of K = 32 per plane and tile, into group g's D buffer for the tiles i ≡ g (mod NG).  The
    // whole warp waits and forms the (warp-uniform) descriptors; one elected lane issues the
    // MMAs and their commit.
    if (warp == R::issuer && ntiles > 0) {
      const uint32_t idesc = idesc_f16(128, kN);   // e4m3 × e4m3 → f32 has the same fields
      const uint32_t frag_s = s32(smem + L::frag);
      bool ok = mbar_wait(&op_bar, 0);
      for (int i = 0; i < ntiles && ok; ++i) {
        const int ab = L::abufs == 2 ? (i & 1) : 0;
        const int g = i % NG;
        ok = mbar_wait(&a_full[ab], (i / L::abufs) & 1) &&
             (i < NG || mbar_wait(&d_free[g], ((i / NG) - 1) & 1));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_after();
        if (elect_one()) {
#pragma unroll
          for (int j = 0; j < NB; ++j) {
            const uint32_t d = tmem + L::d_col + g * L::d_cols + j * kN;
            const int v0 = j == NB - 1 ? NKV : 2 * j;
            const int nv = j == NB - 1 ? 1 : (2 * j + 1 < NKV ? 2 : 1);
#pragma unroll
            for (int o = 0; o < 2; ++o) {
              if (o < nv) {
                const uint32_t a0 = tmem + ab * L::a_cols + 32 * (v0 + o);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                  mma_f8(d, a0 + 8 * ks,
                         smem_desc(frag_s + (v0 + o) * kBImg + ks * 256, 128, kBSbo), idesc,
                         (o > 0 || ks > 0) ? 1u : 0u);
              }
            }
          }
          mma_commit(&mma_done[g]);
        }
        __syncwarp();
      }
      if (!ok && lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ========================================================== softmax / value warps
    const int sw_ = warp - kEWarps;                       // 0 .. 4·NG − 1
    const int stid = tid - kEWarps * 32;
    const int q = warp & 3;                               // TMEM lane quadrant
    const int grp = sw_ >> 2;                             // tiles i ≡ grp (mod NG)
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const int g = lane >> 2, c = lane & 3;
    // the query operand and its constants (and the value pair table) have landed
    bool okp = mbar_wait(&op_bar, 0) && (VB != 4 || mbar_wait(&prol_bar, 0));
    if (!okp) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    float hA[2], hCm[2], hB[2], hCq[2];
    {
      const float* cst = reinterpret_cast<const float*>(smem + L::frag + NP * kBImg);
      const float* offp = cst + kCstFloats;   // [slice][index planes | sign plane][column]
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int col = 2 * c + k;
        float oi = 0.f, os = 0.f;
#pragma unroll
        for (int sl = 0; sl < kSlices; ++sl) {
          oi += offp[sl * 16 + col];
          os += offp[sl * 16 + 8 + col];
        }
        hA[k] = cst[col * 4 + 0];
        hCm[k] = cst[col * 4 + 1] + oi;
        hB[k] = cst[col * 4 + 2];
        hCq[k] = cst[col * 4 + 3] + os;
      }
    }
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f}, lw_run[2] = {0.f, 0.f};
    const uint32_t* lut_lane = reinterpret_cast<const uint32_t*>(smem + L::lut) + lane;

    for (int i = grp; i < ntiles && okp; i += NG) {
      const int st = (i >> 1) % kStages;
      const int hrow = (i & 1) * kTile;                   // the tile's first row in the stage
      const int db = grp;
      const bool okw = mbar_wait(&mma_done[db], (i / NG) & 1) &&
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
    // ---- this split's record, in the rotated domain: (M, L, acc[128]) per head; item (head,
    // 4 coordinates), one 16-byte store
    float* rec = a.part + ((bh * a.nsplit + split) * a.G) * kRec;
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
      *reinterpret_cast<float4*>(rec + head * kRec + 4 + j0) = make_float4(v4[0], v4[1], v4[2], v4[3]);
      if (j0 == 0) {
        rec[head * kRec + 0] = cML[col];                       // base-2 maximum
        rec[head * kRec + 1] = cML[8 + col];
      }
    }
  }

  // ============================================================ end of the split
  // The main loop is over: the next kernel in the stream may launch now and fetch its
  // constants while the records are merged (it waits for this grid to complete before it
  // touches anything this grid reads or writes).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the records are released at device scope; the split that takes the last ticket of its
  // (batch, KV head) merges them
  tc_before();
  named_sync(kBarAll, kCompute);
  tc_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
  if (tid == 0) {
    // acquire-release: releases the CTA's records (ordered before by the barrier) and, for
    // the last split, acquires every other split's
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(a.counters + bh) : "memory");
    s_ticket = old == used - 1 ? 1 : 0;
  }
  named_sync(kBarAll, kCompute);
  if (s_ticket != 1) return;
  // out_h = Πᵀ·(Σ_r w_r·acc_r) / Σ_r w_r·L_r with w_r = 2^(M_r − max M).  The records come
  // into shared memory by bulk copies, in chunks of whole splits; warp h computes the weights
  // of head h from the records' (M, L) meanwhile.
  const float* recs = a.part + bh * (long long)a.nsplit * a.G * kRec;
  float* mrg = reinterpret_cast<float*>(smem + L::mrg_acc);     // [128][8]
  float* s_w = reinterpret_cast<float*>(smem + L::mrg_w);       // [2][8][kMaxSplits]
  // [parts·G][kPartPitch]: the pitch of 132 floats keeps the coordinate-major reads below free
  // of bank conflicts
  constexpr int kPartPitch = TQ_D + 4;
  static_assert((kCompute / 32) * kPartPitch * 4 <= L::pi_off - L::mrg_part, "merge partials");
  float* rpart = reinterpret_cast<float*>(smem + L::mrg_part);
  float* srec = reinterpret_cast<float*>(smem + L::rec_off);    // [chunk][G][kRec]
  const int rec_bytes = a.G * kRec * 4;
  const int chunk = (L::total - L::rec_off) / rec_bytes;
  // a chunk comes in as up to 8 bulk copies of whole records, all in flight at once
  auto issue_chunk = [&](int r0) {
    const int n = min(chunk, used - r0);
    mbar_expect_tx(&rec_bar, (unsigned)(n * rec_bytes));
    const int per = (n + 7) / 8;
    for (int q0 = 0; q0 < n; q0 += per) {
      const int m = min(per, n - q0);
      bulk_g2s(srec + (long long)q0 * a.G * kRec, recs + (long long)(r0 + q0) * a.G * kRec,
               (unsigned)(m * rec_bytes), &rec_bar);
    }
  };
  // the copies are issued by a thread of the last compute warp, which has no weights to compute
  const bool issuer = tid == kCompute - 32;
  if (issuer) {
    asm volatile("fence.proxy.async.global;" ::: "memory");   // records → bulk copies
    // the first chunk of records, then Π for the rotation back (its region is free: the
    // ring's data is consumed and the operand images are read)
    fence_async_smem();
    issue_chunk(0);
    mbar_expect_tx(&pi_bar, TQ_D * TQ_D * 4);
    bulk_g2s(smem + L::pi_off, a.pi, TQ_D * TQ_D * 4, &pi_bar);
  }
  if (warp < a.G) {
    // every (M, L) of the head requested at once
    float mv[kMaxSplits / 32], lv[kMaxSplits / 32];
#pragma unroll
    for (int u = 0; u < kMaxSplits / 32; ++u) {
      const int r = lane + 32 * u;
      const long long o = ((long long)r * a.G + warp) * kRec;
      mv[u] = r < used ? __ldcg(&recs[o]) : 0.f;
      lv[u] = r < used ? __ldcg(&recs[o + 1]) : 0.f;
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < kMaxSplits / 32; ++u) {
      const int r = lane + 32 * u;
      if (r < used) {
        const float mm = lv[u] > 0.f ? mv[u] : -INFINITY;
        s_w[warp * kMaxSplits + r] = mm;
        s_w[(8 + warp) * kMaxSplits + r] = lv[u];
        mx = fmaxf(mx, mm);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float Ls = 0.f;
    for (int r = lane; r < used; r += 32) {
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
  // Warp (part, head) adds up the records r ≡ part (mod parts) of its head, four coordinates
  // a lane (16-byte shared loads; the weight is one broadcast load per record); the parts'
  // sums meet in shared memory.
  const int parts = (kCompute / 32) / a.G;                     // G ≤ 8: at least one
  const bool mact = warp < parts * a.G;
  const int mp = warp / a.G, mh = warp - (warp / a.G) * a.G;
  float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
  for (int r0 = 0, ph = 0; r0 < used; r0 += chunk, ph ^= 1) {
    const bool okr = mbar_wait(&rec_bar, (unsigned)ph);
    if (!okr && tid == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    const int n = min(chunk, used - r0);
    if (okr && mact) {
      const float* wv = s_w + mh * kMaxSplits + r0;
      const float4* av = reinterpret_cast<const float4*>(srec + mh * kRec + 4) + lane;
      const int step4 = a.G * kRec / 4;
      int r = mp;
      for (; r + 3 * parts < n; r += 4 * parts) {   // four records' loads in flight
        float w[4];
        float4 v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          w[e] = wv[r + e * parts];
          v[e] = av[(r + e * parts) * step4];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float4& xx = (e & 1) ? x1 : x0;
          xx.x = fmaf(w[e], v[e].x, xx.x); xx.y = fmaf(w[e], v[e].y, xx.y);
          xx.z = fmaf(w[e], v[e].z, xx.z); xx.w = fmaf(w[e], v[e].w, xx.w);
        }
      }
      for (; r < n; r += parts) {
        const float w0 = wv[r];
        const float4 v0 = av[r * step4];
        x0.x = fmaf(w0, v0.x, x0.x); x0.y = fmaf(w0, v0.y, x0.y);
        x0.z = fmaf(w0, v0.z, x0.z); x0.w = fmaf(w0, v0.w, x0.w);
      }
    }
    if (r0 + chunk < used) {
      named_sync(kBarAll, kCompute);   // the chunk is consumed
      if (issuer) {
        fence_async_smem();
        issue_chunk(r0 + chunk);
      }
    }
  }
  if (mact)
    reinterpret_cast<float4*>(rpart + (mp * a.G + mh) * kPartPitch)[lane] =
        make_float4(x0.x + x1.x, x0.y + x1.y, x0.z + x1.z, x0.w + x1.w);
  named_sync(kBarAll, kCompute);
  // the merged accumulators, coordinate-major: mrg[j][h] (heads ≥ G are 0)
  for (int item = tid; item < 8 * TQ_D; item += kCompute) {
    const int j = item >> 3, h = item & 7;
    float v = 0.f;
    if (h < a.G)
      for (int p = 0; p < parts; ++p) v += rpart[(p * a.G + h) * kPartPitch + j];
    mrg[item] = v;
  }
  named_sync(kBarAll, kCompute);
  // rotation back, out_h = Πᵀ·mrg_h: warp w takes the rows j of Π in [128w/15, 128(w+1)/15),
  // lane l the output coordinates 4l..4l+3 of every head (one 16-byte load of Π and one or two
  // of mrg per 16 or 32 FMAs); the 15 partial sums go to the record area, free by now
  constexpr int kRotParts = kCompute / 32;
  float* rot = srec;                                            // [15][8][128]
  {
    const bool okpi = mbar_wait(&pi_bar, 0);   // every thread: the CTA may not finish before it
    if (!okpi && lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    constexpr int NH = HILO ? 4 : 8;                            // heads ≥ G have mrg = 0
    const int j0 = (TQ_D * warp) / kRotParts, j1 = (TQ_D * (warp + 1)) / kRotParts;
    const float* pis = reinterpret_cast<const float*>(smem + L::pi_off);
    float o[4][NH];
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
      for (int h = 0; h < NH; ++h) o[e][h] = 0.f;
    if (okpi) {
      for (int j = j0; j < j1; ++j) {
        const float4 p4 = *reinterpret_cast<const float4*>(pis + j * TQ_D + 4 * lane);
        float m[8];
        const float4 ma = *reinterpret_cast<const float4*>(mrg + 8 * j);
        m[0] = ma.x; m[1] = ma.y; m[2] = ma.z; m[3] = ma.w;
        if (NH == 8) {
          const float4 mb = *reinterpret_cast<const float4*>(mrg + 8 * j + 4);
          m[4] = mb.x; m[5] = mb.y; m[6] = mb.z; m[7] = mb.w;
        }
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          o[0][h] = fmaf(p4.x, m[h], o[0][h]);
          o[1][h] = fmaf(p4.y, m[h], o[1][h]);
          o[2][h] = fmaf(p4.z, m[h], o[2][h]);
          o[3][h] = fmaf(p4.w, m[h], o[3][h]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < NH; ++h)
      *reinterpret_cast<float4*>(rot + (warp * 8 + h) * TQ_D + 4 * lane) =
          make_float4(o[0][h], o[1][h], o[2][h], o[3][h]);
  }
  named_sync(kBarAll, kCompute);
  for (int item = tid; item < a.G * TQ_D; item += kCompute) {
    const int h = item >> 7, i = item & 127;
    const float Lh = s_hL[h];
    float x = 0.f;
#pragma unroll
    for (int p = 0; p < kRotParts; ++p) x += rot[(p * 8 + h) * TQ_D + i];
    const float v = Lh > 0.f ? x / Lh : 0.f;
    const long long e = ((long long)b * a.Hq + kvh * a.G + h) * TQ_D + i;
    if (a.out_dtype == TQ_F32) static_cast<float*>(a.out)[e] = v;
    else if (a.out_dtype == TQ_BF16) static_cast<__nv_bfloat16*>(a.out)[e] = __float2bfloat16_rn(v);
    else static_cast<__half*>(a.out)[e] = __float2half_rn(v);
  }
  if (tid == 0) a.counters[bh] = 0;   // ready for the next call
}

// Split count: as many CTAs as can be co-resident (one per SM) when every (batch, KV head)
// gets at least two, else the plan's splits in several waves; splits are whole tiles and only
// those that cover the longest sequence are launched.
template <int KB, int VB, bool HILO>
tq_status launch_one(const tq_mma_launch& a0, bool step, cudaStream_t stream) {
  // two softmax groups: a third (tried) adds no speed, the main loop being bound by the
  // SM's issue and integer-ALU throughput rather than by one warp's latency
  constexpr int NG = 2;
  constexpr int kThreads = Roles<NG>::threads;
  constexpr int smem = TL<KB, VB, HILO, NG>::total;
  // flat caches and page pools are separate instantiations: the flat kernel's producer has no
  // block-table code
  const int paged = a0.kmap.table || a0.vmap.table ? 1 : 0;
  auto kern = paged ? decode_tc_kernel<KB, VB, HILO, NG, true>
                    : decode_tc_kernel<KB, VB, HILO, NG, false>;
  static bool configured[2][64] = {};
  static int max_ctas[2][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return TQ_ERR_CUDA;
  if (!configured[paged][dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    max_ctas[paged][dev] = per_sm * tq_num_sms();
    configured[paged][dev] = true;
  }
  const int units = a0.B * a0.Hkv;
  int ns = max_ctas[paged][dev] / units;
  if (ns > a0.nsplit || ns < 2) ns = a0.nsplit;
  if (ns < 1) ns = 1;
  tq_mma_launch a = a0;
  long long sl = a.max_len > 0 ? (a.max_len + ns - 1) / ns : 1;
  sl = (sl + kTile - 1) / kTile * kTile;
  if (a.max_len > 0) {
    const int used = (int)((a.max_len + sl - 1) / sl);
    if (used < ns) ns = used;
  }
  a.nsplit = ns;
  a.split_len = (int)sl;
  {
    // the operand kernel (or the step's prologue) starts while the previous kernel in the
    // stream ends
    const long long units = (long long)a.B * a.Hkv;
    const int spc = units * kSlices <= 2LL * tq_num_sms() ? 1
                    : units * (kSlices / 2) <= 2LL * tq_num_sms() ? 2 : 4;
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3(kSlices / spc + (step ? (a.app.shared_pi ? 1 : 2) : 0), a.Hkv, a.B);
    pc.blockDim = dim3(step ? kAppendThreads : kPrepThreads);
    pc.stream = stream;
    cudaLaunchAttribute pa[1];
    pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pa[0].val.programmaticStreamSerializationAllowed = 1;
    pc.attrs = pa;
    pc.numAttrs = 1;
    auto prep = step ? (spc == 1   ? step_prologue_kernel<KB, HILO, 1>
                        : spc == 2 ? step_prologue_kernel<KB, HILO, 2>
                                   : step_prologue_kernel<KB, HILO, 4>)
                     : (spc == 1   ? query_prep_tc_kernel<KB, HILO, 1>
                        : spc == 2 ? query_prep_tc_kernel<KB, HILO, 2>
                                   : query_prep_tc_kernel<KB, HILO, 4>);
    if (cudaLaunchKernelEx(&pc, prep, a) != cudaSuccess) return TQ_ERR_CUDA;
  }
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
  if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return TQ_ERR_CUDA;
  return tq_cuda_status(cudaGetLastError());
}

template <int KB, int VB>
tq_status launch_kv(const tq_mma_launch& a, bool step, cudaStream_t stream) {
  return a.G <= 4 ? launch_one<KB, VB, true>(a, step, stream)
                  : launch_one<KB, VB, false>(a, step, stream);
}

template <int KB>
tq_status launch_k(const tq_mma_launch& a, bool step, cudaStream_t stream) {
  switch (a.vbits) {
    case 1: return launch_kv<KB, 1>(a, step, stream);
    case 2: return launch_kv<KB, 2>(a, step, stream);
    case 3: return launch_kv<KB, 3>(a, step, stream);
    case 4: return launch_kv<KB, 4>(a, step, stream);
  }
  return TQ_ERR_UNSUPPORTED;
}

tq_status launch_kbits(const tq_mma_launch& a, bool step, cudaStream_t stream) {
  if (!tq_tc_decode_supported(a.kbits, a.vbits, a.G, a.nsplit)) return TQ_ERR_UNSUPPORTED;
  if (!a.counters || !a.qfrag) return TQ_ERR_INVALID_ARG;
  switch (a.kbits) {
    case 1: return launch_k<1>(a, step, stream);
    case 2: return launch_k<2>(a, step, stream);
    case 3: return launch_k<3>(a, step, stream);
  }
  return TQ_ERR_UNSUPPORTED;
}

// A barrier that nothing ever arrives at, waited on with the kernels' bounded wait: the wait
// gives up after limit_ns of global time and raises TQ_FLAG_TIMEOUT, and the kernel returns.
// No copy, MMA or TMEM allocation is outstanding while it waits.
__global__ void bounded_wait_check_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
  }
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0, limit_ns);
  if (!__any_sync(0xffffffffu, ok) && threadIdx.x == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
}

}  // namespace

extern "C" tq_status tq_check_bounded_wait(uint32_t limit_us, tq_stream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u) return TQ_ERR_INVALID_ARG;
  bounded_wait_check_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      (unsigned long long)limit_us * 1000ull);
  return tq_cuda_status(cudaGetLastError());
}

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
  return launch_kbits(a, false, stream);
}

tq_status tq_launch_decode_step_tc(const tq_mma_launch& a, cudaStream_t stream) {
  if (!a.app.k_new || !a.app.v_new || !a.app.kmT) return TQ_ERR_INVALID_ARG;
  return launch_kbits(a, true, stream);
}

bool tq_step_prologue_fits(int batch, int kv_heads, int appends) {
  // the prologue runs one CTA of 512 threads per SM (its append CTAs' registers): use it when
  // all its CTAs fit in one wave
  const long long units = (long long)batch * kv_heads;
  const int sms = tq_num_sms();
  const int spc = units * kSlices <= 2LL * sms ? 1 : units * (kSlices / 2) <= 2LL * sms ? 2 : 4;
  return units * (kSlices / spc + appends) <= sms;
}
