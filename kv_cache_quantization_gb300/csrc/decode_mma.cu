// Split-context decode attention on packed codes with tensor-core contractions.
//
// The estimator of the QJL deep-dive (§五, §六) for key t and query head h is
//   s = ‖x_t‖·⟨Π q_h, c[idx_t]⟩ + ‖r_t‖·√(π/2)/d·⟨S q_h, 2·sign_t − 1⟩,
// and the value side accumulates Σ_t p_t·‖v_t‖·c_v[idx_t] in the rotated domain.  Both
// are contractions between a bit-structured operand and a small dense one, so the CTA
// runs them as mma.sync m16n8k16 (fp16 in, fp32 accumulate):
//
//  * key scores: A = 16 tokens × 16 coordinates taken straight from the packed bit
//    planes, B = 16 coordinates × 8 query columns (the GQA group, or 4 heads × hi/lo
//    halves of the query when G ≤ 4).  A bit becomes an fp16 operand with a single AND:
//    masking bit p (p = 10..14) of a 32-bit word yields an fp16 pair whose halves are 0 or
//    the power of two 2^e(p); the query carries 2^-e(p), so products are exact.  The
//    Lloyd-Max levels are expanded into odd Walsh monomials (XORs of bit planes) so that
//    every plane is a 0/1 matrix; coefficients live in the query operand.
//  * values: A = 16 coordinates × 16 tokens (4-bit codes through a shared-memory table of
//    level pairs; 1–3-bit codes as planes, transposed on load by ldmatrix.trans),
//    B = softmax weights × ‖v‖ transposed from the score accumulators with movmatrix.
//
// Packed K/V chunks stream through a 4-stage shared-memory ring filled by bulk-copy (TMA)
// engines and mbarriers; a dedicated producer warp issues the copies, eight consumer warps
// each own 16 tokens of a 128-token chunk and keep an online softmax; the CTA combines its
// warps and writes one (m, l, acc[128]) record per query head for the LSE merge.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "decode_mma.h"

TQ_DEFINE_FLAGS(tq_take_flags_decode_mma)

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = kConsumerWarps * 32;
constexpr int kTiles = 2;                     // 16-token tiles per warp per chunk
constexpr int kChunk = 16 * kTiles * kConsumerWarps;   // tokens per stage
constexpr int kStages = 4;
constexpr int kRec = TQ_REC;
constexpr unsigned kSpinLimit = 1u << 20;   // polls; a healthy wait needs a few hundred
// most splits per (batch, KV head) the last-CTA merge accepts
constexpr int kMaxSplits = 256;
// per-warp accumulators in the CTA combine: coordinate j of column col at col·140 + j + j/16,
// which spreads the 32 lanes of a fragment store over 32 banks
constexpr int kAccPitch = 140;
__host__ __device__ constexpr int accidx(int col, int j) { return col * kAccPitch + j + (j >> 4); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false after kSpinLimit polls (the caller raises TQ_FLAG_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  for (unsigned i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// ---------------------------------------------------------------- warp-level matrix ops
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
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
__device__ __forceinline__ void mma(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                    uint32_t b0, uint32_t b1) {
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

// ---------------------------------------------------------------- bit-pair expansion
// Pair e (0..15) of a 32-bit word holds bit lo(e) in its low fp16 half and bit lo(e)+16 in
// its high half, each as 0 or 2^exp(e):
//   e = 0..4  : bits 10+e,  26+e   (mask at 10+e)
//   e = 5..9  : bits e,     16+e   (word << 5,  mask at e+5)
//   e = 10..14: bits e-10,  e+6    (word << 10, mask at e)
//   e = 15    : bits 15,    31     (word >> 1,  mask at 14)
// An fp16 with only bit 10/11/12/13/14 set equals 2^-14 / 2^-13 / 2^-11 / 2^-7 / 2^1.
__host__ __device__ constexpr int pair_lo(int e) {
  return e < 5 ? 10 + e : e < 10 ? e : e < 15 ? e - 10 : 15;
}
__host__ __device__ constexpr int pair_pos(int e) { return e < 15 ? 10 + e % 5 : 14; }
__host__ __device__ constexpr int pos_exp(int pos) {
  return pos == 10 ? -14 : pos == 11 ? -13 : pos == 12 ? -11 : pos == 13 ? -7 : 1;
}

template <int E>
__device__ __forceinline__ uint32_t pair_of(uint32_t w, uint32_t w5, uint32_t w10, uint32_t w1) {
  constexpr int pos = pair_pos(E);
  constexpr uint32_t mask = (1u << pos) | (1u << (pos + 16));
  return (E < 5 ? w : E < 10 ? w5 : E < 15 ? w10 : w1) & mask;
}

// A plane word with the three shifted copies the pair extraction draws from; pair e is then
// one AND (e is a compile-time constant once the k-step loops are unrolled).
struct Shifted {
  uint32_t w, w5, w10, w1;
};
__device__ __forceinline__ Shifted shifted(uint32_t w) { return Shifted{w, w << 5, w << 10, w >> 1}; }
__device__ __forceinline__ uint32_t pair_at(const Shifted& x, int e) {
  const int pos = pair_pos(e);
  const uint32_t mask = (1u << pos) | (1u << (pos + 16));
  return (e < 5 ? x.w : e < 10 ? x.w5 : e < 15 ? x.w10 : x.w1) & mask;
}

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

// ---------------------------------------------------------------- query fragments
// The B operands of the key-score MMAs depend only on the lane (g = column, c = word of
// the planes), not on the warp: they are built once per (batch, KV head) by
// query_frag_kernel and copied into every CTA.  Word w of lane l sits at [w][32] + l.
//   w = (v·8 + s)·2 + half           v ≤ NKV (NKV = sign plane): rounded query
//   w = NWB + (v·8 + s)·2 + half     v < NKV, only when G > 4: the rounding residue
// followed by 8 columns × {A, Cm, B, Cq} score constants (floats).
__host__ __device__ constexpr int frag_words(int kb, bool hilo) {
  return (num_vplanes(kb) + 1) * 16 + (hilo ? 0 : num_vplanes(kb) * 16);
}
__host__ __device__ constexpr int frag_bytes(int kb, bool hilo) {
  return frag_words(kb, hilo) * 128 + 8 * 4 * 4;
}
constexpr int kMaxFragBytes = frag_bytes(3, false);
constexpr int kPrepThreads = 256;

// Grid (4 word slices c, KV heads, batch): the CTA for slice c computes Π q and S q only
// for coordinates 32c..32c+31 (the plane word c that lanes with lane % 4 == c hold) and
// writes those lanes' words.  The operand is normalised by ‖q‖ (|(Π q)_j| ≤ ‖q‖) and by
// smax·‖q‖ for the sketch (|(S q)_j| ≤ ‖S_j‖·‖q‖), and the column sums Σ_j (Π q)_j = (Πᵀ1)·q,
// Σ_j (S q)_j = (Sᵀ1)·q come straight from q, so no slice needs another slice's results.
template <int KB, bool HILO>
__global__ void __launch_bounds__(kPrepThreads) query_frag_kernel(const tq_mma_launch a) {
  constexpr int NKV = num_vplanes(KB);
  constexpr int NWB = (NKV + 1) * 16;
  constexpr int NW = frag_words(KB, HILO);
  __shared__ float qf[8][TQ_D];
  __shared__ float part[2][8][8][32];     // [Π|S][k part][head][j in slice]
  __shared__ float qsl[2][8][33];         // [Π|S][head][j in slice]
  __shared__ float s_nq[8], s_uq[8], s_wq[8];
  const int c = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long bh = (long long)b * a.Hkv + kvh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the decode grid may launch now: it streams the cache while this kernel runs and waits
  // for this grid's completion before it reads the fragments
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // 1. the group's queries (fp32), zero beyond G
#pragma unroll
  for (int r = 0; r < 8 * TQ_D / kPrepThreads; ++r) {
    const int i = tid + r * kPrepThreads;
    const int h = i / TQ_D, j = i % TQ_D;
    float v = 0.f;
    if (h < a.G) {
      const long long e = ((long long)b * a.Hq + kvh * a.G + h) * TQ_D + j;
      if (a.q_dtype == TQ_F32) v = static_cast<const float*>(a.q)[e];
      else if (a.q_dtype == TQ_BF16) v = __uint_as_float((uint32_t)static_cast<const uint16_t*>(a.q)[e] << 16);
      else v = __half2float(__ushort_as_half(static_cast<const uint16_t*>(a.q)[e]));
    }
    qf[h][j] = v;
  }
  // this slice of Πᵀ and Sᵀ: thread (k part, j) loads 16 of each (all loads first)
  const int jl = tid & 31, kp = tid >> 5;
  float tp[16], ts[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    tp[k] = __ldg(&a.piT[(16 * kp + k) * TQ_D + 32 * c + jl]);
    ts[k] = __ldg(&a.sT[(16 * kp + k) * TQ_D + 32 * c + jl]);
  }
  const float uk = __ldg(&a.u[lane * 4]), uk1 = __ldg(&a.u[lane * 4 + 1]);
  const float uk2 = __ldg(&a.u[lane * 4 + 2]), uk3 = __ldg(&a.u[lane * 4 + 3]);
  const float wk = __ldg(&a.w[lane * 4]), wk1 = __ldg(&a.w[lane * 4 + 1]);
  const float wk2 = __ldg(&a.w[lane * 4 + 2]), wk3 = __ldg(&a.w[lane * 4 + 3]);
  __syncthreads();
  // 2. per head: ‖q‖, (Πᵀ1)·q, (Sᵀ1)·q (warp h)
  if (warp < a.G) {
    const float* x = qf[warp] + lane * 4;
    float n2 = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
    float uq = uk * x[0] + uk1 * x[1] + uk2 * x[2] + uk3 * x[3];
    float wq = wk * x[0] + wk1 * x[1] + wk2 * x[2] + wk3 * x[3];
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
  // 3. slice products
  for (int h = 0; h < a.G; ++h) {
    float r = 0.f, q2 = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      r = fmaf(tp[k], qf[h][16 * kp + k], r);
      q2 = fmaf(ts[k], qf[h][16 * kp + k], q2);
    }
    part[0][kp][h][jl] = r;
    part[1][kp][h][jl] = q2;
  }
  __syncthreads();
  for (int i = tid; i < 2 * 8 * 32; i += kPrepThreads) {
    const int which = i >> 8, h = (i >> 5) & 7, j = i & 31;
    float v = 0.f;
    if (h < a.G)
      for (int k = 0; k < 8; ++k) v += part[which][k][h][j];
    qsl[which][h][j] = v;
  }
  __syncthreads();
  // 4. fragment words of the 8 lanes (g, c): column g
  uint32_t* out = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(a.qfrag) +
                                              bh * (long long)frag_bytes(KB, HILO));
  for (int i = tid; i < NW * 8; i += kPrepThreads) {
    const int g = i & 7, w = i >> 3;
    const bool residue_tile = w >= NWB;
    const int wv = residue_tile ? w - NWB : w;
    const int v = wv >> 4, s = (wv >> 1) & 7, half = wv & 1;
    const int e = 2 * s + half;
    const int j0 = pair_lo(e), j1 = j0 + 16;          // within the slice
    const float sc = exp2f((float)-pos_exp(pair_pos(e)));
    const int head = HILO ? (g >> 1) : g;
    float x0 = 0.f, x1 = 0.f;
    if (head < a.G && s_nq[head] > 0.f) {
      const bool sign_plane = v == NKV;
      const float coef = sign_plane ? 2.f : a.kd.coef[v];
      const float nrm = sign_plane ? 1.f / (s_nq[head] * a.smax) : 1.f / s_nq[head];
      const float* src = qsl[sign_plane ? 1 : 0][head];
      x0 = src[j0] * nrm * coef * sc;
      x1 = src[j1] * nrm * coef * sc;
    }
    const float r0 = x0 - __half2float(__float2half_rn(x0));
    const float r1 = x1 - __half2float(__float2half_rn(x1));
    // G ≤ 4: odd columns carry the rounding residue of the even column's head
    if (residue_tile || (HILO && (g & 1))) {
      x0 = r0;
      x1 = r1;
    }
    out[w * 32 + 4 * g + c] = pack_half2(x0, x1);
  }
  if (c == 0 && tid < 8) {
    // score constants of column n: A, Cm, B, Cq
    const int n = tid, head = HILO ? (n >> 1) : n;
    float* cst = reinterpret_cast<float*>(out + NW * 32);
    const float nq = head < a.G ? s_nq[head] : 0.f;
    const bool ok = nq > 0.f;
    cst[n * 4 + 0] = nq * a.scale_log2;
    cst[n * 4 + 1] = ok ? a.kd.cst * s_uq[head] / nq : 0.f;
    cst[n * 4 + 2] = nq * a.smax * a.scale_log2 * (1.2533141373155003f / TQ_D);
    cst[n * 4 + 3] = ok ? s_wq[head] / (nq * a.smax) : 0.f;
  }
}

// ---------------------------------------------------------------- shared-memory layout
template <int KB, int VB>
struct Layout {
  static constexpr int kplanes = 0;
  static constexpr int ksgn = kplanes + KB * kChunk * 16;
  static constexpr int kxn = ksgn + kChunk * 16;
  static constexpr int krn = kxn + kChunk * 4;
  static constexpr int vcodes = krn + kChunk * 4;
  static constexpr int vcode_bytes = VB == 4 ? kChunk * 64 : VB * kChunk * 16;
  static constexpr int vxn = vcodes + vcode_bytes;
  static constexpr int stage = vxn + kChunk * 4;            // bytes per stage
  static constexpr int ring = kStages * stage;
  static constexpr int lut = ring;                           // VB == 4: 256 × 32 words
  static constexpr int lut_bytes = VB == 4 ? 256 * 32 * 4 : 0;
  static constexpr int frag = lut + lut_bytes;               // query fragments + constants
  static constexpr int total = frag + kMaxFragBytes;
  // the CTA combine reuses everything above (ring, table and query buffer are dead by
  // then): per warp m, l, Σw [3][8] and acc [8][128]
  static constexpr int comb_acc = 0;
  static constexpr int comb_stats = kConsumerWarps * 8 * kAccPitch * 4;
  static_assert(comb_stats + (kConsumerWarps * 3 + kConsumerWarps) * 8 * 4 <= total, "combine buffer");
};

// ---------------------------------------------------------------- the kernel
template <int KB, int VB, bool HILO>
__global__ void __launch_bounds__(kThreads, 1) decode_mma_kernel(const tq_mma_launch a) {
  using L = Layout<KB, VB>;
  constexpr int NKV = num_vplanes(KB);                      // key virtual planes
  constexpr int NVV = VB == 4 ? 0 : num_vplanes(VB);
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t prol_bar;

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
  const int nchunks = t_end > t_begin ? (t_end - t_begin + kChunk - 1) / kChunk : 0;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    mbar_init(&prol_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ------------------------------------------------------------ copies (thread 0)
  // Thread 0 keeps kStages − 1 chunks in flight ahead of the one being consumed: it issues
  // chunk c into stage c % kStages once every warp has released that stage.
  auto issue = [&](int c) {
    const int st = c % kStages;
    const int t0 = t_begin + c * kChunk;
    const int n = min(kChunk, a.cap - t0);   // multiple of 64 (capacity is)
    unsigned char* base = smem + st * L::stage;
    const unsigned bytes = (unsigned)n * (KB * 16 + 16 + 4 + 4 + (VB == 4 ? 64 : VB * 16) + 4);
    mbar_expect_tx(&full_bar[st], bytes);
    for (int p = 0; p < KB; ++p)
      bulk_g2s(base + L::kplanes + p * kChunk * 16, a.kidx + ((bh * KB + p) * a.cap + t0) * 16,
               n * 16, &full_bar[st]);
    bulk_g2s(base + L::ksgn, a.ksgn + (bh * a.cap + t0) * 16, n * 16, &full_bar[st]);
    bulk_g2s(base + L::kxn, a.kxn + bh * a.cap + t0, n * 4, &full_bar[st]);
    bulk_g2s(base + L::krn, a.krn + bh * a.cap + t0, n * 4, &full_bar[st]);
    if (VB == 4) {
      bulk_g2s(base + L::vcodes, a.vidx + (bh * a.cap + t0) * 64, n * 64, &full_bar[st]);
    } else {
      for (int p = 0; p < VB; ++p)
        bulk_g2s(base + L::vcodes + p * kChunk * 16, a.vidx + ((bh * VB + p) * a.cap + t0) * 16,
                 n * 16, &full_bar[st]);
    }
    bulk_g2s(base + L::vxn, a.vxn + bh * a.cap + t0, n * 4, &full_bar[st]);
  };
  int issued = 0;   // chunks issued so far (meaningful in thread 0 only)
  if (tid == 0) {
    constexpr unsigned fb = frag_bytes(KB, HILO);
    mbar_expect_tx(&prol_bar, fb + (VB == 4 ? 256 * 32 * 4 : 0));
    if (VB == 4) bulk_g2s(smem + L::lut, a.lut, 256 * 32 * 4, &prol_bar);
    for (; issued < nchunks && issued < kStages; ++issued) issue(issued);
    // launched as a dependent of the fragment kernel: everything above only reads the
    // codec and the cache; the fragments are that kernel's output
    asm volatile("griddepcontrol.wait;" ::: "memory");
    bulk_g2s(smem + L::frag, reinterpret_cast<const unsigned char*>(a.qfrag) + bh * (long long)fb,
             fb, &prol_bar);
  }

  // ------------------------------------------------------------ prologue
  // query fragments (and the value pair table) arrive by bulk copy as well
  if (tid == 0 && !mbar_wait(&prol_bar, 0)) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
  __syncthreads();
  const int g = lane >> 2, c = lane & 3;
  uint32_t bq[NKV + 1][8][2];
  uint32_t bql[HILO ? 1 : NKV][8][2];
  {
    const uint32_t* fw = reinterpret_cast<const uint32_t*>(smem + L::frag) + lane;
#pragma unroll
    for (int v = 0; v <= NKV; ++v)
#pragma unroll
      for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int half = 0; half < 2; ++half) bq[v][s][half] = fw[((v * 8 + s) * 2 + half) * 32];
    if (!HILO) {
#pragma unroll
      for (int v = 0; v < NKV; ++v)
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
          for (int half = 0; half < 2; ++half)
            bql[v][s][half] = fw[((NKV + 1) * 16 + (v * 8 + s) * 2 + half) * 32];
    }
  }
  // score constants of this thread's columns (2c, 2c+1)
  float hA[2], hCm[2], hB[2], hCq[2];
  {
    const float* cst = reinterpret_cast<const float*>(smem + L::frag + frag_words(KB, HILO) * 128);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int col = HILO ? 2 * c : 2 * c + k;
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
  bool timed_out = false;

  // ------------------------------------------------------------ main loop
  for (int ch = 0; ch < nchunks; ++ch) {
    const int st = ch % kStages;
    if (!mbar_wait(&full_bar[st], (ch / kStages) & 1)) {
      atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
      timed_out = true;
      break;
    }
    const unsigned char* base = smem + st * L::stage;
    const float* kxn = reinterpret_cast<const float*>(base + L::kxn);
    const float* krn = reinterpret_cast<const float*>(base + L::krn);
    const float* vxn = reinterpret_cast<const float*>(base + L::vxn);
    const int t_chunk = t_begin + ch * kChunk;           // absolute index of the chunk's token 0
    const int r8 = lane & 7, m8 = (lane >> 3) & 1;       // ldmatrix row addressing

    // ---- key scores of the warp's two tiles: D[token][column]; one chain per tile
    float dm[kTiles][4] = {}, dq[kTiles][4] = {}, dml[kTiles][4] = {};
    {
      uint32_t pw[kTiles][3][2] = {}, sw[kTiles][2];
#pragma unroll
      for (int T = 0; T < kTiles; ++T) {
        const int row = 32 * warp + 16 * T + r8 + 8 * m8;
        if (KB >= 2) {
          // matrices: plane0 rows 0-7, plane0 rows 8-15, plane1 rows 0-7, plane1 rows 8-15
          const int p = lane >> 4;
          ldsm_x4(smem_u32(base + L::kplanes + p * kChunk * 16 + row * 16), pw[T][0][0],
                  pw[T][0][1], pw[T][1][0], pw[T][1][1]);
        }
        if (KB == 1 || KB == 3) {
          const int p = KB - 1;
          ldsm_x2(smem_u32(base + L::kplanes + p * kChunk * 16 + row * 16), pw[T][p][0], pw[T][p][1]);
        }
        ldsm_x2(smem_u32(base + L::ksgn + row * 16), sw[T][0], sw[T][1]);
      }
#pragma unroll
      for (int v = 0; v <= NKV; ++v) {
        Shifted x[kTiles][2];   // [tile][row g / row g + 8]
#pragma unroll
        for (int T = 0; T < kTiles; ++T)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const uint32_t words[3] = {pw[T][0][hr], pw[T][1][hr], pw[T][2][hr]};
            x[T][hr] = shifted(v < NKV ? vplane_word<KB>(words, v) : sw[T][hr]);
          }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
#pragma unroll
          for (int T = 0; T < kTiles; ++T) {
            const uint32_t a0 = pair_at(x[T][0], 2 * s), a1 = pair_at(x[T][1], 2 * s);
            const uint32_t a2 = pair_at(x[T][0], 2 * s + 1), a3 = pair_at(x[T][1], 2 * s + 1);
            mma(v < NKV ? dm[T] : dq[T], a0, a1, a2, a3, bq[v][s][0], bq[v][s][1]);
            if (!HILO && v < NKV) mma(dml[T], a0, a1, a2, a3, bql[v][s][0], bql[v][s][1]);
          }
        }
      }
      if (!HILO) {
#pragma unroll
        for (int T = 0; T < kTiles; ++T)
#pragma unroll
          for (int i = 0; i < 4; ++i) dm[T][i] += dml[T][i];
      }
    }
    // ---- scores → base-2 logits; rows: token g (k = 0) and g + 8 (k = 1) of each tile
    float lg[kTiles][2][2];   // [tile][row][column pair]
#pragma unroll
    for (int T = 0; T < kTiles; ++T) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int tl = 32 * warp + 16 * T + g + 8 * k;
        const bool valid = t_chunk + tl < t_end;
        const float xn = kxn[tl], rn = krn[tl];
        if (HILO) {
          const float m = dm[T][2 * k] + dm[T][2 * k + 1], q = dq[T][2 * k] + dq[T][2 * k + 1];
          const float sc = xn * hA[0] * (m - hCm[0]) + rn * hB[0] * (q - hCq[0]);
          lg[T][k][0] = lg[T][k][1] = valid ? sc : -INFINITY;
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float sc = xn * hA[h] * (dm[T][2 * k + h] - hCm[h]) +
                             rn * hB[h] * (dq[T][2 * k + h] - hCq[h]);
            lg[T][k][h] = valid ? sc : -INFINITY;
          }
        }
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
      for (int i = 0; i < 8; ++i) {
        acc[i][0] *= corr[0];
        acc[i][1] *= corr[1];
        acc[i][2] *= corr[0];
        acc[i][3] *= corr[1];
      }
    }
    float w[kTiles][2][2];
#pragma unroll
    for (int T = 0; T < kTiles; ++T) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        // tokens past the sequence (or past the capacity in a short last chunk) may hold
        // stale bytes: their weight is exactly zero, never 0 × (stale norm)
        const int tl = 32 * warp + 16 * T + g + 8 * k;
        const bool valid = t_chunk + tl < t_end;
        const float vn = vxn[tl];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float pr = valid ? exp2f(lg[T][k][h] - m_run[h]) : 0.f;
          l_run[h] += pr;
          w[T][k][h] = valid ? pr * vn : 0.f;
          lw_run[h] += w[T][k][h];
        }
      }
    }
    // ---- value accumulation: acc[coord][column] += Σ_t A[coord][t] · B[t][column]
#pragma unroll
    for (int T = 0; T < kTiles; ++T) {
      const int trow0 = 32 * warp + 16 * T;              // tile's first token in the chunk
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
          for (int i = 0; i < 4; ++i) {
            const uint32_t a0 = lut_lane[((klo01 >> (8 * i)) & 0xffu) << 5];
            const uint32_t a1 = lut_lane[((khi01 >> (8 * i)) & 0xffu) << 5];
            const uint32_t a2 = lut_lane[((klo23 >> (8 * i)) & 0xffu) << 5];
            const uint32_t a3 = lut_lane[((khi23 >> (8 * i)) & 0xffu) << 5];
            mma(acc[4 * half + i], a0, a1, a2, a3, bw0, bw1);
          }
        }
      } else {
        // planes transposed on load: pair word = {chunk g of token 2c, chunk g of token 2c+1}
        uint32_t mw[3][2] = {};
#pragma unroll
        for (int p = 0; p < VB; ++p)
          ldsm_x2_t(smem_u32(base + L::vcodes + p * kChunk * 16 + (trow0 + r8 + 8 * m8) * 16),
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
          for (int i = 0; i < 8; ++i)
            mma(acc[i], pair_at(e0, 2 * i), pair_at(e0, 2 * i + 1), pair_at(e1, 2 * i),
                pair_at(e1, 2 * i + 1), bw0, bw1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[st]);
    if (tid == 0 && ch + kStages < nchunks) {
      if (!mbar_wait(&empty_bar[st], (ch / kStages) & 1)) {
        atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
        timed_out = true;
        break;
      }
      issue(ch + kStages);
      ++issued;
    }
  }
  if (timed_out && tid == 0) {
    // a stage never filled or was never released: let the copies this thread issued land
    // before the CTA's shared memory is reused or released (bounded as well)
    for (int c = issued - kStages > 0 ? issued - kStages : 0; c < issued; ++c)
      mbar_wait(&full_bar[c % kStages], (c / kStages) & 1);
  }

  // ------------------------------------------------------------ CTA combine
  // l and Σw over the 16 rows of each column (lanes sharing c)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], o);
      lw_run[h] += __shfl_xor_sync(0xffffffffu, lw_run[h], o);
    }
  }
  // the merge grid may be scheduled now (it waits for this grid's completion)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  consumer_sync();   // every warp is done with the ring: reuse it
  float* cacc = reinterpret_cast<float*>(smem + L::comb_acc);           // [warp][col][140]
  float* cst = reinterpret_cast<float*>(smem + L::comb_stats);          // [warp][3][8]
  float* fac = cst + kConsumerWarps * 3 * 8;                            // [warp][8]
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int hi_row = k >> 1;                  // 0: row g, 1: row g + 8
      const int col = 2 * c + (k & 1);
      int coord;
      float v = acc[i][k];
      if (VB == 4) {
        coord = 16 * g + 2 * i + hi_row;
        v *= a.vc_unscale;
      } else {
        const int e = 2 * i + hi_row;
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
      cst[(warp * 3 + 0) * 8 + col] = m_run[k];
      cst[(warp * 3 + 1) * 8 + col] = l_run[k];
      cst[(warp * 3 + 2) * 8 + col] = lw_run[k];
    }
  }
  consumer_sync();
  // per column: the CTA maximum and each warp's rescaling factor, computed once
  __shared__ float s_M[8], s_L[8], s_LW[8];
  if (tid < 8) {
    const int col = tid;
    float M = -INFINITY;
    for (int wp = 0; wp < kConsumerWarps; ++wp) M = fmaxf(M, cst[(wp * 3) * 8 + col]);
    float Lsum = 0.f, lw = 0.f;
    for (int wp = 0; wp < kConsumerWarps; ++wp) {
      const float mw_ = cst[(wp * 3) * 8 + col];
      const float f = (M == -INFINITY || mw_ == -INFINITY) ? 0.f : exp2f(mw_ - M);
      fac[wp * 8 + col] = f;
      Lsum += f * cst[(wp * 3 + 1) * 8 + col];
      lw += f * cst[(wp * 3 + 2) * 8 + col];
    }
    s_M[col] = M;
    s_L[col] = Lsum;
    s_LW[col] = lw;
  }
  consumer_sync();
  float* rec_base = a.part + ((bh * a.nsplit + split) * a.G) * kRec;
  for (int i = tid; i < a.G * TQ_D; i += kConsumerWarps * 32) {
    const int head = i / TQ_D, j = i % TQ_D;
    const int col = HILO ? 2 * head : head;
    float acc_j = 0.f;
#pragma unroll
    for (int wp = 0; wp < kConsumerWarps; ++wp) {
      float av = cacc[accidx(wp * 8 + col, j)];
      if (HILO) av += cacc[accidx(wp * 8 + col + 1, j)];
      acc_j = fmaf(fac[wp * 8 + col], av, acc_j);
    }
    if (VB != 4) acc_j -= a.vd.cst * s_LW[col];
    float* rec = rec_base + head * kRec;
    if (j == 0) {
      // natural-log maximum (the merge combines with expf)
      rec[0] = s_M[col] == -INFINITY ? -INFINITY : s_M[col] * 0.69314718055994531f;
      rec[1] = s_L[col];
    }
    rec[2 + j] = acc_j;
  }
}

// ---------------------------------------------------------------- merge
// One CTA of 512 threads per (batch, query head), launched as a dependent of the split
// kernel: Π is prefetched into registers before the dependency wait; the split records are
// then read with all loads in flight, combined with log-sum-exp weights and rotated back,
// out = Πᵀ·acc / L.
constexpr int kMergeThreads = 512;
__global__ void __launch_bounds__(kMergeThreads) merge_mma_kernel(const tq_mma_launch a) {
  __shared__ float s_w[kMaxSplits];
  __shared__ float s_part[4][TQ_D], s_acc[TQ_D], s_red[32];
  __shared__ float s_M, s_L;
  const int row = blockIdx.x;            // b * Hq + h
  const int b = row / a.Hq, h = row % a.Hq;
  const int kvh = h / a.G, g = h % a.G;
  const long long bh = (long long)b * a.Hkv + kvh;
  const int tid = threadIdx.x, j = tid & 127, q = tid >> 7, warp = tid >> 5, lane = tid & 31;
  float tp[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) tp[k] = __ldg(&a.pi[(32 * q + k) * TQ_D + j]);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float* recs = a.part + (bh * a.nsplit * a.G + g) * kRec;   // split s at + s·G·kRec
  float m = -INFINITY, l = 0.f;
  if (tid < a.nsplit) {
    m = __ldcg(&recs[(long long)tid * a.G * kRec]);
    l = __ldcg(&recs[(long long)tid * a.G * kRec + 1]);
    if (!(l > 0.f)) m = -INFINITY;
  }
  // M = max over splits (block reduction)
  float mx = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) s_red[warp] = mx;
  __syncthreads();
  if (tid < 32) {
    float v = tid < kMergeThreads / 32 ? s_red[tid] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (tid == 0) s_M = v;
  }
  __syncthreads();
  const float M = s_M;
  float lw = 0.f;
  if (tid < a.nsplit) {
    const float w = (M == -INFINITY || m == -INFINITY) ? 0.f : expf(m - M);
    s_w[tid] = w;
    lw = w * l;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
  __syncthreads();
  if (lane == 0) s_red[warp] = lw;
  __syncthreads();
  if (tid < 32) {
    float v = tid < kMergeThreads / 32 ? s_red[tid] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (tid == 0) s_L = v;
  }
  // acc_j: splits q, q+4, q+8, ... of thread (q, j), loads issued together
  float acc = 0.f;
  {
    float v[16];
    const int n = (a.nsplit - q + 3) / 4;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      v[i] = i < n ? __ldcg(&recs[(long long)(q + 4 * i) * a.G * kRec + 2 + j]) : 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i < n) acc = fmaf(s_w[q + 4 * i], v[i], acc);
    for (int i = 16; i < n; ++i)   // more than 64 splits
      acc = fmaf(s_w[q + 4 * i], __ldcg(&recs[(long long)(q + 4 * i) * a.G * kRec + 2 + j]), acc);
  }
  s_part[q][j] = acc;
  __syncthreads();
  if (tid < TQ_D) s_acc[tid] = (s_part[0][tid] + s_part[1][tid]) + (s_part[2][tid] + s_part[3][tid]);
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int k = 0; k < 32; ++k) r = fmaf(tp[k], s_acc[32 * q + k], r);
  s_part[q][j] = r;
  __syncthreads();
  if (tid < TQ_D) {
    const float L = s_L;
    const float o = L > 0.f ? ((s_part[0][tid] + s_part[1][tid]) + (s_part[2][tid] + s_part[3][tid])) / L : 0.f;
    const long long e = (long long)row * TQ_D + tid;
    if (a.out_dtype == TQ_F32) static_cast<float*>(a.out)[e] = o;
    else if (a.out_dtype == TQ_BF16) static_cast<__nv_bfloat16*>(a.out)[e] = __float2bfloat16_rn(o);
    else static_cast<__half*>(a.out)[e] = __float2half_rn(o);
  }
}

template <int KB, int VB, bool HILO>
tq_status launch_one(const tq_mma_launch& a, cudaStream_t stream) {
  constexpr int smem = Layout<KB, VB>::total;
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return TQ_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(decode_mma_kernel<KB, VB, HILO>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return TQ_ERR_CUDA;
    configured[dev] = true;
  }
  query_frag_kernel<KB, HILO><<<dim3(4, a.Hkv, a.B), kPrepThreads, 0, stream>>>(a);
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
  if (cudaLaunchKernelEx(&cfg, decode_mma_kernel<KB, VB, HILO>, a) != cudaSuccess)
    return TQ_ERR_CUDA;
  cudaLaunchConfig_t mcfg = cfg;
  mcfg.gridDim = dim3(a.B * a.Hq);
  mcfg.blockDim = dim3(kMergeThreads);
  mcfg.dynamicSmemBytes = 0;
  if (cudaLaunchKernelEx(&mcfg, merge_mma_kernel, a) != cudaSuccess) return TQ_ERR_CUDA;
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

bool tq_mma_supported(int kbits, int vbits, int G) {
  return kbits >= 1 && kbits <= 3 && vbits >= 1 && vbits <= 4 && G >= 1 && G <= 8;
}

tq_plane_decomp tq_decompose_levels(const tq_codec* c) {
  // Walsh–Hadamard coefficients of the levels over the ±1 bit variables.
  tq_plane_decomp d{};
  const int B = c->ibits, L = c->levels;
  static const int masks[3][4] = {{1, 0, 0, 0}, {1, 2, 0, 0}, {1, 2, 4, 7}};
  const int nv = B == 1 ? 1 : B == 2 ? 2 : 4;
  d.n = nv;
  double cst = 0;
  for (int v = 0; v < nv; ++v) {
    const int m = masks[B - 1][v];
    double a = 0;
    for (int idx = 0; idx < L; ++idx) {
      int prod = 1;
      for (int i = 0; i < B; ++i)
        if (m & (1 << i)) prod *= ((idx >> i) & 1) ? 1 : -1;
      a += (double)c->centroids_d[idx] * prod;
    }
    a /= L;
    d.coef[v] = (float)(2 * a);
    cst += a;
  }
  d.cst = (float)cst;
  return d;
}

tq_status tq_launch_decode_mma(const tq_mma_launch& a, cudaStream_t stream) {
  if (!tq_mma_supported(a.kbits, a.vbits, a.G)) return TQ_ERR_UNSUPPORTED;
  switch (a.kbits) {
    case 1: return launch_k<1>(a, stream);
    case 2: return launch_k<2>(a, stream);
    case 3: return launch_k<3>(a, stream);
  }
  return TQ_ERR_UNSUPPORTED;
}

float tq_fp16_friendly_scale(const float* levels, int n) {
  // An exhaustive search over σ = 1 + k/2^16: the table is then exact to a few 1e-5 instead
  // of the 2.4e-4 of plain fp16 rounding.
  float best = 1.f;
  double best_err = 1e30;
  for (int k = 0; k < (1 << 16); ++k) {
    const float sg = 1.f + (float)k / 65536.f;
    double worst = 0;
    for (int i = 0; i < n; ++i) {
      const float x = sg * levels[i];
      if (x == 0.f) continue;
      const float r = __half2float(__float2half_rn(x));
      worst = fmax(worst, fabs((double)r - x) / fabs((double)x));
      if (worst >= best_err) break;
    }
    if (worst < best_err) {
      best_err = worst;
      best = sg;
    }
  }
  return best;
}

size_t tq_mma_frag_bytes_max() { return (size_t)kMaxFragBytes; }
