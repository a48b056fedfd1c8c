// Quantisation on the fifth-generation tensor cores (tcgen05, accumulators in TMEM).
//
// QJL deep-dive §二: y = Π x/‖x‖ (rotation), per-coordinate Lloyd-Max index, residual
// ρ = y − c[idx] and the sketch signs sign(M ρ), M = S Πᵀ (so that sign(M ρ) = sign(S r)).
// For a tile of 128 vectors the two 128×128 products are tensor-core GEMMs with
// M = 128 vectors, N = 128 outputs, K = 128 coordinates:
//
//   GEMM 1  D1 = X̂ · Π̂ᵀ     X̂ = x·2^s in fp16, s chosen per vector so that max|x|·2^s lies
//                          in [2^14, 2^15): exact for bf16 and fp16 inputs.  Π̂ = 64·Π as an
//                          fp16 pair hi + lo (22 significant bits): 2 MMAs per k-step.
//   GEMM 2  D2 = ρ̂ · M̂ᵀ     ρ̂ = 256·ρ and M̂ = 8·M, both fp16 pairs: hi·hi + hi·lo + lo·hi,
//                          3 MMAs per k-step.
//
// Both products accumulate in fp32 in TMEM.  The decisions they feed (index cells, sign
// bits) need the rotated coordinates to about 1e-7 in unit-sphere units, which the pairs give
// (2^-22 relative per operand, fp32 accumulation) and a single fp16 operand would not.
//
// Operands sit in shared memory in the canonical K-major layout without swizzle (8-row ×
// 16-byte core matrices; LBO = distance between K-adjacent core matrices, SBO = between
// 8-row groups).  The codec keeps Π̂ and M̂ in exactly that image, so one bulk copy per
// image brings them in once per CTA.  Raw activations arrive by bulk copies (the TMA engine;
// one per run of contiguous vectors) one tile ahead of the tile being computed.
//
// Two threads own vector r of the tile (TMEM lane r): lane r % 32 of warps q and q + 4 of a
// group (the same TMEM lane quadrant q = r / 32), part p taking coordinates 64p onwards.  Each
// reads its part of the row of D1 / D2, decides indices and signs, builds its part of every
// code plane in registers and writes it with one store; the parts of ‖ρ‖² meet in shared
// memory.  One CTA per SM, persistent over tiles, made of groups of 256 threads that take
// alternate tiles, each with its own operand and staging buffers, accumulator columns and
// barriers: one group for the product quantiser (its shared memory holds Π̂ and M̂), two for
// the MSE quantiser, so that one group's conversion and epilogue overlap the other's product
// and copies.
#include <cuda_fp16.h>

#include "tc_ptx.h"
#include "tq_internal.h"

TQ_DEFINE_FLAGS(tq_take_flags_quantize_tc)

namespace {

constexpr int kTileV = 128;                    // vectors per tile (MMA M)
constexpr int kImg = 128 * 128 * 2;            // one 128×128 fp16 operand image (32 KB)
constexpr int kLBO = 128;                      // K-adjacent core matrices
constexpr int kSBO = 16 * 128;                 // 8-row groups: 16 core matrices along K
constexpr int kRawPitch = 256;                 // one raw bf16/fp16 vector
constexpr float kPiScale = 64.f, kMScale = 8.f, kRhoScale = 256.f;

// shared-memory map of the MSE quantiser (bytes from the dynamic base): the codec's Π̂ image,
// then one area per group of 256 threads
struct ML {
  static constexpr int kGroups = 2;
  static constexpr int kParts = 2;                               // threads per vector
  static constexpr int pi = 0;                                   // Π̂ hi | lo
  static constexpr int area = 2 * kImg;                          // group 0's area
  // offsets inside a group's area
  static constexpr int a = 0;                                    // X̂
  static constexpr int raw = kImg;                               // raw vectors of the next tile
  static constexpr int norm = raw + kTileV * kRawPitch;          // float ‖x‖ [128]
  static constexpr int ysc = norm + 4 * kTileV;                  // float D1 → y scale [128]
  static constexpr int gsize = ysc + 4 * kTileV;
  // mbarriers: the codec's image, then (raw tile, MMA) per group; then the TMEM slot
  static constexpr int bars = area + kGroups * gsize;
  static constexpr int total = bars + 8 * (1 + 2 * kGroups) + 8;
  static constexpr int tmem_cols = 256;                          // D1 per group
};
// shared-memory map of the product quantiser: the codec's Π̂ and M̂ images, two tile buffers
// (each holds a tile's raw vectors, then X̂ in place, then ρ̂ hi), the ρ̂ lo image, and small
// per-tile arrays
struct PL {
  static constexpr int kParts = 4;                               // threads per vector
  static constexpr int kThreads = 128 * kParts + 32;             // compute warps + issuer warp
  static constexpr int pi = 0;                                   // Π̂ hi | lo
  static constexpr int m = 2 * kImg;                             // M̂ hi | lo
  static constexpr int buf = 4 * kImg;                           // tile buffers [2]
  static constexpr int lo = 6 * kImg;                            // ρ̂ lo
  static constexpr int ns = 7 * kImg;                            // float ‖x‖·2^s [2][128]
  static constexpr int rr = ns + 2 * 4 * kTileV;                 // float ‖ρ‖² of parts 1..3
  static constexpr int sexp = rr + (kParts - 1) * 4 * kTileV;    // int8 s [2][128]
  // mbarriers: the codec's images, raw tile [2], GEMM 1, GEMM 2, X̂ ready, ρ̂ ready; then the
  // TMEM slot
  static constexpr int bars = sexp + 2 * kTileV;
  static constexpr int total = bars + 8 * 7 + 8;
  static constexpr int tmem_cols = 256;                          // D1 | D2
};
static_assert(ML::total <= 227 * 1024 && PL::total <= 227 * 1024, "shared memory budget");
static_assert(ML::gsize % 1024 == 0 && PL::bars % 8 == 0, "alignment");

__device__ __forceinline__ uint32_t s32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// byte offset of element (row r, column k) in a canonical K-major 128 × 128 fp16 image
__device__ __forceinline__ int canon(int r, int k) {
  return (r >> 3) * kSBO + (k >> 3) * kLBO + (r & 7) * 16 + (k & 7) * 2;
}
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)(kLBO >> 4) << 16) |
         ((uint64_t)(kSBO >> 4) << 32) | ((uint64_t)1 << 46);
}
// kind::f16 with fp16 A and B, fp32 accumulator, both K-major, M = 128, N = 128
constexpr uint32_t kIdesc =
    (1u << 4) | ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          s32(bar))
      : "memory");
}
// bounded wait (the thread is suspended, not spinning, while the phase is incomplete)
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity) {
  return tq::mbar_wait(bar, parity);
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void async_proxy_fence() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// barrier of one group of nt threads (named barrier 1 + group), and its AND-reduction
__device__ __forceinline__ void group_sync(int group, int nt) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(nt) : "memory");
}
__device__ __forceinline__ bool group_sync_and(int group, bool v, int nt) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(1 + group), "r"(nt)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(s32(dst)), "l"(src), "r"(bytes), "r"(s32(bar))
      : "memory");
}
__device__ __forceinline__ void arrive_expect(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s32(bar)),
               "r"(bytes)
               : "memory");
}

struct TcArgs {
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
  int capacity;
  const void* img;           // Π̂ hi | lo (| M̂ hi | lo for prod), canonical images
  tq_levels lv;
  bool narrow;               // batch·heads·tokens < 2^32: vector indices split in 32 bits
};

// (batch·heads + head, token) of vector gi of the flattened (batch, head, token) range; the
// 32-bit division is a short sequence, the 64-bit one a long dependent chain
__device__ __forceinline__ void split_vec(const TcArgs& a, long long gi, int& bh, int& t) {
  if (a.narrow) {
    const uint32_t g = (uint32_t)gi, n = (uint32_t)a.tokens;
    bh = (int)(g / n);
    t = (int)(g - (uint32_t)bh * n);
  } else {
    bh = (int)(gi / a.tokens);
    t = (int)(gi - (long long)bh * a.tokens);
  }
}
// element offset of vector gi
__device__ __forceinline__ long long vec_offset(const TcArgs& a, long long gi) {
  int bh, t;
  split_vec(a, gi, bh, t);
  const int b = (int)((uint32_t)bh / (uint32_t)a.heads);
  return (long long)b * a.sb + (long long)(bh - b * a.heads) * a.sh + (long long)t * a.st;
}

// Warp 0: bring the raw vectors of `tile` into the staging buffer.  Where the token stride is
// one vector, the tile's vectors of one (batch, head) are contiguous in memory and move as one
// bulk copy (lane v issues the run that starts at vector v: the tile's first vector or a
// sequence's token 0); otherwise each vector is its own copy.  The TMA engine takes a bulk
// copy at a time, so 128 small copies would hold the issuing warp for microseconds.
__device__ __forceinline__ void issue_tile(const TcArgs& a, long long tile, long long total,
                                           unsigned char* raw, uint64_t* bar, int lane) {
  const long long first = tile * kTileV;
  const int nvalid = (int)min((long long)kTileV, total - first);
  if (lane == 0) arrive_expect(bar, (unsigned)nvalid * kRawPitch);
  __syncwarp();
  const uint16_t* x = static_cast<const uint16_t*>(a.x);
  if (a.st == TQ_D) {
    for (int v = lane; v < nvalid; v += 32) {
      int bh, t;
      split_vec(a, first + v, bh, t);
      if (v > 0 && t > 0) continue;   // inside a run that an earlier vector starts
      const int n = min(nvalid - v, a.tokens - t);
      bulk_g2s(raw + v * kRawPitch, x + vec_offset(a, first + v), (unsigned)n * kRawPitch, bar);
    }
  } else {
    for (int v = lane; v < nvalid; v += 32)
      bulk_g2s(raw + v * kRawPitch, x + vec_offset(a, first + v), kRawPitch, bar);
  }
}

// Index cell of y and its level, for a codebook whose levels are antisymmetric (every
// Lloyd-Max codebook of the symmetric coordinate law is).  With h = 2^(IB−1) levels per
// side, cnt = #{positive boundaries ≤ |y|}; y ≥ 0 gives cell h + cnt, y < 0 cell h−1−cnt.
// This equals #{boundaries ≤ y} except when |y| equals a boundary exactly.
template <int IB>
__device__ __forceinline__ int cell_of(float y, const tq_levels& lv, float& level) {
  constexpr int h = 1 << (IB - 1);
  const float ay = fabsf(y);
  int cnt = 0;
  float c = lv.c[h];
#pragma unroll
  for (int k = 0; k < h - 1; ++k) {
    const bool p = lv.b[h + k] <= ay;
    cnt += p ? 1 : 0;
    c = p ? lv.c[h + k + 1] : c;
  }
  const bool pos = y >= 0.f;
  level = pos ? c : -c;
  return pos ? (h | cnt) : ((h - 1) ^ cnt);
}

// ---- conversion: raw bf16/fp16 vectors → X̂ (fp16, per-vector power-of-two scale) and ‖x‖.
// A warp converts eight vectors: lane (i = lane & 7, g = lane >> 3) takes chunks
// (g + 4j + i) mod 16, j < 4, of vector i of the eight, so that both the staging reads and the
// canonical writes of a quarter-warp fall in distinct banks.
__device__ __forceinline__ int conv_chunk(int lane, int j) {
  return ((lane >> 3) + 4 * j + (lane & 7)) & 15;
}
__device__ __forceinline__ void load_raw(const unsigned char* raw, int v, bool valid, int lane,
                                         uint32_t (&w)[4][4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 u = make_uint4(0, 0, 0, 0);
    if (valid) u = *reinterpret_cast<const uint4*>(raw + v * kRawPitch + conv_chunk(lane, j) * 16);
    w[j][0] = u.x; w[j][1] = u.y; w[j][2] = u.z; w[j][3] = u.w;
  }
}
// X̂ words of the lane's chunks and, agreed by the vector's lanes, ns = ‖x‖·2^s and s, with
// 2^s putting max|x|·2^s in [2^14, 2^15) (s clamped to [-114, 126]): exact in fp16 for bf16 and
// fp16 inputs, and ‖x‖ summed over the scaled values neither overflows nor underflows in fp32
// anywhere in the bf16 range.
__device__ __forceinline__ void convert_chunks(const uint32_t (&w)[4][4], int dtype,
                                               uint32_t (&hw)[4][4], float& ns, int& s) {
  float f[4][8];
  float mx = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (dtype == TQ_BF16) {
        f[j][2 * e] = __uint_as_float(w[j][e] << 16);
        f[j][2 * e + 1] = __uint_as_float(w[j][e] & 0xffff0000u);
      } else {
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[j][e]));
        f[j][2 * e] = t.x;
        f[j][2 * e + 1] = t.y;
      }
      mx = fmaxf(mx, fmaxf(fabsf(f[j][2 * e]), fabsf(f[j][2 * e + 1])));
    }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  const int eb = (int)((__float_as_uint(mx) >> 23) & 0xffu);
  s = min(141 - eb, 126);
  const float sc = __uint_as_float((uint32_t)(s + 127) << 23);
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = f[j][2 * e] * sc, x1 = f[j][2 * e + 1] * sc;
      ss = fmaf(x0, x0, ss);
      ss = fmaf(x1, x1, ss);
      const __half2 h2 = __floats2half2_rn(x0, x1);
      hw[j][e] = *reinterpret_cast<const uint32_t*>(&h2);
    }
  ss += __shfl_xor_sync(0xffffffffu, ss, 8);
  ss += __shfl_xor_sync(0xffffffffu, ss, 16);
  ns = sqrtf(ss);
}
__device__ __forceinline__ void store_canon(unsigned char* img, int v, int lane,
                                            const uint32_t (&hw)[4][4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(img + canon(v, 8 * conv_chunk(lane, j))) =
        make_uint4(hw[j][0], hw[j][1], hw[j][2], hw[j][3]);
}
// ‖x‖ and the D1 → y scale from ns = ‖x‖·2^s (D1 = 64·2^s·Π x)
__device__ __forceinline__ float norm_of(float ns, int s) {
  return ns * __uint_as_float((uint32_t)(127 - s) << 23);
}
__device__ __forceinline__ float yscale_of(float ns) {
  return ns > 0.f ? 1.f / (kPiScale * ns) : 0.f;
}

// ---- first epilogue of one 32-coordinate block: the cells of y = dv·ysc, this block's code
// words (index planes: word p holds bit p of the 32 cells; 4-bit nibbles: 4 words), and the
// residual ρ = y − level, returned as Σ ρ² with kRhoScale·ρ left in dv.
template <int IB, bool kNib>
__device__ __forceinline__ float cells_block(float (&dv)[32], float ysc, const tq_levels& lv,
                                             uint32_t (&code)[kNib ? 4 : IB]) {
#pragma unroll
  for (int k = 0; k < (kNib ? 4 : IB); ++k) code[k] = 0;
  float rr = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float y = dv[e] * ysc;
    float level;
    const int q = cell_of<IB>(y, lv, level);
    if constexpr (kNib) {
      code[e >> 3] |= (uint32_t)q << (4 * (e & 7));
    } else {
#pragma unroll
      for (int p = 0; p < IB; ++p) code[p] |= (uint32_t)((q >> p) & 1) << e;
    }
    const float rho = y - level;
    rr = fmaf(rho, rho, rr);
    dv[e] = rho * kRhoScale;
  }
  return rr;
}
// ρ̂ of one block as an fp16 pair into the canonical A images (row r, columns 32·blk + …)
__device__ __forceinline__ void store_rho_pair(const float (&dv)[32], unsigned char* hi_img,
                                               unsigned char* lo_img, int r, int blk) {
#pragma unroll
  for (int c8 = 0; c8 < 4; ++c8) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const float v0 = dv[8 * c8 + 2 * e2], v1 = dv[8 * c8 + 2 * e2 + 1];
      const __half2 hh = __floats2half2_rn(v0, v1);
      const float2 hf = __half22float2(hh);
      const __half2 ll = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
      hi[e2] = *reinterpret_cast<const uint32_t*>(&hh);
      lo[e2] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    const int off = canon(r, 32 * blk + 8 * c8);
    *reinterpret_cast<uint4*>(hi_img + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(lo_img + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}
// GEMM 1 of a tile: D1 = X̂ · (Π̂hi + Π̂lo)ᵀ (one thread)
__device__ __forceinline__ void issue_gemm1(uint32_t d1, uint32_t sa, uint32_t sp) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint64_t ad = sdesc(sa + ks * 2 * kLBO);
    mma_f16(d1, ad, sdesc(sp + ks * 2 * kLBO), ks > 0 ? 1u : 0u);
    mma_f16(d1, ad, sdesc(sp + kImg + ks * 2 * kLBO), 1u);
  }
}
// the tile's vector r: its (batch·heads + head, token) and its sequence's count and position
struct VecDest {
  int bh = 0, t = 0, cnt = 0, p0 = 0;
};
__device__ __forceinline__ VecDest vec_dest(const TcArgs& a, long long first, int r, int nvalid) {
  VecDest d;
  if (r < nvalid) {
    split_vec(a, first + r, d.bh, d.t);
    const int b = (int)((uint32_t)d.bh / (uint32_t)a.heads);
    d.cnt = a.count ? a.count[b] : a.tokens;
    d.p0 = a.pos ? a.pos[b] : 0;
  }
  return d;
}
// its cache position, or -1 (not stored; a position out of range is flagged)
__device__ __forceinline__ int dest_pos(const TcArgs& a, const VecDest& d, int r, int nvalid) {
  if (r >= nvalid || d.t >= d.cnt) return -1;
  const int p = d.p0 + d.t;
  if (p >= 0 && p < a.capacity) return p;
  atomicOr(&g_tq_flags, TQ_FLAG_POS_OVERFLOW);
  return -1;
}

// The MSE quantiser.  One CTA per SM, persistent over tiles, made of two groups of 256 threads
// (two per vector: warps q and q + 4 of a group share TMEM lane quadrant q, part p taking
// coordinates 64p onwards) that take alternate tiles, each with its own operand and staging
// buffers, accumulator columns and barriers, so that one group's conversion and epilogue
// overlap the other's product and copies.  Per tile: conversion, GEMM 1, epilogue.
template <int IB>
__global__ void __launch_bounds__(128 * ML::kParts * ML::kGroups, 1)
    quantize_mse_tc_kernel(TcArgs a) {
  using L = ML;
  constexpr int kGroups = L::kGroups;
  constexpr int kGT = 128 * L::kParts;           // threads per group
  constexpr bool kNib = IB == 4;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this thread's group, and its warp inside the group
  const int group = warp / (kGT / 32), gw = warp % (kGT / 32);
  unsigned char* area = smem + L::area + group * L::gsize;
  float* s_norm = reinterpret_cast<float*>(area + L::norm);
  float* s_ysc = reinterpret_cast<float*>(area + L::ysc);
  uint64_t* bar_const = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* bar_x = bar_const + 1 + 2 * group;
  uint64_t* bar_mma = bar_x + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_const + 1 + 2 * kGroups);
  unsigned char* raw = area + L::raw;
  const long long total = (long long)a.batch * a.heads * a.tokens;
  const long long ntiles = (total + kTileV - 1) / kTileV;
  // the CTA's tiles blockIdx.x + k·gridDim.x go to its groups in turn
  const long long tile0 = blockIdx.x + (long long)group * gridDim.x;
  const long long tstep = (long long)kGroups * gridDim.x;

  if (tid == 0) {
    for (int b = 0; b < 1 + 2 * kGroups; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s32(bar_const + b)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     s32(s_tmem)),
                 "r"(L::tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t d1 = tmem + 128 * group;
  // TMEM lane quadrant (rows 32·quad..) and coordinate part (blocks 2·half..) of this warp
  const int quad = gw & 3, half = gw >> 2;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;

  if (gw == 0) {
    if (warp == 0 && lane == 0 && blockIdx.x < ntiles) {
      arrive_expect(bar_const, 2 * kImg);
      bulk_g2s(smem + L::pi, a.img, 2 * kImg, bar_const);
    }
    if (tile0 < ntiles) issue_tile(a, tile0, total, raw, bar_x, lane);
  }
  bool ok = blockIdx.x >= ntiles || bar_wait(bar_const, 0);
  ok = __syncthreads_and(ok);
  bool x_pending = tile0 < ntiles;        // a raw-tile copy is in flight
  bool mma_pending = false;               // an MMA group is in flight
  uint32_t px = 0, pm = 0;

  for (long long tile = tile0; tile < ntiles && ok; tile += tstep) {
    const long long first = tile * kTileV;
    const int nvalid = (int)min((long long)kTileV, total - first);
    const int r = 32 * quad + lane;   // this thread's vector in the epilogue
    const VecDest vd = vec_dest(a, first, r, nvalid);   // requested now, used after the conversion
    ok = group_sync_and(group, bar_wait(bar_x, px), kGT);
    if (!ok) break;
    px ^= 1;
    x_pending = false;
    // ---- raw → X̂ and ‖x‖: warp w of the group converts vectors 16w.., eight at a time
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const int v = 16 * gw + 8 * pass + (lane & 7);
      uint32_t w[4][4], hw[4][4];
      load_raw(raw, v, v < nvalid, lane, w);
      float ns;
      int s;
      convert_chunks(w, a.dtype, hw, ns, s);
      store_canon(area + L::a, v, lane, hw);
      if (lane < 8) {
        s_norm[v] = norm_of(ns, s);
        s_ysc[v] = yscale_of(ns);
      }
    }
    const int dst = dest_pos(a, vd, r, nvalid);
    const long long slot = (long long)vd.bh * a.capacity + dst;
    async_proxy_fence();   // X̂ (generic writes) → tensor-core reads
    tc_before();
    group_sync(group, kGT);
    tc_after();
    if (gw == 0) {
      if (lane == 0) {
        issue_gemm1(d1, s32(area + L::a), s32(smem + L::pi));
        mma_commit(bar_mma);
      }
      __syncwarp();
    } else if (gw == 1) {
      // the staging buffer is free: the group's next tile comes in while this one is computed
      // (issued beside the MMAs: an MMA issue waits while the tensor core's queue is full)
      const long long next = tile + tstep;
      if (next < ntiles) {
        async_proxy_fence();
        issue_tile(a, next, total, raw, bar_x, lane);
      }
    }
    x_pending = tile + tstep < ntiles;
    mma_pending = true;
    ok = group_sync_and(group, bar_wait(bar_mma, pm), kGT);
    if (!ok) break;
    pm ^= 1;
    mma_pending = false;
    tc_after();

    // ---- epilogue (vector r, coordinate blocks 2·half, 2·half + 1): index codes
    const float n = s_norm[r];
    const float ysc = s_ysc[r];
    uint32_t code[2][kNib ? 4 : IB];
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      float dv[32];
      tmem_ld32(d1 + lane_base + 32 * (2 * half + hb), dv);
      cells_block<IB, kNib>(dv, ysc, a.lv, code[hb]);
    }
    if (dst >= 0) {
      if constexpr (kNib) {
        uint4* dp = reinterpret_cast<uint4*>(a.idx + slot * 64 + 32 * half);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb)
          dp[hb] = make_uint4(code[hb][0], code[hb][1], code[hb][2], code[hb][3]);
      } else {
#pragma unroll
        for (int p = 0; p < IB; ++p) {
          unsigned char* row =
              a.idx + (((long long)vd.bh * IB + p) * a.capacity + dst) * 16 + 8 * half;
          *reinterpret_cast<uint2*>(row) = make_uint2(code[0][p], code[1][p]);
        }
      }
      if (half == 0) a.xnorm[slot] = n;
    }
    tc_before();
    group_sync(group, kGT);   // D1 read and X̂ consumed before the next tile reuses them
    tc_after();
  }
  if (!ok) {
    // a bounded wait gave up: report it, let in-flight copies and MMAs land (bounded) and
    // release the accumulator columns before leaving
    if (tid == group * kGT) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
    if (x_pending) bar_wait(bar_x, px);
    if (mma_pending) bar_wait(bar_mma, pm);
  }
  tc_before();
  __syncthreads();
  tc_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(L::tmem_cols));
}

// The product quantiser.  One CTA per SM, persistent over the tiles blockIdx.x + j·gridDim.x,
// two tiles in flight: 16 compute warps (four threads per vector: TMEM lane quadrant
// q = warp & 3, part p = warp >> 2 taking coordinates 32p..32p+31) and one issuer warp, which
// issues the MMAs and the tiles' bulk copies (an MMA issue waits while the tensor core's queue
// is full, so an issuing compute warp would hold up every barrier of the tile).  Tile j's raw
// vectors arrive in buffer j & 1 and are converted there in place to X̂; GEMM 1 reads them; the
// first epilogue writes ρ̂ hi over X̂ and ρ̂ lo into the lo image; GEMM 2 reads both.  While
// GEMM 2 of tile j runs, the compute warps convert tile j + 1 in the other buffer; while GEMM 1
// of tile j + 1 runs, they take the sign epilogue of tile j, and tile j's buffer receives tile
// j + 2.  The compute warps hand each operand to the issuer on an mbarrier (one arrival per
// warp); the tensor core's commits hand the products back.
template <int IB>
__global__ void __launch_bounds__(PL::kThreads, 1) quantize_prod_tc_kernel(TcArgs a) {
  using L = PL;
  constexpr int kCompute = 128 * L::kParts;   // compute threads (warps 0..15)
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* s_ns = reinterpret_cast<float*>(smem + L::ns);
  float* s_rr = reinterpret_cast<float*>(smem + L::rr);
  signed char* s_exp = reinterpret_cast<signed char*>(smem + L::sexp);
  uint64_t* bar_const = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* bar_x = bar_const + 1;        // [2], one per tile buffer (bulk copies)
  uint64_t* bar_g1 = bar_const + 3;       // GEMM 1 done (tensor-core commit)
  uint64_t* bar_g2 = bar_const + 4;       // GEMM 2 done
  uint64_t* bar_a1 = bar_const + 5;       // X̂ ready (one arrival per compute warp)
  uint64_t* bar_a2 = bar_const + 6;       // ρ̂ ready
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_const + 7);
  unsigned char* lo_img = smem + L::lo;
  const long long total = (long long)a.batch * a.heads * a.tokens;
  const long long ntiles = (total + kTileV - 1) / kTileV;
  const int nt = blockIdx.x < ntiles ? (int)((ntiles - 1 - blockIdx.x) / gridDim.x) + 1 : 0;
  auto tile_first = [&](int j) { return (blockIdx.x + (long long)j * gridDim.x) * kTileV; };
  auto buffer = [&](int j) { return smem + L::buf + (j & 1) * kImg; };

  if (tid == 0) {
    for (int b = 0; b < 7; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s32(bar_const + b)),
                   "r"(b >= 5 ? kCompute / 32 : 1));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     s32(s_tmem)),
                 "r"(L::tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t d1 = tmem, d2 = tmem + 128;

  if (warp == kCompute / 32) {
    // ---- issuer warp: the codec's images and the first two tiles, then per tile its GEMM 1,
    // GEMM 2 and, once GEMM 2 has read the tile's buffer, the copy of the tile two ahead
    bool ok = true;
    uint32_t xbits = 0, xphase = 0;   // copies in flight per buffer; phases issued per buffer
    int g1_issued = 0, g2_issued = 0, g2_seen = 0;
    auto copy_tile = [&](int j) {
      issue_tile(a, tile_first(j) / kTileV, total, buffer(j), bar_x + (j & 1), lane);
      xbits |= 1u << (j & 1);
      xphase ^= 1u << (j & 1);
    };
    if (nt > 0) {
      if (lane == 0) {
        arrive_expect(bar_const, 4 * kImg);
        bulk_g2s(smem + L::pi, a.img, 4 * kImg, bar_const);
      }
      copy_tile(0);
      if (nt > 1) copy_tile(1);
    }
    auto gemm1 = [&](int j) {
      ok = __all_sync(0xffffffffu, tq::mbar_wait(bar_a1, j & 1));   // uniform across the warp
      if (!ok) return;
      tc_after();
      if (lane == 0) {
        issue_gemm1(d1, s32(buffer(j)), s32(smem + L::pi));
        mma_commit(bar_g1);
      }
      __syncwarp();
      ++g1_issued;
    };
    auto gemm2 = [&](int j) {
      ok = __all_sync(0xffffffffu, tq::mbar_wait(bar_a2, j & 1));
      if (!ok) return;
      tc_after();
      if (lane == 0) {
        // D2 = ρ̂hi·M̂hiᵀ + ρ̂hi·M̂loᵀ + ρ̂lo·M̂hiᵀ
        const uint32_t sh = s32(buffer(j)), sl = s32(lo_img);
        const uint32_t smh = s32(smem + L::m), sml = smh + kImg;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t o = ks * 2 * kLBO;
          mma_f16(d2, sdesc(sh + o), sdesc(smh + o), ks > 0 ? 1u : 0u);
          mma_f16(d2, sdesc(sh + o), sdesc(sml + o), 1u);
          mma_f16(d2, sdesc(sl + o), sdesc(smh + o), 1u);
        }
        mma_commit(bar_g2);
      }
      __syncwarp();
      ++g2_issued;
    };
    if (nt > 0) gemm1(0);
    if (nt > 0 && ok) gemm2(0);
    for (int j = 0; j < nt && ok; ++j) {
      if (j + 1 < nt) {
        gemm1(j + 1);
        if (!ok) break;
      }
      // GEMM 2 of tile j has read buffer j & 1 (and its raw copy was consumed before it)
      ok = __all_sync(0xffffffffu, tq::mbar_wait(bar_g2, j & 1));
      if (!ok) break;
      g2_seen = j + 1;
      xbits &= ~(1u << (j & 1));
      if (j + 2 < nt) {
        async_proxy_fence();
        copy_tile(j + 2);
      }
      if (j + 1 < nt) {
        gemm2(j + 1);
        if (!ok) break;
      }
    }
    if (!ok) {
      // a bounded wait gave up: report it and let this warp's copies and MMAs land (bounded)
      if (lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
      for (int k = 0; k < 2; ++k)
        if ((xbits >> k) & 1u) tq::mbar_wait(bar_x + k, ((xphase >> k) & 1u) ^ 1u);
      if (g1_issued > 0) tq::mbar_wait(bar_g1, (g1_issued - 1) & 1);
      if (g2_issued > g2_seen) tq::mbar_wait(bar_g2, (g2_issued - 1) & 1);
    }
  } else {
    // ---- compute warps
    const int quad = warp & 3, part = warp >> 2;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const int r = 32 * quad + lane;   // this thread's vector in the epilogues
    bool ok = nt == 0 || bar_wait(bar_const, 0);
    ok = group_sync_and(0, ok, kCompute);
    uint32_t px = 0, pg1 = 0, pg2 = 0;   // parity of each barrier's next phase
    // vector r of the tile whose sign epilogue comes next: its destination and ‖x‖
    int dst = -1;
    long long slot = 0;
    float n = 0.f;
    VecDest vd;   // vector r of the tile whose first epilogue comes next
    auto hand_over = [&](uint64_t* bar) {   // this warp's operand writes → the issuer
      async_proxy_fence();
      tc_before();
      __syncwarp();
      if (lane == 0) tq::mbar_arrive(bar);
    };
    // conversion of tile j in place
    auto convert = [&](int j) {
      const int k = j & 1;
      unsigned char* b = buffer(j);
      const long long first = tile_first(j);
      const int nvalid = (int)min((long long)kTileV, total - first);
      vd = vec_dest(a, first, r, nvalid);   // used by the first epilogue
      ok = group_sync_and(0, bar_wait(bar_x + k, (px >> k) & 1u), kCompute);
      if (!ok) return;
      px ^= 1u << k;
      const int v = 8 * warp + (lane & 7);
      uint32_t w[4][4], hw[4][4];
      load_raw(b, v, v < nvalid, lane, w);
      group_sync(0, kCompute);   // every raw chunk is in registers before the buffer is rewritten
      float ns;
      int s;
      convert_chunks(w, a.dtype, hw, ns, s);
      store_canon(b, v, lane, hw);
      if (lane < 8) {
        s_ns[k * kTileV + v] = ns;
        s_exp[k * kTileV + v] = (signed char)s;
      }
      hand_over(bar_a1);
      group_sync(0, kCompute);   // the norms are in place for the first epilogue
    };
    // first epilogue of tile j: index planes, ‖x‖, ρ̂, ‖ρ‖
    auto epilogue1 = [&](int j) {
      const int k = j & 1;
      const long long first = tile_first(j);
      const int nvalid = (int)min((long long)kTileV, total - first);
      ok = group_sync_and(0, bar_wait(bar_g1, pg1), kCompute);
      if (!ok) return;
      pg1 ^= 1;
      tc_after();
      dst = dest_pos(a, vd, r, nvalid);
      slot = (long long)vd.bh * a.capacity + dst;
      const float ns = s_ns[k * kTileV + r];
      n = norm_of(ns, s_exp[k * kTileV + r]);
      float dv[32];
      tmem_ld32(d1 + lane_base + 32 * part, dv);
      uint32_t code[IB];
      const float rr = cells_block<IB, false>(dv, yscale_of(ns), a.lv, code);
      store_rho_pair(dv, buffer(j), lo_img, r, part);
      if (part > 0) s_rr[(part - 1) * kTileV + r] = rr;
      hand_over(bar_a2);
      if (dst >= 0) {
#pragma unroll
        for (int p = 0; p < IB; ++p)
          *reinterpret_cast<uint32_t*>(
              a.idx + (((long long)vd.bh * IB + p) * a.capacity + dst) * 16 + 4 * part) = code[p];
        if (part == 0) a.xnorm[slot] = n;
      }
      group_sync(0, kCompute);   // the parts of ‖ρ‖² are in place
      if (part == 0 && dst >= 0) {
        float rt = rr;
#pragma unroll
        for (int pp = 0; pp < L::kParts - 1; ++pp) rt += s_rr[pp * kTileV + r];
        a.rnorm[slot] = n * sqrtf(rt);
      }
    };
    // sign epilogue of tile j
    auto epilogue2 = [&](int j) {
      ok = group_sync_and(0, bar_wait(bar_g2, pg2), kCompute);
      if (!ok) return;
      pg2 ^= 1;
      tc_after();
      float dv[32];
      tmem_ld32(d2 + lane_base + 32 * part, dv);
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 32; ++e) word |= (dv[e] >= 0.f ? 1u : 0u) << e;
      tc_before();   // D2 read before a later GEMM 2 is issued
      if (dst >= 0)   // zero vector: zero residual, all signs +1
        *reinterpret_cast<uint32_t*>(a.sgn + slot * 16 + 4 * part) = n > 0.f ? word : 0xffffffffu;
    };

    if (nt > 0 && ok) {
      convert(0);
      if (ok) epilogue1(0);
    }
    for (int j = 0; j < nt && ok; ++j) {
      if (j + 1 < nt) {
        convert(j + 1);
        if (!ok) break;
      }
      epilogue2(j);
      if (!ok) break;
      if (j + 1 < nt) epilogue1(j + 1);
    }
    if (!ok && tid == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
  }
  tc_before();
  __syncthreads();
  tc_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(L::tmem_cols));
}

template <typename Kernel>
tq_status launch_tc(Kernel kernel, int threads, int smem_bytes, bool& configured,
                    const TcArgs& a, int grid, cudaStream_t stream) {
  if (!configured) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
        cudaSuccess)
      return TQ_ERR_CUDA;
    configured = true;
  }
  kernel<<<grid, threads, smem_bytes, stream>>>(a);
  return tq_cuda_status(cudaGetLastError());
}

template <bool kProd, int IB>
tq_status launch_tc(const TcArgs& a, int grid, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return TQ_ERR_CUDA;
  if (kProd)
    return launch_tc(quantize_prod_tc_kernel<IB>, PL::kThreads, PL::total, configured[dev], a,
                     grid, stream);
  return launch_tc(quantize_mse_tc_kernel<IB>, 128 * ML::kParts * ML::kGroups, ML::total,
                   configured[dev], a, grid, stream);
}

}  // namespace

bool tq_quantize_tc_supported(int dtype) { return dtype == TQ_BF16 || dtype == TQ_F16; }

tq_status tq_launch_quantize_tc(bool prod, const void* x, int dtype, int batch, int heads,
                                int tokens, long long sb, long long sh, long long st,
                                const int* pos, const int* count, uint8_t* idx, uint8_t* sgn,
                                float* xnorm, float* rnorm, int capacity, const tq_codec* c,
                                cudaStream_t stream) {
  TcArgs a{};
  a.x = x; a.dtype = dtype; a.batch = batch; a.heads = heads; a.tokens = tokens;
  a.sb = sb; a.sh = sh; a.st = st; a.pos = pos; a.count = count;
  a.idx = idx; a.sgn = sgn; a.xnorm = xnorm; a.rnorm = rnorm; a.capacity = capacity;
  a.img = c->d_img; a.lv = tq_make_levels(c);
  const long long total = (long long)batch * heads * tokens;
  a.narrow = total < (1ll << 32);
  if (total == 0) return TQ_OK;
  if (!a.img) return TQ_ERR_INVALID_ARG;
  const long long ntiles = (total + kTileV - 1) / kTileV;
  const int sms = tq_num_sms() > 0 ? tq_num_sms() : 1;
  const int grid = (int)(ntiles < sms ? ntiles : sms);
  switch (prod ? 10 + c->ibits : c->ibits) {
    case 11: return launch_tc<true, 1>(a, grid, stream);
    case 12: return launch_tc<true, 2>(a, grid, stream);
    case 13: return launch_tc<true, 3>(a, grid, stream);
    case 14: return launch_tc<true, 4>(a, grid, stream);
    case 1: return launch_tc<false, 1>(a, grid, stream);
    case 2: return launch_tc<false, 2>(a, grid, stream);
    case 3: return launch_tc<false, 3>(a, grid, stream);
    case 4: return launch_tc<false, 4>(a, grid, stream);
  }
  return TQ_ERR_UNSUPPORTED;
}

size_t tq_operand_image_bytes(bool prod) { return (size_t)(prod ? 4 : 2) * kImg; }

// Host: the canonical K-major image of scale·mat (mat row-major [n][k], 128 × 128) as an
// fp16 pair — the hi image followed by the lo image.
void tq_build_operand_image(const double* mat, bool sketch, uint16_t* img) {
  const double scale = sketch ? kMScale : kPiScale;
  for (int n = 0; n < 128; ++n)
    for (int k = 0; k < 128; ++k) {
      const double v = scale * mat[(size_t)n * 128 + k];
      const __half hi = __float2half_rn((float)v);
      const __half lo = __float2half_rn((float)(v - (double)__half2float(hi)));
      const int off = ((n >> 3) * kSBO + (k >> 3) * kLBO + (n & 7) * 16 + (k & 7) * 2) / 2;
      img[off] = __half_as_ushort(hi);
      img[kImg / 2 + off] = __half_as_ushort(lo);
    }
}
