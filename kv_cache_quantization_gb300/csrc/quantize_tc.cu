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
// Π̂, M̂ and X̂ sit in shared memory in the canonical K-major layout without swizzle (8-row ×
// 16-byte core matrices; LBO = distance between K-adjacent core matrices, SBO = between
// 8-row groups).  The codec keeps Π̂ and M̂ in exactly that image, so one bulk copy brings them
// in once per CTA.  Raw activations arrive by bulk copies (the TMA engine; one per run of
// contiguous vectors) into a ring of tile buffers, where they are converted to X̂ in place.
// ρ̂ goes to tensor memory, the A operand of GEMM 2.
//
// The thread that owns vector r of a tile reads row r of D1 / D2 (TMEM lane r), decides its
// part of the indices and signs, builds its part of every code plane in registers and writes
// it with one store.  The warp roles and the pipeline across tiles are described at the
// kernel.
#include <cuda_fp16.h>

#include <type_traits>

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

// Roles of a quantiser CTA: epilogue warps (warp w reads TMEM lane quadrant w % 4, part w / 4 of
// each vector's coordinates), converter warps, an issuer warp (MMAs) and a copy warp.  The
// product code's epilogues, and those of MSE codes of 3 or 4 bits (longer cell searches), carry
// most of the work: two parts of 64 coordinates per vector; for 1- and 2-bit MSE codes the
// conversion does.
template <bool kProd, int IB>
struct Roles {
  static constexpr bool kHeavyEpi = kProd || IB >= 3;
  static constexpr int kEpiWarps = kHeavyEpi ? 8 : 4, kConvWarps = kHeavyEpi ? 4 : 8;
  static constexpr int kParts = kEpiWarps / 4;              // threads per vector
  static constexpr int kBlocks = 4 / kParts;                // 32-coordinate blocks per thread
  static constexpr int kIssuer = kEpiWarps + kConvWarps, kCopier = kIssuer + 1;   // warps
  static constexpr int kThreads = 32 * (kEpiWarps + kConvWarps + 2);
};

// Shared-memory map (bytes from the dynamic base): the codec's images (Π̂ hi | lo, and for the
// product code M̂ hi | lo), the tile buffers (each holds a tile's raw vectors, then X̂ in place),
// per-buffer ‖x‖·2^s and s, part 1's ‖ρ‖², the positive boundaries and levels (3- and 4-bit
// cells), the tile index of each buffer, the mbarriers and the TMEM slot.
template <bool kProd>
struct QL {
  static constexpr int kBufs = kProd ? 3 : 4;
  static constexpr int pi = 0;                                   // Π̂ hi | lo, then M̂ hi | lo
  static constexpr int buf = (kProd ? 4 : 2) * kImg;             // tile buffers [kBufs]
  static constexpr int ns = buf + kBufs * kImg;                  // float ‖x‖·2^s [kBufs][128]
  static constexpr int rr = ns + kBufs * 4 * kTileV;             // float ‖ρ‖² of part 1 [128]
  static constexpr int sexp = rr + 4 * kTileV;                   // int8 s [kBufs][128]
  static constexpr int tab = sexp + kBufs * kTileV;              // float boundaries, levels [16]
  static constexpr int tiles = tab + 16 * 4;                     // long long tile index [kBufs]
  // codec images; per buffer: raw tile in, X̂ ready, buffer free for the next copy; per D1
  // slot: GEMM 1 done; then the epilogue done per D1 slot (MSE code), or epilogue 1 done,
  // epilogue 2 done, GEMM 2 done, part 1's ‖ρ‖² in place
  static constexpr int nbars = 1 + 3 * kBufs + 2 + (kProd ? 4 : 2);
  static constexpr int bars = tiles + 8 * 4;
  static constexpr int total = bars + 8 * nbars + 8;
  static constexpr int tmem_cols = kProd ? 512 : 256;
};
// TMEM columns: D1 [2], then for the product code D2 | ρ̂ hi | ρ̂ lo
constexpr int kD2Col = 256, kRhoCol = 384;
static_assert(QL<true>::total <= 227 * 1024 && QL<false>::total <= 227 * 1024,
              "shared memory budget");

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
  int capacity;              // slots per sequence
  tq_rowmap map;             // flat, or the pool's block table
  int rowcap;                // slots per cache row: capacity (flat) or page_tokens (paged)
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

// Whether a tile holds a vector to store: with per-sequence counts, tiles past a sequence's
// count (the padding of a ragged batch) are skipped; a tile that runs into the next sequence is
// kept.
__device__ __forceinline__ bool tile_live(const TcArgs& a, long long tile) {
  if (!a.count) return true;
  int bh, t;
  split_vec(a, tile * kTileV, bh, t);
  if (t + kTileV > a.tokens) return true;
  return t < a.count[(uint32_t)bh / (uint32_t)a.heads];
}
// A cursor over the live tiles among tile0 + k·stride, in order: the position (batch, head,
// token) of the candidate's first vector advances by additions, and a sequence's count is read
// when the cursor enters its batch row.
struct LiveCursor {
  long long tile, ntiles;
  int stride, b, h, t, cb, cnt;
  __device__ __forceinline__ LiveCursor(const TcArgs& a, long long tile0, int stride_,
                                        long long ntiles_)
      : tile(tile0), ntiles(ntiles_), stride(stride_), cb(-1), cnt(0) {
    int bh;
    split_vec(a, tile0 * kTileV, bh, t);
    b = (int)((uint32_t)bh / (uint32_t)a.heads);
    h = bh - b * a.heads;
  }
  __device__ __forceinline__ bool live(const TcArgs& a) {
    if (!a.count || t + kTileV > a.tokens) return true;
    if (b != cb) {
      cb = b;
      cnt = a.count[b];
    }
    return t < cnt;
  }
  __device__ __forceinline__ void step(const TcArgs& a) {
    tile += stride;
    long long tt = (long long)t + (long long)stride * kTileV;
    if (tt >= a.tokens) {
      const long long q = tt / a.tokens;   // sequences passed (rarely more than one)
      tt -= q * a.tokens;
      const long long hh = h + q;
      b += (int)(hh / a.heads);
      h = (int)(hh % a.heads);
    }
    t = (int)tt;
  }
  // the next live tile (≥ ntiles when there is none)
  __device__ __forceinline__ long long next(const TcArgs& a) {
    while (tile < ntiles && !live(a)) step(a);
    const long long r = tile;
    if (tile < ntiles) step(a);
    return r;
  }
};

// Bring the raw vectors of `tile` into a tile buffer (one warp).  Where the token stride is one
// vector, the tile's vectors of one (batch, head) are contiguous in memory and move as one bulk
// copy: for sequences of at least 32 tokens lane 0 walks the tile's runs (at most a few), else
// lane v issues the run that starts at vector v (the tile's first vector or a sequence's token 0).
// Otherwise each vector is its own copy.
__device__ __forceinline__ void issue_tile(const TcArgs& a, long long tile, long long total,
                                           unsigned char* raw, uint64_t* bar, int lane) {
  const long long first = tile * kTileV;
  const int nvalid = (int)min((long long)kTileV, total - first);
  if (lane == 0) arrive_expect(bar, (unsigned)nvalid * kRawPitch);
  __syncwarp();
  const uint16_t* x = static_cast<const uint16_t*>(a.x);
  if (a.st == TQ_D && a.tokens >= 32) {
    if (lane == 0) {
      int bh, t;
      split_vec(a, first, bh, t);
      int b = (int)((uint32_t)bh / (uint32_t)a.heads), h = bh - b * a.heads;
      for (int v = 0; v < nvalid;) {
        const int n = min(nvalid - v, a.tokens - t);
        const long long off = (long long)b * a.sb + (long long)h * a.sh + (long long)t * TQ_D;
        bulk_g2s(raw + v * kRawPitch, x + off, (unsigned)n * kRawPitch, bar);
        v += n;
        t = 0;
        if (++h == a.heads) {
          h = 0;
          ++b;
        }
      }
    }
  } else if (a.st == TQ_D) {
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
// The same cell by binary search over the positive boundaries, with the positive boundaries
// and levels in a shared-memory table (tab[0..7] boundaries, tab[8..15] levels): IB − 1
// comparisons instead of 2^(IB−1) − 1 for 3- and 4-bit codes.  Ties go up, as above.
template <int IB>
__device__ __forceinline__ int cell_of_search(float y, const float* tab, float& level) {
  constexpr int h = 1 << (IB - 1);
  const float ay = fabsf(y);
  int cnt = 0;
#pragma unroll
  for (int st = h / 2; st >= 1; st >>= 1)
    if (tab[cnt + st - 1] <= ay) cnt += st;
  const float c = tab[8 + cnt];
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
  // per chunk: its values, max |x| and Σ x² in chains of 8 (four chains run side by side)
  float f[4][8];
  float mx[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
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
    }
    float mh[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) mh[e] = fmaxf(fabsf(f[j][2 * e]), fabsf(f[j][2 * e + 1]));
    mx[j] = fmaxf(fmaxf(mh[0], mh[1]), fmaxf(mh[2], mh[3]));
  }
  float m = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
  const int eb = (int)((__float_as_uint(m) >> 23) & 0xffu);
  s = min(141 - eb, 126);
  const float sc = __uint_as_float((uint32_t)(s + 127) << 23);
  float ss[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    ss[j] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = f[j][2 * e] * sc, x1 = f[j][2 * e + 1] * sc;
      ss[j] = fmaf(x0, x0, ss[j]);
      ss[j] = fmaf(x1, x1, ss[j]);
      const __half2 h2 = __floats2half2_rn(x0, x1);
      hw[j][e] = *reinterpret_cast<const uint32_t*>(&h2);
    }
  }
  float t = (ss[0] + ss[1]) + (ss[2] + ss[3]);
  t += __shfl_xor_sync(0xffffffffu, t, 8);
  t += __shfl_xor_sync(0xffffffffu, t, 16);
  ns = sqrtf(t);
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
                                             const float* tab, uint32_t (&code)[kNib ? 4 : IB]) {
  float rr = 0.f;
  if constexpr (IB == 2 && !kNib) {
    // Two index bits, levels ±c0, ±c1, boundaries 0, ±b.  The decisions are taken on sign
    // bits, which a funnel shift gathers into a word one coordinate per instruction: bit 1 of
    // the cell is "y non-negative" (sign of y clear) and bit 0 is "bit 1 equals |y| > b" (sign
    // of t = b − |y| set); the level is c0 or c1 by the sign of t, carrying the sign of y.
    // Only a y of exactly ±0 or |y| of exactly b (inside the decision's exclusion band) can
    // fall on the other side than the comparison y ≥ boundary would put it.  A zero vector
    // (ysc = 0) takes the upper middle cell outright.
    const float b = lv.b[2];
    const uint32_t c0 = __float_as_uint(lv.c[2]), dc = c0 ^ __float_as_uint(lv.c[3]);
    uint32_t sy = 0, sb = 0;
#pragma unroll
    for (int e = 31; e >= 0; --e) {
      const float y = dv[e] * ysc;
      const float t = b - fabsf(y);
      const uint32_t yb = __float_as_uint(y), tb = __float_as_uint(t);
      sy = __funnelshift_l(yb, sy, 1);
      sb = __funnelshift_l(tb, sb, 1);
      const uint32_t big = (uint32_t)((int32_t)tb >> 31);
      const float level = __uint_as_float((c0 ^ (dc & big)) ^ (yb & 0x80000000u));
      const float rho = y - level;
      rr = fmaf(rho, rho, rr);
      dv[e] = rho * kRhoScale;
    }
    if (!(ysc > 0.f)) sy = sb = 0;
    code[0] = sy ^ sb;
    code[1] = ~sy;
  } else {
#pragma unroll
    for (int k = 0; k < (kNib ? 4 : IB); ++k) code[k] = 0;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float y = dv[e] * ysc;
      float level;
      int q;
      if constexpr (IB >= 3) q = cell_of_search<IB>(y, tab, level);
      else q = cell_of<IB>(y, lv, level);
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
  }
  return rr;
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
// its cache row and slot in the row, or -1 (not stored; a position out of range, or a page
// outside the pool, is flagged)
template <bool kPaged>
__device__ __forceinline__ int dest_slot(const TcArgs& a, const VecDest& d, int r, int nvalid,
                                         long long& row) {
  if (r >= nvalid || d.t >= d.cnt) return -1;
  const int p = d.p0 + d.t;
  if (p < 0 || p >= a.capacity) {
    atomicOr(&g_tq_flags, TQ_FLAG_POS_OVERFLOW);
    return -1;
  }
  if constexpr (!kPaged) {
    row = d.bh;
    return p;
  }
  const int b = (int)((uint32_t)d.bh / (uint32_t)a.heads);
  int slot;
  if (!tq_map_slot(a.map, a.heads, b, d.bh - b * a.heads, p, row, slot)) {
    atomicOr(&g_tq_flags, TQ_FLAG_PAGE);
    return -1;
  }
  return slot;
}

// Converter warp cw: tile j's raw vectors, once in buffer j % NB, become X̂ in place, with
// ‖x‖·2^s and s per vector; then the warp hands the buffer to the issuer.  An 8-vector group's
// canonical image occupies exactly the bytes of its 8 raw rows, so a warp that holds a group's
// raw chunks in registers may overwrite them.  False when the wait gave up.
template <int NB, int kConvWarps>
__device__ __forceinline__ bool convert_tile(const TcArgs& a, int j, long long total,
                                             const long long* s_tile, unsigned char* b,
                                             float* s_ns, signed char* s_exp, uint64_t* bar_x,
                                             uint64_t* bar_a1, int cw, int lane) {
  const int k = j % NB;
  if (!__all_sync(0xffffffffu, tq::mbar_wait(bar_x + k, (j / NB) & 1))) return false;
  const int nvalid = (int)min((long long)kTileV, total - s_tile[k] * kTileV);
  for (int g8 = cw; g8 < kTileV / 8; g8 += kConvWarps) {
    const int v = 8 * g8 + (lane & 7);
    uint32_t w[4][4], hw[4][4];
    load_raw(b, v, v < nvalid, lane, w);
    __syncwarp();   // the group's raw rows are in registers
    float ns;
    int s;
    convert_chunks(w, a.dtype, hw, ns, s);
    store_canon(b, v, lane, hw);
    if (lane < 8) {
      s_ns[k * kTileV + v] = ns;
      s_exp[k * kTileV + v] = (signed char)s;
    }
  }
  async_proxy_fence();   // X̂ (generic writes) → tensor-core reads
  __syncwarp();
  if (lane == 0) tq::mbar_arrive(bar_a1 + k);
  return true;
}

// Index codes of vector r's part (NBLK 32-column blocks of D1 from column d1c)
template <int IB, bool kNib, int NBLK>
__device__ __forceinline__ float epilogue_cells(uint32_t d1c, float ysc, const tq_levels& lv,
                                                const float* tab, float (&dv)[NBLK][32],
                                                uint32_t (&code)[NBLK][kNib ? 4 : IB]) {
  float rr = 0.f;
#pragma unroll
  for (int hb = 0; hb < NBLK; ++hb) {
    tmem_ld32(d1c + 32 * hb, dv[hb]);
    rr += cells_block<IB, kNib>(dv[hb], ysc, lv, tab, code[hb]);
  }
  return rr;
}
// stores of a part's index codes (planes: 4·NBLK bytes of each plane; nibbles: 16·NBLK bytes)
template <int IB, bool kNib, int NBLK, typename RowT>
__device__ __forceinline__ void store_codes(const TcArgs& a, RowT row, int dst, long long slot,
                                            int part, const uint32_t (&code)[NBLK][kNib ? 4 : IB]) {
  if constexpr (kNib) {
    uint4* dp = reinterpret_cast<uint4*>(a.idx + slot * 64 + 16 * NBLK * part);
#pragma unroll
    for (int hb = 0; hb < NBLK; ++hb)
      dp[hb] = make_uint4(code[hb][0], code[hb][1], code[hb][2], code[hb][3]);
  } else {
#pragma unroll
    for (int p = 0; p < IB; ++p) {
      unsigned char* dp =
          a.idx + (((long long)row * IB + p) * a.rowcap + dst) * 16 + 4 * NBLK * part;
      if constexpr (NBLK == 4)
        *reinterpret_cast<uint4*>(dp) = make_uint4(code[0][p], code[1][p], code[2][p], code[3][p]);
      else
        *reinterpret_cast<uint2*>(dp) = make_uint2(code[0][p], code[1][p]);
    }
  }
}

// The quantisers.  One CTA per SM, persistent over the tiles blockIdx.x + j·gridDim.x, with
// warp roles (an MMA issue waits while the tensor core's queue is full, so MMAs come from a warp
// that does nothing else):
//   converter warps  tile j's raw vectors → X̂ in buffer j % NB (in place);
//   issuer warp      the tile copies, GEMM 1 (X̂ · Π̂ᵀ → D1) and for the product code GEMM 2
//                    (ρ̂ · M̂ᵀ → D2, ρ̂ read from TMEM);
//   epilogue warps   MSE code: the index codes and ‖x‖ from D1.  Product code: epilogue 1 (the
//                    index planes, ‖x‖, ρ̂ hi | lo into TMEM, ‖ρ‖) and epilogue 2 (the signs of
//                    D2), in the order epilogue 1 of tile j, epilogue 2 of tile j − 1.
// D1 has two slots, so GEMM 1 of tile j + 2 runs while epilogue 1 of tile j + 1 reads the other
// slot; GEMM 2 of tile j (once the signs of tile j − 1 are read from D2) runs under the cells of
// tile j + 1, whose ρ̂ goes to TMEM once GEMM 2 of tile j has read the previous one.
// Hand-overs are mbarriers: the converters' and epilogues' arrivals (one per warp) and the tensor
// core's commits.  Every barrier's next phase can only complete after each of its waiters has
// passed the previous one (the barriers that would otherwise run two phases ahead of a waiter
// come one per buffer or accumulator slot), so waits on a phase's parity are exact.  kPaged:
// the cache is a page pool, each vector's slot found through the block table.
template <bool kProd, int IB, bool kPaged>
__global__ void __launch_bounds__(Roles<kProd, IB>::kThreads, 1) quantize_tc_kernel(TcArgs a) {
  using L = QL<kProd>;
  using R = Roles<kProd, IB>;
  constexpr int kEpiWarps = R::kEpiWarps, kConvWarps = R::kConvWarps;
  constexpr int NBLK = R::kBlocks;
  constexpr int NB = L::kBufs;
  constexpr bool kNib = !kProd && IB == 4;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* s_ns = reinterpret_cast<float*>(smem + L::ns);
  float* s_rr = reinterpret_cast<float*>(smem + L::rr);
  signed char* s_exp = reinterpret_cast<signed char*>(smem + L::sexp);
  float* s_tab = reinterpret_cast<float*>(smem + L::tab);
  // the tile in each buffer, written by the copy warp before the copy's barrier arrival and
  // read behind the barriers that follow it
  long long* s_tile = reinterpret_cast<long long*>(smem + L::tiles);
  uint64_t* bar_const = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* bar_x = bar_const + 1;          // [NB] raw tile in the buffer (bulk copies)
  uint64_t* bar_a1 = bar_x + NB;            // [NB] X̂ in the buffer (converter warps)
  uint64_t* bar_free = bar_a1 + NB;         // [NB] buffer free: GEMM 1 and the epilogue done
                                            // with its tile (issuer warp)
  uint64_t* bar_g1 = bar_free + NB;         // [2] GEMM 1 into D1[slot] done (tensor-core commit)
  uint64_t* bar_a2 = bar_g1 + 2;            // epilogue (1) done: [2] per D1 slot (MSE), [1]
  uint64_t* bar_a3 = bar_a2 + 1;            // epilogue 2 done (product code)
  uint64_t* bar_g2 = bar_a3 + 1;            // GEMM 2 done (product code)
  uint64_t* bar_rr = bar_g2 + 1;            // part 1's ‖ρ‖² of the tile in place (product code)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_const + L::nbars);
  const long long total = (long long)a.batch * a.heads * a.tokens;
  const long long ntiles = (total + kTileV - 1) / kTileV;
  // The CTA's tiles are the live ones among blockIdx.x + k·gridDim.x; the copy warp walks them in
  // order and records the j-th in s_tile[j % NB] for the other roles.
  auto tile_valid = [&](long long tile) {
    return (int)min((long long)kTileV, total - tile * kTileV);
  };
  auto buffer = [&](int j) { return smem + L::buf + (j % NB) * kImg; };

  if (tid == 0) {
    for (int b = 0; b < L::nbars; ++b) {
      int count = 1;                                                    // copies, commits
      if (b >= 1 + NB && b < 1 + 2 * NB) count = kConvWarps;            // bar_a1
      if (b >= 3 + 3 * NB && b < 5 + 3 * NB) count = kEpiWarps;         // bar_a2, bar_a2/a3
      if (kProd && b == 6 + 3 * NB) count = kEpiWarps / 2;              // bar_rr
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s32(bar_const + b)),
                   "r"(count));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     s32(s_tmem)),
                 "r"(L::tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid >= 32 && tid < 48) {   // the positive boundaries and levels (3- and 4-bit cells)
    constexpr int h = 1 << (IB - 1);
    const int k = tid - 32;
    if (k < 8) s_tab[k] = k < h - 1 ? a.lv.b[h + k] : INFINITY;
    else s_tab[k] = k - 8 < h ? a.lv.c[h + k - 8] : 0.f;
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = *s_tmem;
  // the number of live tiles: every thread tests one tile per round
  int nt = 0;
  const long long mine = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  for (long long k0 = 0; k0 < mine; k0 += blockDim.x) {
    const long long k = k0 + tid;
    nt += __syncthreads_count(k < mine && tile_live(a, blockIdx.x + k * gridDim.x));
  }

  if (warp == R::kCopier) {
    // ================================================================ copy warp
    // the codec's images, the first NB tiles, then tile j + NB into buffer j % NB once the issuer
    // has seen GEMM 1 and the epilogue done with tile j (the barrier's next phase needs the copy
    // issued here)
    bool ok = true;
    uint32_t cbits = 0, cpar = 0;   // buffers with a copy issued; per buffer, copies mod 2
    LiveCursor cur(a, blockIdx.x, gridDim.x, ntiles);
    auto copy_tile = [&](int j) {   // the j-th live tile: the next one on this warp's cursor
      const long long tile = cur.next(a);
      if (lane == 0) s_tile[j % NB] = tile;   // before issue_tile's barrier arrival
      __syncwarp();
      issue_tile(a, tile, total, buffer(j), bar_x + j % NB, lane);
      cbits |= 1u << (j % NB);
      cpar ^= 1u << (j % NB);
    };
    if (nt > 0) {
      if (lane == 0) {
        arrive_expect(bar_const, (kProd ? 4 : 2) * kImg);
        bulk_g2s(smem + L::pi, a.img, (kProd ? 4 : 2) * kImg, bar_const);
      }
      for (int j = 0; j < NB && j < nt; ++j) copy_tile(j);
    }
    for (int j = 0; j + NB < nt && ok; ++j) {
      ok = __all_sync(0xffffffffu, tq::mbar_wait(bar_free + j % NB, (j / NB) & 1));
      if (!ok) break;
      async_proxy_fence();
      copy_tile(j + NB);
    }
    if (!ok) {
      // a bounded wait gave up: report it and let this warp's copies land (bounded)
      if (lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
      for (int b = 0; b < NB; ++b)
        if ((cbits >> b) & 1u) tq::mbar_wait(bar_x + b, ((cpar >> b) & 1u) ^ 1u);
    }
  } else if (warp == R::kIssuer) {
    // ================================================================ issuer warp
    bool ok = true;
    uint64_t* last_bar = nullptr;   // barrier and phase of the last MMA commit
    uint32_t last_par = 0;
    auto wait = [&](uint64_t* bar, uint32_t par) {
      ok = ok && __all_sync(0xffffffffu, tq::mbar_wait(bar, par));
      return ok;
    };
    auto gemm1 = [&](int j) {   // X̂ of tile j · Π̂ᵀ → D1[j & 1]; then its buffer is free
      if (lane == 0) {
        issue_gemm1(tmem + 128 * (j & 1), s32(buffer(j)), s32(smem + L::pi));
        mma_commit(bar_g1 + (j & 1));
      }
      __syncwarp();
      last_bar = bar_g1 + (j & 1);
      last_par = (j >> 1) & 1;
    };
    // tile j's buffer (and its norms) may take tile j + NB: its epilogue (1) has waited for its
    // GEMM 1 and read the norms
    auto release = [&](int j) {
      if (lane == 0) tq::mbar_arrive(bar_free + j % NB);
    };
    if (nt > 0) wait(bar_const, 0);
    if constexpr (kProd) {
      for (int j = 0; j < 2 && j < nt && ok; ++j)
        if (wait(bar_a1 + j, 0)) {
          tc_after();
          gemm1(j);
        }
      for (int j = 0; j < nt && ok; ++j) {
        // epilogue 1 of tile j done: D1[j & 1] read, ρ̂ of tile j in TMEM
        if (!wait(bar_a2, j & 1)) break;
        release(j);
        // the signs of tile j − 1 read from D2
        if (j > 0 && !wait(bar_a3, (j - 1) & 1)) break;
        tc_after();
        if (lane == 0) {
          // D2 = ρ̂hi·M̂hiᵀ + ρ̂hi·M̂loᵀ + ρ̂lo·M̂hiᵀ
          const uint32_t d2 = tmem + kD2Col;
          const uint32_t rh = tmem + kRhoCol, rl = rh + 64;
          const uint32_t smh = s32(smem + L::pi + 2 * kImg), sml = smh + kImg;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t o = ks * 2 * kLBO;
            tq::mma_ts(d2, rh + 8 * ks, sdesc(smh + o), kIdesc, ks > 0 ? 1u : 0u);
            tq::mma_ts(d2, rh + 8 * ks, sdesc(sml + o), kIdesc, 1u);
            tq::mma_ts(d2, rl + 8 * ks, sdesc(smh + o), kIdesc, 1u);
          }
          mma_commit(bar_g2);
        }
        __syncwarp();
        last_bar = bar_g2;
        last_par = j & 1;
        if (j + 2 < nt) {
          if (!wait(bar_a1 + (j + 2) % NB, ((j + 2) / NB) & 1)) break;
          tc_after();
          gemm1(j + 2);   // into D1[j & 1], read by epilogue 1 of tile j
        }
      }
    } else {
      for (int j = 0; j < nt && ok; ++j) {
        if (!wait(bar_a1 + j % NB, (j / NB) & 1)) break;
        // the epilogue of tile j − 2 has read D1[j & 1]
        if (j >= 2) {
          if (!wait(bar_a2 + (j & 1), ((j - 2) >> 1) & 1)) break;
          release(j - 2);
        }
        tc_after();
        gemm1(j);
      }
    }
    if (!ok) {
      // a bounded wait gave up: report it and let this warp's MMAs land (bounded)
      if (lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
      if (last_bar) tq::mbar_wait(last_bar, last_par);
    }
  } else if (warp >= kEpiWarps) {
    // ================================================================ converter warps
    bool ok = true;
    for (int j = 0; j < nt && ok; ++j)
      ok = convert_tile<NB, kConvWarps>(a, j, total, s_tile, buffer(j), s_ns, s_exp, bar_x,
                                        bar_a1, warp - kEpiWarps, lane);
    if (!ok && lane == 0) atomicOr(&g_tq_flags, TQ_FLAG_TIMEOUT);
  } else {
    // ================================================================ epilogue warps
    const int quad = warp & 3, part = warp >> 2;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const int r = 32 * quad + lane;   // this thread's vector
    bool ok = true;
    // vector r of the tile whose signs come next: destination (cache row, slot in the row, and
    // row·rowcap + slot), ‖x‖ (product code); a flat cache's rows (batch·heads + head) fit 32 bits
    using RowT = typename std::conditional<kPaged, long long, int>::type;
    int dst = -1;
    RowT row = 0;
    long long slot = 0;
    float n = 0.f;
    auto begin = [&](int j, uint64_t* g1, uint32_t par) {
      // the converters' norms and the tile index of tile j (an acquire of their arrival, which
      // has completed before GEMM 1 was issued), then its destination, during GEMM 1
      ok = __all_sync(0xffffffffu, tq::mbar_wait(bar_a1 + j % NB, (j / NB) & 1));
      const long long tile = s_tile[j % NB];
      const int nvalid = tile_valid(tile);
      const VecDest vd = vec_dest(a, tile * kTileV, r, nvalid);   // in flight during the wait
      ok = __all_sync(0xffffffffu, ok && tq::mbar_wait(g1, par));
      if (!ok) return;
      tc_after();
      long long rw = 0;
      dst = dest_slot<kPaged>(a, vd, r, nvalid, rw);
      row = (RowT)rw;
      slot = (long long)row * a.rowcap + dst;
    };
    if constexpr (kProd) {
      auto epilogue1 = [&](int j) {
        begin(j, bar_g1 + (j & 1), (j >> 1) & 1);
        if (!ok) return;
        const int k = j % NB;
        const float ns = s_ns[k * kTileV + r];
        n = norm_of(ns, s_exp[k * kTileV + r]);
        float dv[2][32];
        uint32_t code[2][IB];
        const float rr = epilogue_cells<IB, false, 2>(tmem + 128 * (j & 1) + lane_base + 64 * part,
                                                      yscale_of(ns), a.lv, s_tab, dv, code);
        // ρ̂ (scaled residual) as fp16 pairs hi | lo into TMEM (K-major A operand of GEMM 2:
        // column c of a row holds coordinates 2c, 2c + 1), once GEMM 2 of tile j − 1 has read it
        if (j > 0) {
          ok = __all_sync(0xffffffffu, tq::mbar_wait(bar_g2, (j - 1) & 1));
          if (!ok) return;
          tc_after();
        }
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int w = 0; w < 16; ++w) {
            const float v0 = dv[hb][2 * w], v1 = dv[hb][2 * w + 1];
            const __half2 hh = __floats2half2_rn(v0, v1);
            const float2 hf = __half22float2(hh);
            const __half2 ll = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
            hi[w] = *reinterpret_cast<const uint32_t*>(&hh);
            lo[w] = *reinterpret_cast<const uint32_t*>(&ll);
          }
          const uint32_t col = lane_base + 32 * part + 16 * hb;
          tq::tmem_st_32x32b_x16(tmem + kRhoCol + col, hi);
          tq::tmem_st_32x32b_x16(tmem + kRhoCol + 64 + col, lo);
        }
        tq::tmem_wait_st();
        tc_before();
        // the two parts' ‖ρ‖² meet in shared memory; part 0 reads before its hand-over, so that
        // part 1 (which writes the next tile's only after GEMM 2 of this tile, after that
        // hand-over) cannot overwrite it early
        float rt = rr;
        if (part == 1) {
          s_rr[r] = rr;
          __syncwarp();
          if (lane == 0) tq::mbar_arrive(bar_rr);
        } else {
          ok = __all_sync(0xffffffffu, tq::mbar_wait(bar_rr, j & 1));
          if (!ok) return;
          rt += s_rr[r];
        }
        __syncwarp();
        if (lane == 0) tq::mbar_arrive(bar_a2);
        if (dst >= 0) {
          store_codes<IB, false, 2>(a, row, dst, slot, part, code);
          if (part == 0) {
            a.xnorm[slot] = n;
            a.rnorm[slot] = n * sqrtf(rt);
          }
        }
      };
      // signs of tile j (GEMM 2 of tile j wrote D2 after the signs of tile j − 1 were read)
      auto epilogue2 = [&](int j, int jdst, long long jslot, float jn) {
        ok = __all_sync(0xffffffffu, tq::mbar_wait(bar_g2, j & 1));
        if (!ok) return;
        tc_after();
        uint32_t word[2];
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          float dv[32];
          tmem_ld32(tmem + kD2Col + lane_base + 64 * part + 32 * hb, dv);
          // bit e = 1 where z_e is non-negative: the sign bits gathered by funnel shifts and
          // inverted (a z of exactly −0 lies inside the sign decision's exclusion band)
          uint32_t w = 0;
#pragma unroll
          for (int e = 31; e >= 0; --e) w = __funnelshift_l(__float_as_uint(dv[e]), w, 1);
          word[hb] = jn > 0.f ? ~w : 0xffffffffu;   // zero vector: zero residual, all signs +1
        }
        tc_before();   // D2 read before GEMM 2 of tile j + 1
        __syncwarp();
        if (lane == 0) tq::mbar_arrive(bar_a3);
        if (jdst >= 0)
          *reinterpret_cast<uint2*>(a.sgn + jslot * 16 + 8 * part) = make_uint2(word[0], word[1]);
      };
      if (nt > 0) epilogue1(0);
      for (int j = 1; j < nt && ok; ++j) {
        const int pdst = dst;
        const long long pslot = slot;
        const float pn = n;
        epilogue1(j);
        if (!ok) break;
        epilogue2(j - 1, pdst, pslot, pn);
      }
      if (nt > 0 && ok) epilogue2(nt - 1, dst, slot, n);
    } else {
      for (int j = 0; j < nt && ok; ++j) {
        begin(j, bar_g1 + (j & 1), (j >> 1) & 1);
        if (!ok) break;
        const int k = j % NB;
        // the norms are read before the hand-over below frees the buffer slot for tile j + NB
        const float ns = s_ns[k * kTileV + r];
        const float xn = norm_of(ns, s_exp[k * kTileV + r]);
        float dv[NBLK][32];
        uint32_t code[NBLK][kNib ? 4 : IB];
        epilogue_cells<IB, kNib, NBLK>(tmem + 128 * (j & 1) + lane_base + 32 * NBLK * part,
                                       yscale_of(ns), a.lv, s_tab, dv, code);
        tc_before();   // D1 read before GEMM 1 of tile j + 2
        __syncwarp();
        if (lane == 0) tq::mbar_arrive(bar_a2 + (j & 1));
        if (dst >= 0) {
          store_codes<IB, kNib, NBLK>(a, row, dst, slot, part, code);
          if (part == 0) a.xnorm[slot] = xn;
        }
      }
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

template <bool kProd, int IB, bool kPaged>
tq_status launch_tc_layout(const TcArgs& a, int grid, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return TQ_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(quantize_tc_kernel<kProd, IB, kPaged>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             QL<kProd>::total) != cudaSuccess)
      return TQ_ERR_CUDA;
    configured[dev] = true;
  }
  constexpr int threads = Roles<kProd, IB>::kThreads;
  quantize_tc_kernel<kProd, IB, kPaged><<<grid, threads, QL<kProd>::total, stream>>>(a);
  return tq_cuda_status(cudaGetLastError());
}

// Flat caches and page pools are separate instantiations: the flat kernel carries no code of
// the block-table lookup.
template <bool kProd, int IB>
tq_status launch_tc(const TcArgs& a, int grid, cudaStream_t stream) {
  return a.map.table ? launch_tc_layout<kProd, IB, true>(a, grid, stream)
                     : launch_tc_layout<kProd, IB, false>(a, grid, stream);
}

}  // namespace

bool tq_quantize_tc_supported(int dtype) { return dtype == TQ_BF16 || dtype == TQ_F16; }

tq_status tq_launch_quantize_tc(bool prod, const void* x, int dtype, int batch, int heads,
                                int tokens, long long sb, long long sh, long long st,
                                const int* pos, const int* count, uint8_t* idx, uint8_t* sgn,
                                float* xnorm, float* rnorm, int capacity, const tq_rowmap& map,
                                const tq_codec* c, cudaStream_t stream) {
  TcArgs a{};
  a.x = x; a.dtype = dtype; a.batch = batch; a.heads = heads; a.tokens = tokens;
  a.sb = sb; a.sh = sh; a.st = st; a.pos = pos; a.count = count;
  a.idx = idx; a.sgn = sgn; a.xnorm = xnorm; a.rnorm = rnorm; a.capacity = capacity;
  a.map = map; a.rowcap = tq_row_slots(map, capacity);
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
