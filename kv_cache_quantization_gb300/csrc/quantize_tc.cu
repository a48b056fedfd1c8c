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
// image brings them in once per CTA.  Raw activations arrive by per-vector bulk copies
// (the TMA engine) one tile ahead of the tile being computed.
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

constexpr int kParts = 2;                      // threads per vector
constexpr int kGT = 128 * kParts;              // threads per group
__host__ __device__ constexpr int groups_of(bool prod) { return prod ? 1 : 2; }
constexpr int kTileV = 128;                    // vectors per tile (MMA M)
constexpr int kImg = 128 * 128 * 2;            // one 128×128 fp16 operand image (32 KB)
constexpr int kLBO = 128;                      // K-adjacent core matrices
constexpr int kSBO = 16 * 128;                 // 8-row groups: 16 core matrices along K
constexpr int kRawPitch = 256;                 // one raw bf16/fp16 vector
constexpr float kPiScale = 64.f, kMScale = 8.f, kRhoScale = 256.f;

// shared-memory map (bytes from the dynamic base): the codec's images, then one area per group
template <bool kProd>
struct QL {
  static constexpr int kGroups = groups_of(kProd);
  static constexpr int pi = 0;                                   // Π̂ hi | lo
  static constexpr int m = 2 * kImg;                             // M̂ hi | lo (prod)
  static constexpr int area = kProd ? 4 * kImg : 2 * kImg;       // group 0's area
  // offsets inside a group's area
  static constexpr int a = 0;                                    // X̂, then ρ̂ hi (prod)
  static constexpr int rho_lo = kImg;                            // ρ̂ lo (prod)
  static constexpr int raw = kProd ? 2 * kImg : kImg;            // raw vectors of the next tile
  static constexpr int norm = raw + kTileV * kRawPitch;          // float ‖x‖ [128]
  static constexpr int ysc = norm + 4 * kTileV;                  // float D1 → y scale [128]
  static constexpr int rr = ysc + 4 * kTileV;                    // float ‖ρ‖² parts [2][128]
  static constexpr int gsize = rr + (kProd ? 2 : 0) * 4 * kTileV;
  // mbarriers: the codec's images, then (raw tile, MMA) per group; then the TMEM slot
  static constexpr int bars = area + kGroups * gsize;
  static constexpr int total = bars + 8 * (1 + 2 * kGroups) + 8;
  static constexpr int tmem_cols = 256;                          // D1 | D2, or D1 per group
};
static_assert(QL<true>::total <= 227 * 1024 && QL<false>::total <= 227 * 1024,
              "shared memory budget");
static_assert(QL<true>::gsize % 1024 == 0 && QL<false>::gsize % 1024 == 0, "area alignment");

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
// barrier of one group (named barrier 1 + group, kGT threads), and its AND-reduction
__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(kGT) : "memory");
}
__device__ __forceinline__ bool group_sync_and(int group, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(1 + group), "r"(kGT)
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
};

// element offset of vector gi of the flattened (batch, head, token) range
__device__ __forceinline__ long long vec_offset(const TcArgs& a, long long gi) {
  const int t = (int)(gi % a.tokens);
  const int bh = (int)(gi / a.tokens);
  return (long long)(bh / a.heads) * a.sb + (long long)(bh % a.heads) * a.sh + (long long)t * a.st;
}

// Warp 0: bring the raw vectors of `tile` into the staging buffer (one bulk copy each).
__device__ __forceinline__ void issue_tile(const TcArgs& a, long long tile, long long total,
                                           unsigned char* raw, uint64_t* bar, int lane) {
  const long long first = tile * kTileV;
  const int nvalid = (int)min((long long)kTileV, total - first);
  if (lane == 0) arrive_expect(bar, (unsigned)nvalid * kRawPitch);
  __syncwarp();
  for (int v = lane; v < nvalid; v += 32)
    bulk_g2s(raw + v * kRawPitch,
             static_cast<const uint16_t*>(a.x) + vec_offset(a, first + v), kRawPitch, bar);
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

template <bool kProd, int IB>
__global__ void __launch_bounds__(kGT * groups_of(kProd), 1) quantize_tc_kernel(TcArgs a) {
  using L = QL<kProd>;
  constexpr int kGroups = L::kGroups;
  constexpr int kBlkPart = 4 / kParts;           // 32-coordinate blocks per thread
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this thread's group, and its warp inside the group
  const int group = warp / (kGT / 32), gw = warp % (kGT / 32);
  unsigned char* area = smem + L::area + group * L::gsize;
  float* s_norm = reinterpret_cast<float*>(area + L::norm);
  float* s_ysc = reinterpret_cast<float*>(area + L::ysc);
  float* s_rr = reinterpret_cast<float*>(area + L::rr);
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
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s32(bar_const)));
    for (int b = 1; b < 1 + 2 * kGroups; ++b)
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
  const uint32_t d1 = tmem + 128 * group, d2 = tmem + 128;   // D2: the product quantiser's
  // TMEM lane quadrant (rows 32·quad..) and coordinate part (blocks kBlkPart·half..) of this
  // warp
  const int quad = gw & 3, half = gw >> 2;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;

  if (gw == 0) {
    if (warp == 0 && lane == 0 && blockIdx.x < ntiles) {
      const unsigned bytes = kProd ? 4 * kImg : 2 * kImg;
      arrive_expect(bar_const, bytes);
      bulk_g2s(smem + L::pi, a.img, 2 * kImg, bar_const);
      if (kProd) bulk_g2s(smem + L::m, static_cast<const unsigned char*>(a.img) + 2 * kImg,
                          2 * kImg, bar_const);
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
    ok = group_sync_and(group, bar_wait(bar_x, px));
    if (!ok) break;
    px ^= 1;
    x_pending = false;
    // ---- raw → X̂ (fp16, per-vector power-of-two scale) and ‖x‖.  Warp w of the group
    // converts vectors 32w/kParts.., eight at a time: lane (i = lane & 7, g = lane >> 3) takes
    // chunks (g + 4j + i) mod 16 of vector i, so that both the staging reads and the canonical
    // writes of a quarter-warp fall in distinct banks.
    {
      const int i = lane & 7, g = lane >> 3;
#pragma unroll 1
      for (int pass = 0; pass < 4 / kParts; ++pass) {
        const int v = (32 / kParts) * gw + 8 * pass + i;
        const bool valid = v < nvalid;
        uint32_t w[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = (g + 4 * j + i) & 15;
          uint4 u = make_uint4(0, 0, 0, 0);
          if (valid) u = *reinterpret_cast<const uint4*>(raw + v * kRawPitch + ch * 16);
          w[j][0] = u.x; w[j][1] = u.y; w[j][2] = u.z; w[j][3] = u.w;
        }
        float f[4][8];
        float mx = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (a.dtype == TQ_BF16) {
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
        // 2^s with max|x|·2^s in [2^14, 2^15); s clamped to [-114, 126].  ‖x‖ is summed
        // over the scaled values too, so it neither overflows nor underflows in fp32
        // anywhere in the bf16 range.
        const int eb = (int)((__float_as_uint(mx) >> 23) & 0xffu);
        const int s = min(141 - eb, 126);
        const float sc = __uint_as_float((uint32_t)(s + 127) << 23);
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = (g + 4 * j + i) & 15;
          uint32_t hw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = f[j][2 * e] * sc, x1 = f[j][2 * e + 1] * sc;
            ss = fmaf(x0, x0, ss);
            ss = fmaf(x1, x1, ss);
            const __half2 h2 = __floats2half2_rn(x0, x1);
            hw[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(area + L::a + canon(v, 8 * ch)) =
              make_uint4(hw[0], hw[1], hw[2], hw[3]);
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 8);
        ss += __shfl_xor_sync(0xffffffffu, ss, 16);
        if (g == 0) {
          const float inv_sc = __uint_as_float((uint32_t)(127 - s) << 23);
          const float ns = sqrtf(ss);     // ‖x‖·2^s
          s_norm[v] = ns * inv_sc;
          s_ysc[v] = ns > 0.f ? 1.f / (kPiScale * ns) : 0.f;
        }
      }
    }
    async_proxy_fence();   // X̂ (generic writes) → tensor-core reads
    tc_before();
    group_sync(group);
    tc_after();
    if (gw == 0) {
      // the staging buffer is free: fetch the group's next tile while this one is computed
      const long long next = tile + tstep;
      if (next < ntiles) {
        async_proxy_fence();
        issue_tile(a, next, total, raw, bar_x, lane);
      }
      // ---- GEMM 1: D1 = X̂ · (Π̂hi + Π̂lo)ᵀ
      if (lane == 0) {
        const uint32_t sa = s32(area + L::a), sp = s32(smem + L::pi);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t ad = sdesc(sa + ks * 2 * kLBO);
          mma_f16(d1, ad, sdesc(sp + ks * 2 * kLBO), ks > 0 ? 1u : 0u);
          mma_f16(d1, ad, sdesc(sp + kImg + ks * 2 * kLBO), 1u);
        }
        mma_commit(bar_mma);
      }
      __syncwarp();
    }
    x_pending = tile + tstep < ntiles;
    mma_pending = true;
    ok = group_sync_and(group, bar_wait(bar_mma, pm));
    if (!ok) break;
    pm ^= 1;
    mma_pending = false;
    tc_after();

    // ---- epilogue 1 (vector r, this thread's coordinate blocks): index planes, residual, ‖ρ‖²
    const int r = 32 * quad + lane;
    const long long gi = first + r;
    int dst = -1;
    long long bh = 0;
    if (r < nvalid) {
      const int t = (int)(gi % a.tokens);
      bh = gi / a.tokens;
      const int b = (int)(bh / a.heads);
      const int cnt = a.count ? a.count[b] : a.tokens;
      if (t < cnt) {
        const int p = (a.pos ? a.pos[b] : 0) + t;
        if (p >= 0 && p < a.capacity) dst = p;
        else atomicOr(&g_tq_flags, TQ_FLAG_POS_OVERFLOW);
      }
    }
    const long long slot = bh * a.capacity + dst;
    const float n = s_norm[r];
    const float ysc = s_ysc[r];
    constexpr bool kNib = !kProd && IB == 4;
    // this thread's words: its nibble words (8 coordinates each), or per plane its
    // 32-coordinate words
    constexpr int kWords = kNib ? 4 * kBlkPart : kBlkPart * IB;
    uint32_t code[kWords];
#pragma unroll
    for (int k = 0; k < kWords; ++k) code[k] = 0;
    float rr = 0.f;
#pragma unroll
    for (int hb = 0; hb < kBlkPart; ++hb) {
      const int blk = kBlkPart * half + hb;
      float dv[32];
      tmem_ld32(d1 + lane_base + 32 * blk, dv);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float y = dv[e] * ysc;
        float level;
        const int q = cell_of<IB>(y, a.lv, level);
        if constexpr (kNib) {
          code[4 * hb + (e >> 3)] |= (uint32_t)q << (4 * (e & 7));
        } else {
#pragma unroll
          for (int p = 0; p < IB; ++p) code[kBlkPart * p + hb] |= (uint32_t)((q >> p) & 1) << e;
        }
        const float rho = y - level;
        rr = fmaf(rho, rho, rr);
        dv[e] = rho * kRhoScale;
      }
      if constexpr (kProd) {
        // ρ̂ as an fp16 pair into the canonical A images (row r, columns 32·blk + 8·c8 + …)
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
          *reinterpret_cast<uint4*>(area + L::a + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(area + L::rho_lo + off) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
    }
    if constexpr (kProd) s_rr[half * kTileV + r] = rr;
    if (dst >= 0) {
      if constexpr (kNib) {
        uint4* dp = reinterpret_cast<uint4*>(a.idx + slot * 64 + 16 * kBlkPart * half);
#pragma unroll
        for (int k = 0; k < kBlkPart; ++k)
          dp[k] = make_uint4(code[4 * k], code[4 * k + 1], code[4 * k + 2], code[4 * k + 3]);
      } else {
#pragma unroll
        for (int p = 0; p < IB; ++p) {
          unsigned char* row = a.idx + ((bh * IB + p) * a.capacity + dst) * 16 + 4 * kBlkPart * half;
          if (kBlkPart == 2) *reinterpret_cast<uint2*>(row) = make_uint2(code[2 * p], code[2 * p + 1]);
          else *reinterpret_cast<uint32_t*>(row) = code[p];
        }
      }
      if (half == 0) a.xnorm[slot] = n;
    }
    if constexpr (kProd) {
      async_proxy_fence();   // ρ̂ (generic writes) → tensor-core reads
      tc_before();
      group_sync(group);
      tc_after();
      // ---- GEMM 2: D2 = ρ̂hi·M̂hiᵀ + ρ̂hi·M̂loᵀ + ρ̂lo·M̂hiᵀ
      if (gw == 0) {
        if (lane == 0) {
          const uint32_t sh = s32(area + L::a), sl = s32(area + L::rho_lo);
          const uint32_t smh = s32(smem + L::m), sml = smh + kImg;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t o = ks * 2 * kLBO;
            mma_f16(d2, sdesc(sh + o), sdesc(smh + o), ks > 0 ? 1u : 0u);
            mma_f16(d2, sdesc(sh + o), sdesc(sml + o), 1u);
            mma_f16(d2, sdesc(sl + o), sdesc(smh + o), 1u);
          }
          mma_commit(bar_mma);
        }
        __syncwarp();
      }
      mma_pending = true;
      ok = group_sync_and(group, bar_wait(bar_mma, pm));
      if (!ok) break;
      pm ^= 1;
      mma_pending = false;
      tc_after();
      uint32_t sw[kBlkPart];
#pragma unroll
      for (int hb = 0; hb < kBlkPart; ++hb) {
        float dv[32];
        tmem_ld32(d2 + lane_base + 32 * (kBlkPart * half + hb), dv);
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 32; ++e) word |= (dv[e] >= 0.f ? 1u : 0u) << e;
        sw[hb] = n > 0.f ? word : 0xffffffffu;   // zero vector: zero residual, all signs +1
      }
      if (dst >= 0) {
        unsigned char* srow = a.sgn + slot * 16 + 4 * kBlkPart * half;
        if (kBlkPart == 2) *reinterpret_cast<uint2*>(srow) = make_uint2(sw[0], sw[kBlkPart - 1]);
        else *reinterpret_cast<uint32_t*>(srow) = sw[0];
        if (half == 0) {
          float rt = 0.f;
#pragma unroll
          for (int pp = 0; pp < kParts; ++pp) rt += s_rr[pp * kTileV + r];
          a.rnorm[slot] = n * sqrtf(rt);
        }
      }
    }
    tc_before();
    group_sync(group);   // D1 / D2 read and X̂ / ρ̂ consumed before the next tile reuses them
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

template <bool kProd, int IB>
tq_status launch_tc(const TcArgs& a, int grid, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return TQ_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(quantize_tc_kernel<kProd, IB>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             QL<kProd>::total) != cudaSuccess)
      return TQ_ERR_CUDA;
    configured[dev] = true;
  }
  quantize_tc_kernel<kProd, IB><<<grid, kGT * groups_of(kProd), QL<kProd>::total, stream>>>(a);
  return tq_cuda_status(cudaGetLastError());
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
