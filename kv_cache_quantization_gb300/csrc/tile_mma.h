// Warp-level pieces shared by the split decode kernels: bit-plane and pair-table value
// operands for mma.sync m16n8k16, and one softmax warp's step over its 32 tokens of a tile
// (online softmax, then values accumulated in the rotated domain).  Internal to the library.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "decode_args.h"
#include "tc_ptx.h"

namespace tq {

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

__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
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
// 2^x by the special-function unit (inputs here are ≤ 0; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Fragment layout of one softmax warp's 32 tokens of a tile: two 16-token fragments T, in each
// rows g and g + 8 (k = 0, 1) of the mma.sync fragment (g = lane / 4), and head columns 2c, 2c + 1
// (h = 0, 1; c = lane % 4).

// Online softmax over the fragments.  lg: base-2 logits; ok: the token is valid; vxn: the 32
// tokens' value norms (index 16T + g + 8k), or null for plain values (norm 1).  Updates the
// running maximum and sums (l: Σ p, lw: Σ p·‖v‖), rescales acc when the maximum grows, and
// returns the value weights w = p·‖v‖ (exactly 0 for invalid tokens).  NH = 2: the lane's two
// columns are two heads; NH = 1: both columns are the same head (its weight split into an fp16
// pair for the value product), so only column 0 is computed and column 1 mirrors it.
template <int NH>
__device__ __forceinline__ void online_softmax(const float (&lg)[2][2][2], const bool (&ok)[2][2],
                                               const float* vxn, float (&acc)[8][4],
                                               float (&m_run)[2], float (&l_run)[2],
                                               float (&lw_run)[2], float (&w)[2][2][2], int lane) {
  const int g = lane >> 2;
  // ---- online softmax over the warp's 32 tokens (per column pair).  The warp-wide maximum
  // is needed only when some logit exceeds the running maximum, which after the first tiles
  // is rare: the common tile skips the shuffles.
  bool grow = false;
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const float m = fmaxf(fmaxf(lg[0][0][h], lg[0][1][h]), fmaxf(lg[1][0][h], lg[1][1][h]));
    grow |= m > m_run[h];
  }
  if (__any_sync(0xffffffffu, grow)) {
    float mt[2], corr[2];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      float m = fmaxf(fmaxf(lg[0][0][h], lg[0][1][h]), fmaxf(lg[1][0][h], lg[1][1][h]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
      mt[h] = fmaxf(m_run[h], m);
      corr[h] = m_run[h] == -INFINITY ? 0.f : ex2(m_run[h] - mt[h]);
      l_run[h] *= corr[h];
      lw_run[h] *= corr[h];
      m_run[h] = mt[h];
    }
    if (NH == 1) corr[1] = corr[0];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc[k][0] *= corr[0];
      acc[k][1] *= corr[1];
      acc[k][2] *= corr[0];
      acc[k][3] *= corr[1];
    }
  }
#pragma unroll
  for (int T = 0; T < 2; ++T)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      // tokens past the sequence (or past the capacity in a short last tile) may hold
      // stale bytes: their weight is exactly zero, never 0 × (stale norm)
      const bool valid = ok[T][k];
      const float vn = vxn ? vxn[16 * T + g + 8 * k] : 1.f;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const float pr = valid ? ex2(lg[T][k][h] - m_run[h]) : 0.f;
        l_run[h] += pr;
        w[T][k][h] = valid ? pr * vn : 0.f;
        lw_run[h] += w[T][k][h];
      }
      if (NH == 1) w[T][k][1] = w[T][k][0];
    }
}

// After the last tile: with NH = 1 the second column's statistics are the first's.
template <int NH>
__device__ __forceinline__ void mirror_stats(float (&m_run)[2], float (&l_run)[2],
                                             float (&lw_run)[2]) {
  if (NH == 1) {
    m_run[1] = m_run[0];
    l_run[1] = l_run[0];
    lw_run[1] = lw_run[0];
  }
}

// Values from codes: acc[coord][column] += Σ_t A[coord][t]·w[t][column].  vrows: the 32 tokens'
// value codes (VB = 4: 64-byte nibble rows; VB < 4: 16-byte rows of plane 0, plane p at
// p·plane_stride); lut_lane: this lane's column of the 4-bit pair table; vcoef: odd-Walsh
// coefficients of the value levels (VB < 4).  Coordinate blocks are in the layout the combine
// step expects (VB = 4: coordinate 16g + 2k8 + hi_row; VB < 4: 16g + pair_lo(2k8 + hi_row)).
template <int VB, bool HILO>
__device__ __forceinline__ void values_from_codes(const float (&w)[2][2][2],
                                                  const unsigned char* vrows, int plane_stride,
                                                  const uint32_t* lut_lane, const float* vcoef,
                                                  float (&acc)[8][4], int lane) {
  constexpr int NVV = VB == 4 ? 0 : num_vplanes(VB);
  const int g = lane >> 2, c = lane & 3;
  const int r8 = lane & 7, m8 = (lane >> 3) & 1;
  // ---- value accumulation: acc[coord][column] += Σ_t A[coord][t] · B[t][column]
#pragma unroll
  for (int T = 0; T < 2; ++T) {
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
      const unsigned char* vb = vrows + (16 * T + 2 * c) * 64 + 8 * g;
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
        ldsm_x2_t(s32(vrows + p * plane_stride + (16 * T + r8 + 8 * m8) * 16),
                  mw[p][0], mw[p][1]);
#pragma unroll
      for (int v = 0; v < NVV; ++v) {
        const float coef = vcoef[v];
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
}

// B fragments (16 tokens × 8 columns) of the weights of fragment T: head columns as they are
// (G > 4), or head c's weight split into an fp16 pair in columns 2c, 2c + 1 (G ≤ 4).
template <bool HILO>
__device__ __forceinline__ void weight_fragments(const float (&w)[2][2][2], int T, uint32_t& bw0,
                                                 uint32_t& bw1) {
  if (HILO) {
    const float h0 = __half2float(__float2half_rn(w[T][0][0]));
    const float h1 = __half2float(__float2half_rn(w[T][1][0]));
    bw0 = movm_t(pack_half2(h0, w[T][0][0] - h0));
    bw1 = movm_t(pack_half2(h1, w[T][1][0] - h1));
  } else {
    bw0 = movm_t(pack_half2(w[T][0][0], w[T][0][1]));
    bw1 = movm_t(pack_half2(w[T][1][0], w[T][1][1]));
  }
}

template <int VB, bool HILO>
__device__ __forceinline__ void softmax_values_step(const float (&lg)[2][2][2], const bool (&ok)[2][2],
                                                    const float* vxn, const unsigned char* vrows,
                                                    int plane_stride, const uint32_t* lut_lane,
                                                    const float* vcoef, float (&acc)[8][4],
                                                    float (&m_run)[2], float (&l_run)[2],
                                                    float (&lw_run)[2], int lane) {
  float w[2][2][2];
  online_softmax<HILO ? 1 : 2>(lg, ok, vxn, acc, m_run, l_run, lw_run, w, lane);
  values_from_codes<VB, HILO>(w, vrows, plane_stride, lut_lane, vcoef, acc, lane);
}

}  // namespace tq
