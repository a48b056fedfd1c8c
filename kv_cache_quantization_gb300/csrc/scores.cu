// Raw estimator scores for every (query, key) pair (QJL deep-dive §五 estimator, §六 the
// "attention_score" read path): score = ‖x‖·⟨Π q, c[idx]⟩ + ‖r‖·√(π/2)/d·⟨S q, 2·sign − 1⟩.
// One CTA per (query, block of 128 keys); the CTA rotates and sketches its query in shared
// memory, then each thread scores one key from its packed planes.
#include "tq_internal.h"

namespace {

constexpr int kThreads = 128;
constexpr float kQjlNum = 1.2533141373155003f;   // √(π/2)

__global__ void __launch_bounds__(kThreads) scores_kernel(const float* q, long long q_stride,
                                                          const float* piT, const float* sT,
                                                          const uint8_t* kidx, const uint8_t* ksgn,
                                                          const float* kxn, const float* krn,
                                                          int kbits, int cap, int n, tq_levels kl,
                                                          float* scores, long long s_stride) {
  __shared__ float qf[TQ_D], qr[TQ_D], qs[TQ_D];
  const int qi = blockIdx.y;
  const int j = threadIdx.x;
  qf[j] = q[(long long)qi * q_stride + j];
  __syncthreads();
  float r = 0.f, s = 0.f;
  for (int k = 0; k < TQ_D; ++k) {
    r = fmaf(__ldg(&piT[k * TQ_D + j]), qf[k], r);
    s = fmaf(__ldg(&sT[k * TQ_D + j]), qf[k], s);
  }
  qr[j] = r;
  qs[j] = s;
  __syncthreads();
  const int t = blockIdx.x * kThreads + threadIdx.x;
  if (t >= n) return;
  uint4 planes[4];
  for (int p = 0; p < kbits; ++p)
    planes[p] = *reinterpret_cast<const uint4*>(kidx + ((long long)p * cap + t) * 16);
  const uint4 sg = *reinterpret_cast<const uint4*>(ksgn + (long long)t * 16);
  float mse = 0.f, qj = 0.f;
  for (int w = 0; w < 4; ++w) {
    uint32_t pw[4];
    for (int p = 0; p < 4; ++p) {
      const uint4 u = planes[p];
      pw[p] = w == 0 ? u.x : w == 1 ? u.y : w == 2 ? u.z : u.w;
    }
    const uint32_t sw = w == 0 ? sg.x : w == 1 ? sg.y : w == 2 ? sg.z : sg.w;
    for (int bit = 0; bit < 32; ++bit) {
      const int jj = w * 32 + bit;
      int idx = 0;
      for (int p = 0; p < kbits; ++p) idx |= ((pw[p] >> bit) & 1) << p;
      mse = fmaf(qr[jj], kl.c[idx], mse);
      qj = ((sw >> bit) & 1) ? qj + qs[jj] : qj - qs[jj];
    }
  }
  scores[(long long)qi * s_stride + t] = kxn[t] * mse + krn[t] * (kQjlNum / TQ_D) * qj;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" tq_status tq_prod_scores(const tq_codec* kc, const float* q, int32_t nq,
                                    int64_t q_stride, tq_prod_cache keys, int32_t capacity,
                                    int32_t n, float* scores, int64_t scores_stride,
                                    tq_stream_t stream) {
  tq_status st = tq_check_codec(kc, TQ_PROD);
  if (st != TQ_OK) return st;
  if (!q || !scores || !keys.idx || !keys.sgn || !keys.xnorm || !keys.rnorm)
    return TQ_ERR_INVALID_ARG;
  if (keys.pages) return TQ_ERR_UNSUPPORTED;   // flat caches only
  if (nq < 0 || nq > 65535 || n < 0 || capacity <= 0 || capacity % TQ_CAPACITY_ALIGN || n > capacity)
    return TQ_ERR_INVALID_ARG;
  if (q_stride < TQ_D || scores_stride < n) return TQ_ERR_INVALID_ARG;
  if (!aligned16(keys.idx) || !aligned16(keys.sgn)) return TQ_ERR_INVALID_ARG;
  if (nq == 0 || n == 0) return TQ_OK;
  dim3 grid((n + kThreads - 1) / kThreads, nq);
  scores_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      q, q_stride, kc->d_piT, kc->d_sT, keys.idx, keys.sgn, keys.xnorm, keys.rnorm, kc->ibits,
      capacity, n, tq_make_levels(kc), scores, scores_stride);
  return tq_cuda_status(cudaGetLastError());
}
