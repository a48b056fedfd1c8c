// Quality of attention on compressed keys: softmax KL divergence and top-1 agreement between
// the attention weights of exact keys and of the key estimator, per query.
//
// The MLX-port article ("对称 vs 非对称", and its KLD / Top-1 measurement notes) compares the
// model's output distribution with and without compression by KL divergence and top-1
// agreement.  Without models, the same two statistics are taken here at the attention level:
// for a query q, p = softmax(scale·⟨q, k_t⟩) over exact keys and p̂ = softmax(scale·ŝ_t) over
// the estimator scores ŝ_t of the compressed keys (QJL deep-dive §五), KL(p ‖ p̂) =
// Σ_t p_t (log p_t − log p̂_t), and whether argmax p = argmax p̂.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "tq_internal.h"

namespace {

constexpr int kKeys = 128;   // keys a CTA of the exact-score kernel takes

__device__ __forceinline__ float key_elem(const void* k, int dtype, long long i) {
  if (dtype == TQ_F32) return static_cast<const float*>(k)[i];
  const uint16_t u = static_cast<const uint16_t*>(k)[i];
  if (dtype == TQ_BF16) return __uint_as_float((uint32_t)u << 16);
  return __half2float(__ushort_as_half(u));
}

// S[i][t] = ⟨q_i, k_t⟩ (fp32).  Grid (ceil(n / 128), nq), one thread per key: the query row in
// shared memory, the key row read once per query.
__global__ void __launch_bounds__(kKeys) exact_scores_kernel(const float* q, const void* k,
                                                             int dtype, int n, float* s) {
  __shared__ float qs[TQ_D];
  const int i = blockIdx.y;
  qs[threadIdx.x] = q[(long long)i * TQ_D + threadIdx.x];
  __syncthreads();
  const int t = blockIdx.x * kKeys + threadIdx.x;
  if (t >= n) return;
  float acc = 0.f;
  for (int j = 0; j < TQ_D; ++j) acc = fmaf(qs[j], key_elem(k, dtype, (long long)t * TQ_D + j), acc);
  s[(long long)i * n + t] = acc;
}

// One CTA per query: maxima and their first positions, the two partition functions and
// Σ e^{a_t − M_a}·(a_t − b_t), with a = scale·exact, b = scale·estimated scores;
// KL = that sum / Z_a − (M_a + log Z_a) + (M_b + log Z_b).
constexpr int kRed = 256;
__global__ void __launch_bounds__(kRed) quality_kernel(const float* se, const float* sc, int n,
                                                       float scale, float* kl, int* top_e,
                                                       int* top_c) {
  __shared__ float r0[kRed], r1[kRed], r2[kRed];
  __shared__ int i0[kRed], i1[kRed];
  const int i = blockIdx.x, tid = threadIdx.x;
  const float* a = se + (long long)i * n;
  const float* b = sc + (long long)i * n;
  float ma = -INFINITY, mb = -INFINITY;
  int ia = n, ib = n;
  for (int t = tid; t < n; t += kRed) {
    const float x = scale * a[t], y = scale * b[t];
    if (x > ma) { ma = x; ia = t; }
    if (y > mb) { mb = y; ib = t; }
  }
  r0[tid] = ma; r1[tid] = mb; i0[tid] = ia; i1[tid] = ib;
  __syncthreads();
  for (int w = kRed / 2; w > 0; w >>= 1) {
    if (tid < w) {
      if (r0[tid + w] > r0[tid] || (r0[tid + w] == r0[tid] && i0[tid + w] < i0[tid])) {
        r0[tid] = r0[tid + w]; i0[tid] = i0[tid + w];
      }
      if (r1[tid + w] > r1[tid] || (r1[tid + w] == r1[tid] && i1[tid + w] < i1[tid])) {
        r1[tid] = r1[tid + w]; i1[tid] = i1[tid + w];
      }
    }
    __syncthreads();
  }
  const float Ma = r0[0], Mb = r1[0];
  if (tid == 0) { top_e[i] = i0[0]; top_c[i] = i1[0]; }
  __syncthreads();
  float za = 0.f, zb = 0.f, cross = 0.f;
  for (int t = tid; t < n; t += kRed) {
    const float x = scale * a[t], y = scale * b[t];
    const float ea = expf(x - Ma);
    za += ea;
    zb += expf(y - Mb);
    cross = fmaf(ea, x - y, cross);
  }
  r0[tid] = za; r1[tid] = zb; r2[tid] = cross;
  __syncthreads();
  for (int w = kRed / 2; w > 0; w >>= 1) {
    if (tid < w) { r0[tid] += r0[tid + w]; r1[tid] += r1[tid + w]; r2[tid] += r2[tid + w]; }
    __syncthreads();
  }
  if (tid == 0) kl[i] = r2[0] / r0[0] - (Ma + logf(r0[0])) + (Mb + logf(r1[0]));
}

}  // namespace

extern "C" size_t tq_attention_quality_scratch_bytes(int32_t nq, int32_t n) {
  if (nq <= 0 || n <= 0) return 0;
  return 2 * (size_t)nq * n * sizeof(float);
}

extern "C" tq_status tq_attention_quality(const tq_codec* kc, const float* q, int32_t nq,
                                          const void* k, tq_dtype k_dtype, tq_prod_cache codes,
                                          int32_t capacity, int32_t n, float softmax_scale,
                                          void* scratch, size_t scratch_bytes, float* kl,
                                          int32_t* top1_exact, int32_t* top1_comp,
                                          tq_stream_t stream_) {
  tq_status st = tq_check_codec(kc, TQ_PROD);
  if (st != TQ_OK) return st;
  if (!q || !k || !scratch || !kl || !top1_exact || !top1_comp) return TQ_ERR_INVALID_ARG;
  if (codes.pages) return TQ_ERR_UNSUPPORTED;   // flat caches only
  if (k_dtype != TQ_F32 && k_dtype != TQ_F16 && k_dtype != TQ_BF16) return TQ_ERR_UNSUPPORTED;
  if (nq <= 0 || nq > 65535 || n <= 0 || n > capacity) return TQ_ERR_INVALID_ARG;
  if (scratch_bytes < tq_attention_quality_scratch_bytes(nq, n)) return TQ_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)TQ_D);
  float* se = static_cast<float*>(scratch);
  float* sc = se + (size_t)nq * n;
  exact_scores_kernel<<<dim3((n + kKeys - 1) / kKeys, nq), kKeys, 0, stream>>>(q, k, k_dtype, n, se);
  if ((st = tq_cuda_status(cudaGetLastError())) != TQ_OK) return st;
  st = tq_prod_scores(kc, q, nq, TQ_D, codes, capacity, n, sc, n, stream_);
  if (st != TQ_OK) return st;
  quality_kernel<<<nq, kRed, 0, stream>>>(se, sc, n, scale, kl, top1_exact, top1_comp);
  return tq_cuda_status(cudaGetLastError());
}
