// Host-side part of the library: status strings, the Lloyd-Max codebook solver, the QR
// rotation, and codec creation (device copies of Π, Πᵀ, Sᵀ and M = S Πᵀ).
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <vector>

#include <cuda_fp16.h>

#include "tq_internal.h"
#include "decode_args.h"

extern "C" const char* tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "TQ_OK";
    case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG";
    case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED";
    case TQ_ERR_CUDA: return "TQ_ERR_CUDA";
    case TQ_ERR_TIMEOUT: return "TQ_ERR_TIMEOUT";
    case TQ_ERR_DEVICE_STATUS: return "TQ_ERR_DEVICE_STATUS";
    case TQ_ERR_SCRATCH_LIMIT: return "TQ_ERR_SCRATCH_LIMIT";
  }
  return "TQ_UNKNOWN_STATUS";
}

extern "C" const char* tq_version(void) { return "tq 0.1 (sm_103a)"; }

extern "C" size_t tq_code_bytes(tq_kind kind, int bits) {
  if (kind == TQ_PROD) {
    if (bits < 2 || bits > 5) return 0;
    return (size_t)(bits - 1) * 16 + 16 + 8;
  }
  if (kind == TQ_MSE) {
    if (bits < 1 || bits > 4) return 0;
    return (size_t)bits * 16 + 4;
  }
  return 0;
}

// ----------------------------------------------------------------------------------------
// Lloyd-Max codebook for the sphere-coordinate law (QJL deep-dive, §二 step 2).
//
// The unnormalised density w(t) = (1 − t²)^k, k = (d − 3)/2, has the antiderivative of
// t·w(t) in closed form, −(1 − t²)^(k+1) / (2(k+1)); the cell mass ∫ w is integrated with
// composite Gauss–Legendre quadrature (the normalising constant cancels in the centroid).
// ----------------------------------------------------------------------------------------
namespace {

struct GaussLegendre {
  std::vector<double> x, w;  // nodes / weights on [-1, 1]
  explicit GaussLegendre(int n) : x(n), w(n) {
    const double pi = 3.14159265358979323846;
    for (int i = 0; i < n; ++i) {
      double z = std::cos(pi * (i + 0.75) / (n + 0.5));
      double dp = 0;
      for (int it = 0; it < 100; ++it) {
        double p0 = 1, p1 = z;  // Legendre recurrence
        for (int j = 2; j <= n; ++j) {
          double p2 = ((2.0 * j - 1) * z * p1 - (j - 1.0) * p0) / j;
          p0 = p1;
          p1 = p2;
        }
        dp = n * (z * p1 - p0) / (z * z - 1);
        double dz = p1 / dp;
        z -= dz;
        if (std::fabs(dz) < 1e-16) break;
      }
      x[i] = z;
      w[i] = 2.0 / ((1 - z * z) * dp * dp);
    }
  }
};

double weight_mass(double a, double b, double k, const GaussLegendre& gl) {
  // ∫_a^b (1 − t²)^k dt with 64 equal panels of n-point Gauss–Legendre.
  const int panels = 64;
  double h = (b - a) / panels, total = 0;
  for (int p = 0; p < panels; ++p) {
    double lo = a + p * h, mid = lo + 0.5 * h, acc = 0;
    for (size_t i = 0; i < gl.x.size(); ++i) {
      double t = mid + 0.5 * h * gl.x[i];
      double u = 1 - t * t;
      acc += gl.w[i] * (u > 0 ? std::exp(k * std::log(u)) : 0.0);
    }
    total += 0.5 * h * acc;
  }
  return total;
}

double weight_moment(double a, double b, double k) {
  auto prim = [k](double t) {
    double u = 1 - t * t;
    return u > 0 ? -std::exp((k + 1) * std::log(u)) / (2 * (k + 1)) : 0.0;
  };
  return prim(b) - prim(a);
}

}  // namespace

extern "C" tq_status tq_lloyd_max_codebook(int d, int index_bits, double* centroids) {
  if (!centroids || d < 4 || index_bits < 1 || index_bits > 4) return TQ_ERR_INVALID_ARG;
  const int L = 1 << index_bits;
  const double k = (d - 3) / 2.0;
  GaussLegendre gl(32);
  std::vector<double> c(L), edge(L + 1), next(L);
  for (int i = 0; i < L; ++i) c[i] = (-2.5 + 5.0 * i / (L - 1)) / std::sqrt((double)d);
  for (int it = 0; it < 200000; ++it) {
    edge[0] = -1;
    edge[L] = 1;
    for (int i = 1; i < L; ++i) edge[i] = 0.5 * (c[i - 1] + c[i]);
    double moved = 0;
    for (int i = 0; i < L; ++i) {
      next[i] = weight_moment(edge[i], edge[i + 1], k) / weight_mass(edge[i], edge[i + 1], k, gl);
      moved = std::fmax(moved, std::fabs(next[i] - c[i]));
    }
    c = next;
    if (moved < 1e-15) break;
  }
  // the law is symmetric: make the levels exactly antisymmetric (middle boundary = 0)
  for (int i = 0; i < L; ++i) centroids[i] = 0.5 * (c[i] - c[L - 1 - i]);
  return TQ_OK;
}

// ----------------------------------------------------------------------------------------
// Rotation (QJL deep-dive, §二 step 1: a random orthogonal Π from a QR decomposition).
// Householder QR of G, Q accumulated explicitly, columns negated where R_ii < 0.
// ----------------------------------------------------------------------------------------
extern "C" tq_status tq_rotation_from_gaussian(int d, const double* g, double* pi) {
  if (!g || !pi || d < 1 || d > 4096) return TQ_ERR_INVALID_ARG;
  std::vector<double> a(g, g + (size_t)d * d);   // working copy, becomes R
  std::vector<double> q((size_t)d * d, 0.0);
  for (int i = 0; i < d; ++i) q[(size_t)i * d + i] = 1.0;
  std::vector<double> v(d);
  for (int col = 0; col < d - 1; ++col) {
    double norm = 0;
    for (int r = col; r < d; ++r) norm += a[(size_t)r * d + col] * a[(size_t)r * d + col];
    norm = std::sqrt(norm);
    if (norm == 0) continue;
    double x0 = a[(size_t)col * d + col];
    double alpha = x0 > 0 ? -norm : norm;    // reflect to avoid cancellation
    for (int r = 0; r < d; ++r) v[r] = 0;
    v[col] = x0 - alpha;
    for (int r = col + 1; r < d; ++r) v[r] = a[(size_t)r * d + col];
    double vv = 0;
    for (int r = col; r < d; ++r) vv += v[r] * v[r];
    if (vv == 0) continue;
    // A ← (I − 2 v vᵀ / vᵀv) A
    for (int c2 = col; c2 < d; ++c2) {
      double dot = 0;
      for (int r = col; r < d; ++r) dot += v[r] * a[(size_t)r * d + c2];
      double f = 2 * dot / vv;
      for (int r = col; r < d; ++r) a[(size_t)r * d + c2] -= f * v[r];
    }
    // Q ← Q (I − 2 v vᵀ / vᵀv)
    for (int r = 0; r < d; ++r) {
      double dot = 0;
      for (int c2 = col; c2 < d; ++c2) dot += q[(size_t)r * d + c2] * v[c2];
      double f = 2 * dot / vv;
      for (int c2 = col; c2 < d; ++c2) q[(size_t)r * d + c2] -= f * v[c2];
    }
  }
  for (int c2 = 0; c2 < d; ++c2) {
    double s = a[(size_t)c2 * d + c2] < 0 ? -1.0 : 1.0;
    for (int r = 0; r < d; ++r) pi[(size_t)r * d + c2] = s * q[(size_t)r * d + c2];
  }
  return TQ_OK;
}

// ----------------------------------------------------------------------------------------
// Codec
// ----------------------------------------------------------------------------------------
int tq_num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

tq_status tq_check_codec(const tq_codec* c, tq_kind kind) {
  if (!c) return TQ_ERR_INVALID_ARG;
  if (c->kind != kind) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

tq_status tq_rowmap_of(const tq_pages* pages, int capacity, tq_rowmap* out) {
  if (!out) return TQ_ERR_INVALID_ARG;
  *out = tq_rowmap{nullptr, 0, 0, 0};
  if (!pages) return TQ_OK;
  if (!pages->block_table || pages->max_pages < 1 || pages->num_pages < 1) return TQ_ERR_INVALID_ARG;
  if (pages->page_tokens <= 0 || pages->page_tokens % TQ_CAPACITY_ALIGN) return TQ_ERR_INVALID_ARG;
  if ((long long)pages->max_pages * pages->page_tokens != (long long)capacity) return TQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(pages->block_table) % 4) return TQ_ERR_INVALID_ARG;
  *out = tq_rowmap{pages->block_table, pages->max_pages, pages->page_tokens, pages->num_pages};
  return TQ_OK;
}

tq_levels tq_make_levels(const tq_codec* c) {
  tq_levels l;
  std::memset(&l, 0, sizeof(l));
  l.levels = c->levels;
  for (int i = 0; i < 16; ++i) {
    l.c[i] = c->centroids[i];
    l.b[i] = c->boundaries[i];
  }
  return l;
}

static void free_codec(tq_codec* c) {
  if (!c) return;
  cudaFree(c->d_pi);
  cudaFree(c->d_piT);
  cudaFree(c->d_sT);
  cudaFree(c->d_mT);
  cudaFree(c->d_lut);
  cudaFree(c->d_u);
  cudaFree(c->d_w);
  cudaFree(c->d_img);
  std::free(c);
}

extern "C" tq_status tq_codec_create(int d, tq_kind kind, int bits, const double* pi,
                                     const double* s, const double* centroids, tq_codec** out) {
  if (!out || !pi || !centroids) return TQ_ERR_INVALID_ARG;
  *out = nullptr;
  if (kind != TQ_PROD && kind != TQ_MSE) return TQ_ERR_INVALID_ARG;
  if (d != TQ_HEAD_DIM) return TQ_ERR_UNSUPPORTED;
  int ibits;
  if (kind == TQ_PROD) {
    if (!s) return TQ_ERR_INVALID_ARG;
    if (bits < 2 || bits > 5) return TQ_ERR_UNSUPPORTED;
    ibits = bits - 1;
  } else {
    if (bits < 1 || bits > 4) return TQ_ERR_UNSUPPORTED;
    ibits = bits;
  }
  const int L = 1 << ibits;
  for (int i = 0; i < L; ++i)
    if (!std::isfinite(centroids[i]) || (i > 0 && !(centroids[i] > centroids[i - 1])))
      return TQ_ERR_INVALID_ARG;
  for (int i = 0; i < d * d; ++i)
    if (!std::isfinite(pi[i]) || (s && kind == TQ_PROD && !std::isfinite(s[i])))
      return TQ_ERR_INVALID_ARG;

  tq_codec* c = (tq_codec*)std::calloc(1, sizeof(tq_codec));
  if (!c) return TQ_ERR_CUDA;
  c->d = d;
  c->kind = kind;
  c->bits = bits;
  c->ibits = ibits;
  c->levels = L;
  if (cudaGetDevice(&c->device) != cudaSuccess) {
    std::free(c);
    return TQ_ERR_CUDA;
  }
  for (int i = 0; i < 16; ++i) {
    c->centroids[i] = i < L ? (float)centroids[i] : 0.f;
    c->centroids_d[i] = i < L ? centroids[i] : 0.0;
    c->boundaries[i] = i < L - 1 ? (float)(0.5 * (centroids[i] + centroids[i + 1])) : 0.f;
  }

  c->lut_scale = tq_fp16_friendly_scale(c->centroids, L);
  const size_t n = (size_t)d * d;
  std::vector<float> h_pi(n), h_piT(n), h_sT(n), h_mT(n);
  std::vector<double> h_m(kind == TQ_PROD ? n : 0);
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) {
      h_pi[(size_t)i * d + j] = (float)pi[(size_t)i * d + j];
      h_piT[(size_t)j * d + i] = (float)pi[(size_t)i * d + j];
    }
  if (kind == TQ_PROD) {
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < d; ++j) h_sT[(size_t)j * d + i] = (float)s[(size_t)i * d + j];
    // M = S Πᵀ: M[i][j] = Σ_k S[i][k] Π[j][k]  (double), stored transposed.
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < d; ++j) {
        double acc = 0;
        for (int k = 0; k < d; ++k) acc += s[(size_t)i * d + k] * pi[(size_t)j * d + k];
        h_mT[(size_t)j * d + i] = (float)acc;
        h_m[(size_t)i * d + j] = acc;
      }
  }
  // the digest lets a decode step tell that its key and value codecs share Π (then one CTA
  // appends both with one load of Πᵀ)
  uint64_t dig = 1469598103934665603ull;
  const unsigned char* pb = reinterpret_cast<const unsigned char*>(h_pi.data());
  for (size_t i = 0; i < n * sizeof(float); ++i) dig = (dig ^ pb[i]) * 1099511628211ull;
  c->pi_digest = dig;
  cudaError_t e = cudaSuccess;
  const size_t bytes = n * sizeof(float);
  e = cudaMalloc(&c->d_pi, bytes);
  if (e == cudaSuccess) e = cudaMalloc(&c->d_piT, bytes);
  if (e == cudaSuccess) e = cudaMemcpy(c->d_pi, h_pi.data(), bytes, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(c->d_piT, h_piT.data(), bytes, cudaMemcpyHostToDevice);
  if (kind == TQ_PROD) {
    if (e == cudaSuccess) e = cudaMalloc(&c->d_sT, bytes);
    if (e == cudaSuccess) e = cudaMalloc(&c->d_mT, bytes);
    if (e == cudaSuccess) e = cudaMemcpy(c->d_sT, h_sT.data(), bytes, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(c->d_mT, h_mT.data(), bytes, cudaMemcpyHostToDevice);
  }
  {
    // tensor-core operand images (64·Π, then 8·M for keys), each as an fp16 hi/lo pair
    const bool prod = kind == TQ_PROD;
    const size_t ib = tq_operand_image_bytes(prod);
    std::vector<uint16_t> img(ib / 2);
    tq_build_operand_image(pi, false, img.data());
    if (prod) tq_build_operand_image(h_m.data(), true, img.data() + ib / 4);
    if (e == cudaSuccess) e = cudaMalloc(&c->d_img, ib);
    if (e == cudaSuccess) e = cudaMemcpy(c->d_img, img.data(), ib, cudaMemcpyHostToDevice);
  }
  {
    // column sums Πᵀ·1 and Sᵀ·1, and the largest row norm of S (query normalisation)
    std::vector<float> u(d), w(d, 0.f);
    double smax = 0;
    for (int k = 0; k < d; ++k) {
      double su = 0, sw = 0;
      for (int j = 0; j < d; ++j) {
        su += pi[(size_t)j * d + k];
        if (kind == TQ_PROD) sw += s[(size_t)j * d + k];
      }
      u[k] = (float)su;
      w[k] = (float)sw;
    }
    if (kind == TQ_PROD)
      for (int j = 0; j < d; ++j) {
        double rn = 0;
        for (int k = 0; k < d; ++k) rn += s[(size_t)j * d + k] * s[(size_t)j * d + k];
        smax = std::fmax(smax, std::sqrt(rn));
      }
    c->smax = (float)(smax * (1.0 + 1e-6));
    if (e == cudaSuccess) e = cudaMalloc(&c->d_u, d * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&c->d_w, d * sizeof(float));
    if (e == cudaSuccess) e = cudaMemcpy(c->d_u, u.data(), d * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(c->d_w, w.data(), d * sizeof(float), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess && kind == TQ_MSE && ibits == 4) {
    // decode pair table: key = code of token t | code of token t+1 << 4, entry = the two
    // (scaled) levels as an fp16 pair, replicated 32× so that every lane has its own bank
    std::vector<uint32_t> lut(256 * 32);
    for (int key = 0; key < 256; ++key) {
      const __half lo = __float2half_rn(c->lut_scale * c->centroids[key & 15]);
      const __half hi = __float2half_rn(c->lut_scale * c->centroids[key >> 4]);
      uint16_t ulo, uhi;
      std::memcpy(&ulo, &lo, 2);
      std::memcpy(&uhi, &hi, 2);
      for (int k = 0; k < 32; ++k) lut[key * 32 + k] = (uint32_t)ulo | ((uint32_t)uhi << 16);
    }
    e = cudaMalloc(&c->d_lut, lut.size() * 4);
    if (e == cudaSuccess)
      e = cudaMemcpy(c->d_lut, lut.data(), lut.size() * 4, cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) {
    free_codec(c);
    return TQ_ERR_CUDA;
  }
  *out = c;
  return TQ_OK;
}

extern "C" tq_status tq_codec_destroy(tq_codec* codec) {
  if (!codec) return TQ_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(codec->device);
  free_codec(codec);
  cudaSetDevice(prev);
  return TQ_OK;
}

// Odd-Walsh decomposition of a codec's levels (index bits ≤ 3): the coefficients of the
// levels over the odd monomials of the ±1 bit variables (see decode_args.h).
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

// Scale σ in [1, 2) for which σ·levels are closest to fp16 numbers (worst relative error).
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
