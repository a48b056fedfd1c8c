// Internal definitions shared by the library's translation units (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tq.h"

#define TQ_D 128
// partial record of one (split, query head): m, l, acc[128], padded to a 16-byte multiple
#define TQ_REC 132

// Codec: immutable after creation.  Small constants travel to kernels by value.
struct tq_codec {
  int d;
  tq_kind kind;
  int bits;        // total bits (prod) or index bits (mse)
  int ibits;       // index bits
  int levels;      // 2^ibits
  int device;
  float* d_pi;     // Π   row-major [d][d]
  float* d_piT;    // Πᵀ  row-major [d][d]  (PT[k][j] = Π[j][k])
  float* d_sT;     // Sᵀ  row-major [d][d]  (prod only)
  float* d_mT;     // Mᵀ  row-major [d][d], M = S Πᵀ (prod only)
  uint32_t* d_lut; // 4-bit MSE only: pair table [256 keys][32 copies] of fp16 level pairs
  float* d_u;      // Πᵀ·1 (Σ_j Π[j][k]): Σ_j (Π q)_j = u·q
  float* d_w;      // Sᵀ·1 (prod only)
  float smax;      // max_j ‖row j of S‖ (prod only): |(S q)_j| ≤ smax·‖q‖
  float centroids[16];
  float boundaries[16];
  double centroids_d[16];
  float lut_scale;   // fp16-friendly scale of the levels (decode pair table)
  void* d_img;       // tensor-core operand images: 64·Π as an fp16 pair, then (prod) 8·M
  uint64_t pi_digest;  // FNV-1a of the float32 Π: equal for codecs that share the rotation
};

// Constants passed by value to kernels.
struct tq_levels {
  float c[16];
  float b[16];
  int levels;
};

// Where a cache keeps a (sequence, head, token): the flat layout (table null) holds row
// b·heads + h of `capacity` slots; a paged pool holds row page·heads + h of page_tokens slots,
// the page from the block table (include/tq.h, tq_pages).  Passed by value to kernels.
struct tq_rowmap {
  const int32_t* table;   // device [batch][max_pages], or null (flat)
  int max_pages, page_tokens, num_pages;
};

// The row map of a cache argument: flat for pages == null, else the block table after the
// checks the header states (capacity = max_pages·page_tokens); TQ_ERR_INVALID_ARG otherwise.
tq_status tq_rowmap_of(const tq_pages* pages, int capacity, tq_rowmap* out);

#ifdef __CUDACC__
// Slots a row holds: capacity (flat) or page_tokens (paged).
__host__ __device__ __forceinline__ int tq_row_slots(const tq_rowmap& m, int capacity) {
  return m.table ? m.page_tokens : capacity;
}
// Row and slot of token t (0 ≤ t < capacity) of sequence b, head h.  False for a paged
// cache whose table entry lies outside [0, num_pages): the caller skips the token and raises
// TQ_FLAG_PAGE.
__device__ __forceinline__ bool tq_map_slot(const tq_rowmap& m, int heads, int b, int h, int t,
                                            long long& row, int& slot) {
  if (!m.table) {
    row = (long long)b * heads + h;
    slot = t;
    return true;
  }
  const int q = t / m.page_tokens;
  const int pg = __ldg(m.table + (long long)b * m.max_pages + q);
  row = (long long)pg * heads + h;
  slot = t - q * m.page_tokens;
  return pg >= 0 && pg < m.num_pages;
}
#endif

// Device status words.  Kernels are compiled without relocatable device code, so every
// translation unit that raises flags owns its word and a host function that reads and
// clears it (on the current device); tq_device_status() ORs them together.
#ifdef __CUDACC__
#define TQ_DEFINE_FLAGS(reader)                                               \
  static __device__ unsigned int g_tq_flags = 0;                              \
  unsigned int reader() {                                                     \
    unsigned int v = 0, z = 0;                                                \
    if (cudaMemcpyFromSymbol(&v, g_tq_flags, sizeof(v)) != cudaSuccess) return ~0u; \
    if (cudaMemcpyToSymbol(g_tq_flags, &z, sizeof(z)) != cudaSuccess) return ~0u;   \
    return v;                                                                 \
  }
#endif
unsigned int tq_take_flags_quantize();
unsigned int tq_take_flags_attention();
unsigned int tq_take_flags_quantize_tc();
unsigned int tq_take_flags_decode_tc();
unsigned int tq_take_flags_decode_asym();
unsigned int tq_take_flags_store();

static inline tq_status tq_cuda_status(cudaError_t e) {
  return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

// Host helpers implemented in host.cpp
tq_status tq_check_codec(const tq_codec* c, tq_kind kind);
int tq_num_sms();

// Launch helpers implemented in the .cu files
tq_levels tq_make_levels(const tq_codec* c);
// Tensor-core quantiser (quantize_tc.cu)
bool tq_quantize_tc_supported(int dtype);
tq_status tq_launch_quantize_tc(bool prod, const void* x, int dtype, int batch, int heads,
                                int tokens, long long sb, long long sh, long long st,
                                const int* pos, const int* count, uint8_t* idx, uint8_t* sgn,
                                float* xnorm, float* rnorm, int capacity, const tq_rowmap& map,
                                const tq_codec* c, cudaStream_t stream);
size_t tq_operand_image_bytes(bool prod);
// FFMA tile quantiser, one CTA per tile of 64 vectors; tiles without a vector to write (count)
// leave at once (quantize.cu).
tq_status tq_launch_quantize_tiles(const tq_codec* c, bool prod, const void* x, tq_dtype dt,
                                   int batch, int heads, int tokens, long long sb, long long sh,
                                   long long st, const int* pos, const int* count, uint8_t* idx,
                                   uint8_t* sgn, float* xnorm, float* rnorm, int capacity,
                                   cudaStream_t stream);
void tq_build_operand_image(const double* mat, bool sketch, uint16_t* img);
float tq_fp16_friendly_scale(const float* levels, int n);
