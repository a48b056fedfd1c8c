// Launch interface of the tensor-core split-decode kernel (decode_tc.cu), used by
// attention.cu.  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "append_args.h"
#include "tq_internal.h"

// A codebook written as a sum over "virtual bit planes": with s_i = 2·bit_i − 1 the
// antisymmetric Lloyd-Max levels expand into odd Walsh monomials,
//   c(idx) = Σ_S a_S Π_{i∈S} s_i = Σ_S (2 a_S)·X_S − Σ_S a_S,
// where X_S is the XOR of the index bits in S (|S| odd).  coef[v] = 2 a_S, cst = Σ a_S.
struct tq_plane_decomp {
  int n;             // number of virtual planes
  float coef[4];
  float cst;
};

struct tq_mma_launch {
  int B, Hq, Hkv, G, cap, nsplit, split_len;
  float scale_log2;            // softmax scale × log2(e)
  const void* q;               // [B][Hq][128] queries (q_dtype)
  int q_dtype;
  const float* piT;            // Πᵀ, Sᵀ of the key codec
  const float* sT;
  const float* u;              // Πᵀ·1 and Sᵀ·1 of the key codec
  const float* w;
  float smax;                  // largest row norm of S
  void* qfrag;                 // workspace: per (b, KV head) query operand images
  const uint8_t* kidx;
  const uint8_t* ksgn;
  const float* kxn;
  const float* krn;
  int kbits;                   // key index bits (1..3)
  tq_plane_decomp kd;
  const uint8_t* vidx;
  const float* vxn;
  tq_rowmap kmap, vmap;        // the caches' row maps (flat, or block tables); cap = slots per
                               // sequence
  int vbits;                   // value bits (1..4)
  tq_plane_decomp vd;          // value decomposition (vbits ≤ 3)
  const uint32_t* lut;         // vbits == 4: 256 × 32 pair table of the value codec (device)
  float vc_unscale;            // 1 / the table's level scale
  const int* seq_lens;
  float* part;                 // [B][Hkv][nsplit][G][130]
  const float* pi;             // Π of the value codec (row-major): out = Πᵀ·acc / L
  const float* vpiT;           // Πᵀ of the value codec (row-major)
  void* out;                   // [B][Hq][128]
  int out_dtype;
  int* counters;               // [B][Hkv] split tickets (cleared by the operand kernel)
  int max_len;                 // longest sequence (tokens) of the call
  float s_idx, s_sgn;          // power-of-two scales of the e4m3 query operand
  // attended tokens of batch b: seq_lens[b] + len_add; the last `fresh` of them may be written
  // by the programmatic-launch primary, so the split kernel reads them only after its wait
  int len_add, fresh;
  // query rows per sequence: row b attends cache row b / qps (1 for decode; a prefill chunk's
  // length for tq_prefill_attention), and with causal = 1 row b also its chunk's first
  // b % qps + 1 tokens (appended to the cache after the sequence's seq_lens tokens)
  int qps, causal;
  // decode step with the appends in the prologue kernel: the step's new key and value,
  // appended at seq_lens[b]
  tq::AppendKV app;
};

// Odd-Walsh decomposition of a codec's levels (index bits ≤ 3).
tq_plane_decomp tq_decompose_levels(const tq_codec* c);
// Tensor-core (tcgen05) split decode with in-kernel query operand and last-CTA merge.
bool tq_tc_decode_supported(int kbits, int vbits, int G, int nsplit);
tq_status tq_launch_decode_tc(const tq_mma_launch& a, cudaStream_t stream);
// The same after a prologue kernel that appends the step's new key and value and builds the
// query operand in one launch.
tq_status tq_launch_decode_step_tc(const tq_mma_launch& a, cudaStream_t stream);
// Whether that prologue, with `appends` append CTAs per (batch, KV head), fits in one wave of
// CTAs (else the appends run as their own launch).
bool tq_step_prologue_fits(int batch, int kv_heads, int appends);
// The appends of a decode step as one launch (quantize.cu), a programmatic-launch secondary.
tq_status tq_launch_append_kv(const tq::AppendKV& a, int batch, cudaStream_t stream);
// Workspace bytes per (batch, KV head) for its query operand images.
size_t tq_tc_frag_bytes_max();
// Power-of-two scales of the e4m3 query operand for a key codec's decomposition.
void tq_tc_operand_scales(const tq_plane_decomp& kd, float* s_idx, float* s_sgn);

// Launch interface of the asymmetric split-decode kernel (decode_asym.cu): FP16 keys,
// MSE-coded values and an FP16 tail; one record per (batch, KV head, split) in the layout of
// the CUDA-core path's merge kernel, which runs after it.
struct tq_asym_launch {
  // TMA descriptors (128-byte swizzle, boxes of 64 columns × 128 rows) of the FP16 keys
  // [B·Hkv·cap][128] and of the tail's keys and values [B·Hkv·tail_cap][128]
  CUtensorMap kmap, ktmap, vtmap;
  int B, Hq, Hkv, G, cap, tail_cap;
  int nsplit_main, nsplit, split_len, tail_split;
  float scale_log2;            // softmax scale × log2(e)
  const void* q;               // [B][Hq][128] queries (q_dtype)
  int q_dtype;
  const __half* kf16;          // [B][Hkv][cap][128]
  const __half* ktail;         // [B][Hkv][tail_cap][128]
  const __half* vtail;
  const int* tail_lens;
  const uint8_t* vidx;
  const float* vxn;
  int vbits;
  tq_plane_decomp vd;          // value decomposition (vbits ≤ 3)
  const uint32_t* lut;         // vbits == 4: pair table of the value codec (device)
  float vc_unscale;            // 1 / the table's level scale
  const int* seq_lens;
  float* part;                 // [B][Hkv][nsplit][G][TQ_REC]
};

bool tq_asym_tc_supported(int vbits, int G, int split_len, int tail_split);
// TMA descriptor of an FP16 row-major matrix [rows][128] for the asymmetric kernel.
tq_status tq_asym_encode_rows(CUtensorMap* map, const void* base, long long rows);
tq_status tq_launch_decode_asym_tc(const tq_asym_launch& a, cudaStream_t stream);
