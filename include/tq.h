/*
 * tq.h — C ABI of the TurboQuant KV-cache library for GB300 (sm_103a).
 *
 * Keys are coded with the TurboQuant product quantiser and values with the MSE-only
 * quantiser; decode attention reads the packed codes directly.  Sources, by page:
 *
 *   [QJL]  "TurboQuant QJL投影深度剖析：揭秘注意力分数背后的无偏内积估计器原理"
 *          (bjdmk.com.cn): §二 the three-stage compression pipeline, §四 the QJL sign
 *          sketch and its constant √(π/2)/d, §五 the combined unbiased estimator and the
 *          packed (indices, sign bytes, ‖r‖, ‖x‖) record, §六 the read path (forward-rotated
 *          and pre-sketched query, fused online-softmax decode attention), per-layer seeds.
 *   [MLX]  the MLX-port article (cf-1.com): "背景" K = full TurboQuant, V = MSE-only;
 *          "对称 vs 非对称" the asymmetric K = FP16 / V = turbo mode; quick start
 *          (`key_bits=0`, `min_compress_tokens`).
 *
 * Conventions shared by every call
 *   - head_dim d must be 128 (TQ_HEAD_DIM); anything else returns TQ_ERR_UNSUPPORTED.
 *   - Pointers named "device" must be device (or managed) memory on the current device;
 *     pointers named "host" are host memory.  The library never frees caller memory and
 *     keeps no pointer to it after a call returns.
 *   - Every device call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Arguments are validated on the host before any launch; a failed
 *     validation returns an error code and launches nothing.  Launch failures return
 *     TQ_ERR_CUDA.  Conditions only visible on the device (a position or length beyond the
 *     capacity) make the kernel skip the offending tokens and raise a bit in a per-device
 *     status word that tq_device_status() reads.
 *   - Hot calls (quantise, scores, decode) allocate nothing: decode attention takes a
 *     caller-owned workspace sized by tq_decode_workspace_bytes().
 *
 * Packed code layout (one KV head, one token, d = 128)
 *   A 16-byte plane holds one bit per coordinate: coordinate j is bit (j % 8) of byte j / 8.
 *   - Product code of a key, b total bits (b ≥ 2): (b−1) index planes (plane p = bit p of
 *     each coordinate's Lloyd-Max index), one sign plane (bit = 1 iff (S r)_j ≥ 0),
 *     ‖x‖ (float) and ‖r‖ (float).  [QJL] §二 step 3 ("d/8 bytes"), §五.
 *   - MSE code of a value, B bits: B index planes, except B = 4 which is nibble-packed
 *     (byte k = idx(2k) | idx(2k+1) << 4, 64 bytes), and ‖x‖ (float).
 *   Cache arrays are plane-major per (batch, head) so that a run of tokens of one plane is
 *   contiguous:
 *     prod idx  : uint8 [batch][heads][b−1][capacity][16]
 *     prod sgn  : uint8 [batch][heads][capacity][16]
 *     prod xnorm, rnorm : float [batch][heads][capacity]
 *     mse idx   : uint8 [batch][heads][B][capacity][16]   (B ≤ 3)
 *                 uint8 [batch][heads][capacity][64]      (B = 4)
 *     mse xnorm : float [batch][heads][capacity]
 *   capacity must be a positive multiple of 64 and every array 16-byte aligned.
 *   Paged caches (tq_pages below) keep the same layout with pages in place of sequences.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_HEAD_DIM 128
#define TQ_MAX_GROUP 8          /* maximum query heads per KV head (GQA group) */
#define TQ_CAPACITY_ALIGN 64

/* A cudaStream_t without requiring the CUDA headers. */
typedef struct CUstream_st* tq_stream_t;

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,   /* null pointer, bad size, stride or alignment */
  TQ_ERR_UNSUPPORTED = 2,   /* valid but not built: d != 128, bit width, dtype, group > 8 */
  TQ_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  TQ_ERR_TIMEOUT = 4,       /* a bounded device-side wait gave up */
  TQ_ERR_DEVICE_STATUS = 5, /* the device status word reports skipped tokens */
  TQ_ERR_SCRATCH_LIMIT = 6  /* the call needs more scratch than the library's static array */
} tq_status;

typedef enum { TQ_F32 = 0, TQ_F16 = 1, TQ_BF16 = 2 } tq_dtype;
typedef enum { TQ_PROD = 0, TQ_MSE = 1 } tq_kind;

/* Human-readable name of a status code (static string, never NULL). */
const char* tq_status_string(tq_status s);

/* ------------------------------------------------------------------ host-side constants */

/* Lloyd-Max codebook for one coordinate of a uniform point on the unit sphere S^{d−1},
 * density ∝ (1 − t²)^((d−3)/2) on [−1, 1] ([QJL] §二 step 2: continuous 1-D k-means for
 * the rotated-coordinate law).  Writes 2^index_bits centroids, ascending, unit-sphere
 * scale, to `centroids` (host, caller-owned).  Decision boundaries are the midpoints.
 * index_bits in 1..4.  Pure host code; needs no GPU. */
tq_status tq_lloyd_max_codebook(int d, int index_bits, double* centroids);

/* Random rotation from a Gaussian matrix ([QJL] §二 step 1: rotation by QR): Π = Q of
 * G = Q R with diag(R) > 0.  `g` and `pi` are host, row-major d×d, caller-owned;
 * y = Π x.  Pure host code; needs no GPU. */
tq_status tq_rotation_from_gaussian(int d, const double* g, double* pi);

/* ------------------------------------------------------------------ codec */

typedef struct tq_codec tq_codec;

/* Creates an immutable codec on the current device.
 *   kind = TQ_PROD: keys; `bits` = total bits per coordinate b in 2..5 (b−1 index bits plus
 *          one QJL sign bit, [QJL] §二 "(b−1) + 1"); needs `s`.
 *   kind = TQ_MSE : values; `bits` = index bits B in 1..4; `s` may be NULL.
 *   pi        : host, d×d row-major rotation Π (float64), copied.
 *   s         : host, d×d row-major Gaussian sketch S (float64), copied; m = d rows.
 *   centroids : host, the 2^(index bits) ascending Lloyd-Max levels (float64), copied.
 * The codec owns device copies of Π, Πᵀ, Sᵀ and M = S Πᵀ (float32) and is safe to use
 * from several streams at once.  Allocates device memory (not a hot call). */
tq_status tq_codec_create(int d, tq_kind kind, int bits, const double* pi, const double* s,
                          const double* centroids, tq_codec** out);

/* Frees a codec (NULL is a no-op).  The caller must ensure no work using it is pending. */
tq_status tq_codec_destroy(tq_codec* codec);

/* ------------------------------------------------------------------ caches */

/* A paged cache: the codes of a sequence live in fixed-size pages of a shared pool instead of
 * one span of `capacity` slots per (sequence, head), so that sequences can grow by whole pages
 * taken from a free list ([QJL] §六: the store appends in chunks; this block table is this
 * library's form of it).  The pool has the flat layout above with `num_pages` in place of
 * batch and `page_tokens` in place of capacity: page q holds, for each head h, the
 * page_tokens slots of row q·heads + h.  Token t of sequence b is slot t % page_tokens of
 * page block_table[b·max_pages + t / page_tokens]; the sequence's capacity is
 * max_pages·page_tokens, which is what the calls' `capacity` argument must be.  A table entry
 * read for a token that is written or attended and lies outside [0, num_pages) makes the
 * kernel skip that token's page and raise TQ_FLAG_PAGE (the decode output of that row is then
 * undefined).  Entries for pages past a sequence's tokens are never read.  Page sizes of 256
 * tokens or more keep the decode's copies per 256-token stage at one or two per array. */
typedef struct {
  const int32_t* block_table;  /* device, int32 [batch][max_pages] */
  int32_t max_pages;           /* entries per sequence, ≥ 1 */
  int32_t page_tokens;         /* slots per page, a positive multiple of 64 */
  int32_t num_pages;           /* pages in the pool, ≥ 1 */
} tq_pages;

typedef struct {
  uint8_t* idx;    /* device, [batch][heads][b−1][capacity][16] */
  uint8_t* sgn;    /* device, [batch][heads][capacity][16] */
  float* xnorm;    /* device, [batch][heads][capacity] */
  float* rnorm;    /* device, [batch][heads][capacity] */
  /* host, NULL for the flat layout; else the pool's block table (read when a call is made:
   * the struct may be reused or freed after the call returns, the table it points to may not
   * change until the work has run).  Taken by tq_quantize_prod / tq_quantize_mse and by
   * tq_decode_attention, its no-alloc form, tq_decode_step and tq_prefill_attention where
   * they decode on the tensor cores (keys of 2 to 4 bits; 5-bit keys return
   * TQ_ERR_UNSUPPORTED); the other calls take flat caches only (TQ_ERR_UNSUPPORTED). */
  const tq_pages* pages;
} tq_prod_cache;

typedef struct {
  uint8_t* idx;    /* device, planes [batch][heads][B][capacity][16] or nibbles [..][capacity][64] */
  float* xnorm;    /* device, [batch][heads][capacity] */
  const tq_pages* pages;   /* as in tq_prod_cache */
} tq_mse_cache;

/* Bytes of packed codes per token per head (norms included): prod b bits → (b−1)·16+16+8;
 * MSE B bits → B·16+4.  Returns 0 for unsupported widths. */
size_t tq_code_bytes(tq_kind kind, int bits);

/* ------------------------------------------------------------------ quantisation */

/* Quantises keys x with the product quantiser and writes the codes into `cache`
 * ([QJL] §二 steps 1–3, §五 quantize()).
 *   x        : device, elements of `x_dtype` (F32/F16/BF16); vector (b, h, t) starts at
 *              x + b*stride_b + h*stride_h + t*stride_t (strides in elements, ≥ 0) and its
 *              d = 128 coordinates are contiguous.
 *   batch, heads, tokens : x holds tokens t < tokens for every (b, h).
 *   pos      : device int32[batch] or NULL (= 0): cache position of token 0 of batch b.
 *   count    : device int32[batch] or NULL (= tokens): tokens of batch b to write (≤ tokens).
 *   cache, capacity : destination cache of shape [batch][heads][capacity]; tokens landing
 *              at or beyond `capacity` are skipped and flagged in the device status word.
 * Appending one decode token per sequence is tokens = 1 with pos = current lengths. */
tq_status tq_quantize_prod(const tq_codec* kc, const void* x, tq_dtype x_dtype, int32_t batch,
                           int32_t heads, int32_t tokens, int64_t stride_b, int64_t stride_h,
                           int64_t stride_t, const int32_t* pos, const int32_t* count,
                           tq_prod_cache cache, int32_t capacity, tq_stream_t stream);

/* Same for values with the MSE-only quantiser (Algorithm 1: rotation + Lloyd-Max index +
 * ‖x‖), [MLX] "背景". */
tq_status tq_quantize_mse(const tq_codec* vc, const void* x, tq_dtype x_dtype, int32_t batch,
                          int32_t heads, int32_t tokens, int64_t stride_b, int64_t stride_h,
                          int64_t stride_t, const int32_t* pos, const int32_t* count,
                          tq_mse_cache cache, int32_t capacity, tq_stream_t stream);

/* ------------------------------------------------------------------ scores */

/* Raw estimator ⟨q, k⟩ ≈ ‖x‖·⟨Π q, c[idx]⟩ + ‖r‖·√(π/2)/d·⟨S q, 2·sign − 1⟩ for every
 * query and key, without 1/√d ([QJL] §五 estimator, §六 "attention_score" path).
 *   q      : device float32, nq rows with row stride q_stride (elements).
 *   keys   : a prod cache with batch = heads = 1 and the given capacity; keys t < n.
 *   scores : device float32 [nq][scores_stride], row i column t = score(q_i, k_t). */
tq_status tq_prod_scores(const tq_codec* kc, const float* q, int32_t nq, int64_t q_stride,
                         tq_prod_cache keys, int32_t capacity, int32_t n, float* scores,
                         int64_t scores_stride, tq_stream_t stream);

/* ------------------------------------------------------------------ quality report */

/* Scratch bytes tq_attention_quality needs (0 if nq ≤ 0 or n ≤ 0). */
size_t tq_attention_quality_scratch_bytes(int32_t nq, int32_t n);

/* How far attention on compressed keys is from attention on the exact keys, per query: the
 * KL divergence KL(p ‖ p̂) of p = softmax(scale·⟨q_i, k_t⟩) over the exact keys and p̂ =
 * softmax(scale·ŝ_t) over the estimator scores of their product codes ([QJL] §五), and the
 * positions of both maxima (top-1 agreement where they are equal).  The attention-level
 * counterpart of [MLX] "对称 vs 非对称"'s KLD / Top-1 comparison.
 *   q       : device float32 [nq][128].
 *   k       : device [n][128] of k_dtype (F32, F16 or BF16), the exact keys.
 *   codes   : the keys' product codes, a cache with batch = heads = 1 and this capacity (n ≤
 *             capacity).
 *   softmax_scale : ≤ 0 selects 1/√128.
 *   scratch : device, ≥ tq_attention_quality_scratch_bytes(nq, n) bytes.
 *   kl      : device float32 [nq]; top1_exact, top1_comp : device int32 [nq] (first position of
 *             the maximum). */
tq_status tq_attention_quality(const tq_codec* kc, const float* q, int32_t nq, const void* k,
                               tq_dtype k_dtype, tq_prod_cache codes, int32_t capacity, int32_t n,
                               float softmax_scale, void* scratch, size_t scratch_bytes, float* kl,
                               int32_t* top1_exact, int32_t* top1_comp, tq_stream_t stream);

/* ------------------------------------------------------------------ decode attention */

typedef struct {
  int32_t batch;          /* B */
  int32_t q_heads;        /* Hq */
  int32_t kv_heads;       /* Hkv; Hq % Hkv == 0 and Hq / Hkv ≤ TQ_MAX_GROUP */
  int32_t head_dim;       /* must be 128 */
  int32_t capacity;       /* cache capacity per (b, kv head), multiple of 64 */
  int32_t max_seq_len;    /* upper bound of seq_lens[b] (≤ capacity); sizes the grid */
  int32_t tail_capacity;  /* asymmetric call: FP16 tail capacity per (b, kv head); else 0 */
  float softmax_scale;    /* ≤ 0 selects 1/√head_dim */
  tq_dtype q_dtype;       /* F32, F16 or BF16 */
  tq_dtype out_dtype;     /* F32, F16 or BF16 */
} tq_attn_desc;

/* Workspace bytes needed by tq_decode_attention / tq_decode_attention_asym for `desc`
 * (0 if desc is invalid).  Depends on the device's SM count (current device). */
size_t tq_decode_workspace_bytes(const tq_attn_desc* desc);

/* One decode step of attention on the compressed cache ([QJL] §六: forward-rotated and
 * pre-sketched query, scores on the packed bits, one online softmax; values accumulated
 * in the rotated domain and rotated back once).  Query head h reads KV head h / G.
 *   q        : device [batch][q_heads][128] of desc->q_dtype.
 *   k, v     : caches of shape [batch][kv_heads][capacity] coded by kc (prod) and vc (MSE).
 *   seq_lens : device int32[batch]; tokens t < seq_lens[b] are attended (clamped to
 *              capacity, flagged if larger).  A zero length gives a zero output row.
 *   out      : device [batch][q_heads][128] of desc->out_dtype.
 *   workspace: device, ≥ tq_decode_workspace_bytes(desc) bytes, 256-byte aligned, scratch
 *              owned by the caller.  It needs no initialisation: the call clears the
 *              per-(batch, KV head) split tickets it keeps there at its start, so one
 *              workspace may serve calls with different descriptors and asymmetric calls in
 *              turn.  Calls that share a workspace must be serialised on one stream. */
tq_status tq_decode_attention(const tq_attn_desc* desc, const tq_codec* kc, const tq_codec* vc,
                              const void* q, tq_prod_cache k, tq_mse_cache v,
                              const int32_t* seq_lens, void* out, void* workspace,
                              size_t workspace_bytes, tq_stream_t stream);

/* Attention of a chunk of n_queries new queries per sequence over the compressed cache (the
 * read path of [QJL] §六 for many queries: each query forward-rotated and pre-sketched once,
 * scores on the packed bits, one softmax per query), e.g. a prefill chunk or several tokens
 * proposed at once.
 *   desc     : desc->batch sequences; desc->max_seq_len bounds the longest query row's attended
 *              length (max(seq_lens) + n_queries when causal).
 *   q, out   : device [batch][n_queries][q_heads][128] of desc->q_dtype / desc->out_dtype.
 *   seq_lens : device int32[batch]: the history length of each sequence.  causal = 0: every
 *              query of sequence b attends its seq_lens[b] tokens; causal = 1: query i attends
 *              seq_lens[b] + i + 1 tokens, the chunk's own keys and values having been appended
 *              to the caches after the history.
 *   workspace: ≥ tq_prefill_workspace_bytes(desc, n_queries) bytes.
 *   Other arguments as tq_decode_attention.  Each query row streams its attended tokens (rows
 *   of one sequence read its cache from L2 after the first); key index widths of 1–3 bits and
 *   group sizes up to 8 (the tcgen05 path), else TQ_ERR_UNSUPPORTED. */
size_t tq_prefill_workspace_bytes(const tq_attn_desc* desc, int32_t n_queries);
tq_status tq_prefill_attention(const tq_attn_desc* desc, int32_t n_queries, int32_t causal,
                               const tq_codec* kc, const tq_codec* vc, const void* q,
                               tq_prod_cache k, tq_mse_cache v, const int32_t* seq_lens, void* out,
                               void* workspace, size_t workspace_bytes, tq_stream_t stream);

/* One decode step in a single call ([QJL] §六: the compressed store appends each new token's
 * codes, then the read path attends the whole store; [MLX] quick start: append, then decode):
 * quantises the step's new key (product code) and value (MSE code) of every (batch, KV head)
 * into the caches at position pos[b], then runs decode attention over pos[b] + 1 tokens.  The
 * result equals tq_quantize_prod + tq_quantize_mse (one token at pos) followed by
 * tq_decode_attention with seq_lens = pos + 1; on the tensor-core path the appends and the
 * query operand share one launch.
 *   k_new, v_new : device [batch][kv_heads][128] of kv_dtype (F32, F16 or BF16), 16-byte
 *                  aligned.
 *   pos      : device int32[batch], the append positions (< capacity; a position out of range
 *              is skipped and flagged TQ_FLAG_POS_OVERFLOW).  desc->max_seq_len must be at
 *              least max(pos) + 1.
 *   lens_out : device int32[batch] or NULL; receives pos[b] + 1 (must not alias pos).
 *   Other arguments as tq_decode_attention (same workspace size). */
tq_status tq_decode_step(const tq_attn_desc* desc, const tq_codec* kc, const tq_codec* vc,
                         const void* q, const void* k_new, const void* v_new, tq_dtype kv_dtype,
                         tq_prod_cache k, tq_mse_cache v, const int32_t* pos, int32_t* lens_out,
                         void* out, void* workspace, size_t workspace_bytes, tq_stream_t stream);

/* Asymmetric mode ([MLX] "对称 vs 非对称": K = FP16, V = turbo): keys stay FP16, values
 * are MSE-coded, and the most recent tokens sit uncompressed in an FP16 tail that joins
 * the same softmax.
 *   k_f16    : device fp16 [batch][kv_heads][capacity][128], keys of the compressed segment.
 *   v        : MSE cache [batch][kv_heads][capacity], values of the compressed segment.
 *   seq_lens : device int32[batch], length of the compressed segment.
 *   k_tail, v_tail : device fp16 [batch][kv_heads][tail_capacity][128].
 *   tail_lens: device int32[batch] (≤ tail_capacity).
 *   Other arguments as tq_decode_attention. */
tq_status tq_decode_attention_asym(const tq_attn_desc* desc, const tq_codec* vc, const void* q,
                                   const uint16_t* k_f16, tq_mse_cache v,
                                   const int32_t* seq_lens, const uint16_t* k_tail,
                                   const uint16_t* v_tail, const int32_t* tail_lens, void* out,
                                   void* workspace, size_t workspace_bytes, tq_stream_t stream);

/* ------------------------------------------------------------------ store with an FP16 tail */

/* Bytes of workspace tq_store_append needs for `batch` sequences (0 if batch ≤ 0). */
size_t tq_store_workspace_bytes(int32_t batch);

/* Appends one token per sequence to a cache kept in the asymmetric layout: a compressed part
 * (FP16 keys, MSE-coded values) and an FP16 tail of the most recent tokens ([QJL] §六: the
 * store appends in chunks and keeps recent tokens in full precision; [MLX] quick start:
 * `min_compress_tokens`, and `key_bits=0` for FP16 keys).  For each sequence b the new key and
 * value go to tail slot tail_lens[b]; the append that fills the last of the tail_capacity slots
 * compacts the tail: its keys are copied to k_f16 and its values MSE-coded into v, at positions
 * comp_lens[b] .. comp_lens[b] + tail_capacity − 1, comp_lens[b] grows by tail_capacity and
 * tail_lens[b] returns to 0; otherwise tail_lens[b] grows by one.  The cache is then read with
 * tq_decode_attention_asym (seq_lens = comp_lens, tail_lens = tail_lens, desc->capacity =
 * capacity, desc->tail_capacity = tail_capacity).
 *   vc        : value codec (TQ_MSE).
 *   k_new, v_new : device [batch][kv_heads][128] of dtype (F32, F16 or BF16).
 *   k_f16     : device fp16 [batch][kv_heads][capacity][128], keys of the compressed part.
 *   v         : MSE cache [batch][kv_heads][capacity], values of the compressed part.
 *   k_tail, v_tail : device fp16 [batch][kv_heads][tail_capacity][128].
 *   comp_lens, tail_lens : device int32[batch], read and updated.
 *   workspace : device, ≥ tq_store_workspace_bytes(batch) bytes (no initialisation needed).
 * capacity must be a positive multiple of 64 and tail_capacity a positive multiple of 8; arrays
 * 16-byte aligned.  A sequence whose tail length is out of range, or whose compaction would
 * pass the capacity, is left unchanged and TQ_FLAG_LEN_OVERFLOW is raised.  Several launches on
 * `stream`; allocates nothing. */
tq_status tq_store_append(const tq_codec* vc, int32_t batch, int32_t kv_heads, const void* k_new,
                          const void* v_new, tq_dtype dtype, uint16_t* k_f16, tq_mse_cache v,
                          int32_t capacity, uint16_t* k_tail, uint16_t* v_tail,
                          int32_t tail_capacity, int32_t* comp_lens, int32_t* tail_lens,
                          void* workspace, size_t workspace_bytes, tq_stream_t stream);

/* Decode attention for callers that cannot allocate device memory (no counterpart on the
 * pages: this is a deployment variant of tq_decode_attention, computing exactly the same
 * result).  Callers such as an inference runtime's plugin whose enqueue call may not
 * allocate, a process whose device memory is owned by another framework's pool, or a
 * latency-critical loop that must not enter the allocator (cudaMalloc/cudaFree may
 * synchronise the device) cannot provide the workspace that tq_decode_attention takes.
 * This entry point uses instead a static device array inside the library, of
 * tq_decode_noalloc_scratch_bytes() bytes (8 MiB), which every GPU that loads the library
 * holds until the process exits.  It allocates nothing.
 *   Arguments: as tq_decode_attention, without the workspace.
 *   Returns TQ_ERR_SCRATCH_LIMIT, launching nothing, when tq_decode_workspace_bytes(desc)
 *   exceeds the static size (e.g. very long contexts or large batches: use the workspace
 *   entry point there).
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *   with that device current, so make the first call on each device before capturing any
 *   stream.  The address is cached for the device's primary context: after cudaDeviceReset
 *   (which also destroys every codec on the device) the library must not be used on that
 *   device again.  All calls on a device share the one array: calls that may overlap on the
 *   GPU (different streams without ordering between them) race and must not be issued;
 *   calls ordered on one stream are safe.  The array keeps the previous call's data; the
 *   decode path clears the part that must start at zero (its split tickets) itself. */
tq_status tq_decode_attention_noalloc(const tq_attn_desc* desc, const tq_codec* kc,
                                      const tq_codec* vc, const void* q, tq_prod_cache k,
                                      tq_mse_cache v, const int32_t* seq_lens, void* out,
                                      tq_stream_t stream);

/* Size in bytes of the static scratch array used by tq_decode_attention_noalloc. */
size_t tq_decode_noalloc_scratch_bytes(void);

/* ------------------------------------------------------------------ diagnostics */

/* Bits of the per-device status word (see tq_device_status). */
#define TQ_FLAG_POS_OVERFLOW 0x1u   /* a quantised token landed at or beyond capacity */
#define TQ_FLAG_LEN_OVERFLOW 0x2u   /* a seq_len or tail_len exceeded its capacity */
#define TQ_FLAG_TIMEOUT      0x4u   /* a bounded device-side wait gave up */
#define TQ_FLAG_PAGE         0x8u   /* a block-table entry outside [0, num_pages) was skipped */

/* Synchronises the current device, returns the status word in *flags (host) and clears
 * it.  Returns TQ_ERR_TIMEOUT if TQ_FLAG_TIMEOUT was set, else TQ_ERR_DEVICE_STATUS if any
 * other bit was set, TQ_OK otherwise. */
tq_status tq_device_status(uint32_t* flags);

/* Exercises the bounded device-side wait that every kernel of the library uses on its
 * barriers (no counterpart on the pages: failure detection of this implementation).  Launches
 * one warp on `stream` that waits on a barrier nothing arrives at, with a limit of `limit_us`
 * microseconds (1..1000000) of GPU time; the wait gives up, raises TQ_FLAG_TIMEOUT and the
 * kernel returns, leaving the context usable.  A following tq_device_status() then returns
 * TQ_ERR_TIMEOUT and clears the flag.  Returns TQ_ERR_INVALID_ARG for a limit out of range,
 * TQ_ERR_CUDA if the launch fails. */
tq_status tq_check_bounded_wait(uint32_t limit_us, tq_stream_t stream);

/* Library version string. */
const char* tq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
