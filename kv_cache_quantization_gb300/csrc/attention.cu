// Decode attention on the compressed cache (QJL deep-dive §五–§六) and the asymmetric
// K = FP16 / V = MSE mode (MLX-port article, "对称 vs 非对称").
//
// Three launches per call, all on the caller's stream:
//   1. query prep   — q_rot = Π q and q_sk = S q for every query head ("forward-rotate and
//                     pre-sketch the query once").  Symmetric mode only.
//   2. split decode — grid (context split, KV head, batch); every CTA serves the whole GQA
//                     group of its KV head, scores its tokens straight from the packed bits,
//                     runs a local softmax and accumulates Σ p·‖v‖·c[idx] in the rotated
//                     domain (FP16-tail splits of the asymmetric mode accumulate plain
//                     values instead); it writes (m, l, acc[128]) per query head.
//   3. merge        — log-sum-exp combination of the splits, one rotation back Πᵀ·acc,
//                     division by the softmax denominator, cast to the output dtype.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "decode_args.h"
#include "tq_internal.h"

TQ_DEFINE_FLAGS(tq_take_flags_attention)

namespace {

constexpr int kSplit = 256;          // tokens per split
constexpr int kThreads = 128;
constexpr int kRec = TQ_REC;        // partial record: m, l, acc[128], padding
constexpr float kQjlNum = 1.2533141373155003f;   // √(π/2)

struct Plan {
  int G, nsplit_main, nsplit_tail, nsplit, split_len;
  size_t q_off, part_off, ctr_off, lens_off, bytes;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
  const int n = tq_num_sms();
  return n > 0 ? n : 148;
}

// Context split: one CTA per (batch, KV head, split); about one CTA per SM for the longest
// sequence, splits a multiple of 128 tokens (the tensor-core kernel's chunk).
tq_status plan(const tq_attn_desc* d, bool asym, Plan* p) {
  if (!d) return TQ_ERR_INVALID_ARG;
  if (d->head_dim != TQ_HEAD_DIM) return TQ_ERR_UNSUPPORTED;
  if (d->batch < 0 || d->q_heads <= 0 || d->kv_heads <= 0) return TQ_ERR_INVALID_ARG;
  if (d->q_heads % d->kv_heads) return TQ_ERR_INVALID_ARG;
  if (d->q_heads / d->kv_heads > TQ_MAX_GROUP) return TQ_ERR_UNSUPPORTED;
  if (d->capacity <= 0 || d->capacity % TQ_CAPACITY_ALIGN) return TQ_ERR_INVALID_ARG;
  if (d->max_seq_len < 0 || d->max_seq_len > d->capacity) return TQ_ERR_INVALID_ARG;
  if (d->tail_capacity < 0 || (!asym && d->tail_capacity != 0)) return TQ_ERR_INVALID_ARG;
  for (tq_dtype t : {d->q_dtype, d->out_dtype})
    if (t != TQ_F32 && t != TQ_F16 && t != TQ_BF16) return TQ_ERR_UNSUPPORTED;
  p->G = d->q_heads / d->kv_heads;
  const long long units = (long long)(d->batch > 0 ? d->batch : 1) * d->kv_heads;
  long long want = (sm_count() + units - 1) / units;                // splits per sequence
  // more units than half the SMs: a wave does not give every unit two splits, and ragged
  // lengths leave SMs idle; three splits per sequence (several waves) balance better
  if (units * 2 > sm_count() && want < 3) want = 3;
  if (asym) {
    // the tail's CTAs share the wave: splits of the compressed part plus the tail's per unit
    const long long tail_splits = (d->tail_capacity + kSplit - 1) / kSplit;
    const long long fit = sm_count() / units - tail_splits;
    want = fit >= 1 ? fit : 1;
  }
  long long sl = (d->max_seq_len + want - 1) / (want > 0 ? want : 1);
  sl = (sl + 127) / 128 * 128;
  if (sl < 128) sl = 128;
  p->split_len = (int)sl;
  p->nsplit_main = d->max_seq_len > 0 ? (int)((d->max_seq_len + sl - 1) / sl) : 1;
  p->nsplit_tail = asym ? (d->tail_capacity + kSplit - 1) / kSplit : 0;
  p->nsplit = p->nsplit_main + p->nsplit_tail;
  // per-query vectors (CUDA-core path) or per-(batch, KV head) query fragments
  // (tensor-core path), whichever is larger
  size_t qbytes = (size_t)d->batch * d->q_heads * 2 * TQ_D * sizeof(float);
  const size_t fbytes = (size_t)d->batch * d->kv_heads * tq_tc_frag_bytes_max();
  if (fbytes > qbytes) qbytes = fbytes;
  const size_t pf = (size_t)d->batch * d->kv_heads * p->nsplit * p->G * kRec;
  p->q_off = 0;
  p->part_off = (qbytes + 255) / 256 * 256;
  // split tickets of the tensor-core path: one int per (batch, KV head), cleared by the
  // query-operand kernel at the start of every call
  p->ctr_off = (p->part_off + pf * sizeof(float) + 255) / 256 * 256;
  // a decode step on the CUDA-core path: the attended lengths pos + 1
  p->lens_off = (p->ctr_off + (size_t)d->batch * d->kv_heads * sizeof(int) + 255) / 256 * 256;
  p->bytes = p->lens_off + (size_t)d->batch * sizeof(int);
  return TQ_OK;
}

__device__ __forceinline__ float load_elem(const void* base, int dtype, long long i) {
  if (dtype == TQ_F32) return static_cast<const float*>(base)[i];
  const uint16_t u = static_cast<const uint16_t*>(base)[i];
  if (dtype == TQ_BF16) return __uint_as_float((uint32_t)u << 16);
  return __half2float(__ushort_as_half(u));
}

__device__ __forceinline__ void store_elem(void* base, int dtype, long long i, float v) {
  if (dtype == TQ_F32) static_cast<float*>(base)[i] = v;
  else if (dtype == TQ_BF16) static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  else static_cast<__half*>(base)[i] = __float2half_rn(v);
}

// ---------------------------------------------------------------- 1. query prep
// One CTA of 512 threads per query row: both 128×128 products split four ways over k.
constexpr int kPrepThreads = 512;   // CUDA-core path query prep
__global__ void __launch_bounds__(kPrepThreads) query_prep_kernel(const void* q, int q_dtype,
                                                                  const float* piT, const float* sT,
                                                                  float* qv) {
  __shared__ float qf[TQ_D];
  __shared__ float part[2][4][TQ_D];
  const int row = blockIdx.x;  // b * Hq + h
  const int tid = threadIdx.x, j = tid & 127, kq = tid >> 7;
  if (tid < TQ_D) qf[tid] = load_elem(q, q_dtype, (long long)row * TQ_D + tid);
  __syncthreads();
  float tp[32], ts[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) {   // all loads first: one round trip
    tp[k] = __ldg(&piT[(32 * kq + k) * TQ_D + j]);
    ts[k] = __ldg(&sT[(32 * kq + k) * TQ_D + j]);
  }
  float r = 0.f, s = 0.f;
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    r = fmaf(tp[k], qf[32 * kq + k], r);
    s = fmaf(ts[k], qf[32 * kq + k], s);
  }
  part[0][kq][j] = r;
  part[1][kq][j] = s;
  __syncthreads();
  if (tid < 2 * TQ_D) {
    const int w = tid >> 7;
    qv[(size_t)row * 2 * TQ_D + w * TQ_D + j] =
        (part[w][0][j] + part[w][1][j]) + (part[w][2][j] + part[w][3][j]);
  }
}

struct DecodeArgs {
  int B, Hq, Hkv, G, cap, tail_cap;
  int nsplit_main, nsplit, split_len;
  float scale;
  // symmetric
  const float* qv;
  const uint8_t* kidx;
  const uint8_t* ksgn;
  const float* kxn;
  const float* krn;
  int kbits;                 // key index bits
  tq_levels kl;
  // asymmetric
  const void* q;
  int q_dtype;
  const __half* kf16;
  const __half* ktail;
  const __half* vtail;
  const int* tail_lens;
  // values
  const uint8_t* vidx;
  const float* vxn;
  int vbits;
  tq_levels vl;
  const int* seq_lens;
  float* part;
};

__device__ __forceinline__ int value_index(const DecodeArgs& a, long long bh, int t, int j) {
  if (a.vbits == 4) {
    const uint8_t byte = a.vidx[((long long)bh * a.cap + t) * 64 + (j >> 1)];
    return (byte >> ((j & 1) * 4)) & 15;
  }
  int q = 0;
  for (int p = 0; p < a.vbits; ++p) {
    const uint8_t byte = a.vidx[(((long long)bh * a.vbits + p) * a.cap + t) * 16 + (j >> 3)];
    q |= ((byte >> (j & 7)) & 1) << p;
  }
  return q;
}

// Running softmax state of one CTA (one KV head's query group over one split): m and l per
// head in shared memory, acc[g] of coordinate j = threadIdx.x in registers.
struct RunState {
  float acc[TQ_MAX_GROUP];
};

// Folds one sub-chunk of scores sc[g][0..n_tok) into the running state: new maxima rescale
// l and acc, probabilities replace the scores, values are accumulated.
__device__ void fold_chunk(const DecodeArgs& a, float (*sc)[kSplit], int n_tok, int start,
                           bool plain_values, long long bh, float* s_m, float* s_l, float* s_corr,
                           RunState& rs) {
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  for (int g = warp; g < a.G; g += kThreads / 32) {
    float m = -INFINITY;
    for (int tt = lane; tt < n_tok; tt += 32) m = fmaxf(m, sc[g][tt]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float m_old = s_m[g];
    const float m_new = fmaxf(m_old, m);
    float l = 0.f;
    for (int tt = lane; tt < n_tok; tt += 32) {
      const float p = expf(sc[g][tt] - m_new);
      sc[g][tt] = p;
      l += p;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane == 0) {
      const float corr = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
      s_corr[g] = corr;
      s_m[g] = m_new;
      s_l[g] = s_l[g] * corr + l;
    }
  }
  __syncthreads();
  const int j = tid;
#pragma unroll
  for (int g = 0; g < TQ_MAX_GROUP; ++g)
    if (g < a.G) rs.acc[g] *= s_corr[g];
  for (int tt = 0; tt < n_tok; ++tt) {
    const int t = start + tt;
    float val;
    if (plain_values) {
      val = __half2float(a.vtail[((long long)bh * a.tail_cap + t) * TQ_D + j]);
    } else {
      val = a.vxn[(long long)bh * a.cap + t] * a.vl.c[value_index(a, bh, t, j)];
    }
#pragma unroll
    for (int g = 0; g < TQ_MAX_GROUP; ++g)
      if (g < a.G) rs.acc[g] = fmaf(sc[g][tt], val, rs.acc[g]);
  }
  __syncthreads();   // sc is rewritten by the next sub-chunk
}

__device__ void write_record(const DecodeArgs& a, long long bh, int split, const float* s_m,
                             const float* s_l, const RunState& rs) {
  const int j = threadIdx.x;
  float* rec = a.part + ((bh * a.nsplit + split) * a.G) * kRec;
  for (int g = 0; g < a.G; ++g) {
    if (j == 0) {
      rec[g * kRec + 0] = s_m[g];
      rec[g * kRec + 1] = s_l[g];
    }
    rec[g * kRec + 2 + j] = rs.acc[g];
  }
}

// ---------------------------------------------------------------- 2a. symmetric split decode
// CUDA-core path, used for key codes with 4 index bits (the tensor-core kernel covers 1–3).
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeArgs a) {
  __shared__ float qr[TQ_MAX_GROUP][TQ_D];
  __shared__ float qs[TQ_MAX_GROUP][TQ_D];
  __shared__ float sc[TQ_MAX_GROUP][kSplit];
  __shared__ float s_m[TQ_MAX_GROUP], s_l[TQ_MAX_GROUP], s_corr[TQ_MAX_GROUP];
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long bh = (long long)b * a.Hkv + kvh;
  const int tid = threadIdx.x;
  int len = a.seq_lens[b];
  if (len > a.cap) {
    if (tid == 0 && split == 0 && kvh == 0) atomicOr(&g_tq_flags, TQ_FLAG_LEN_OVERFLOW);
    len = a.cap;
  }
  for (int g = 0; g < a.G; ++g) {
    const long long row = (long long)b * a.Hq + kvh * a.G + g;
    qr[g][tid] = a.qv[row * 2 * TQ_D + tid];
    qs[g][tid] = a.qv[row * 2 * TQ_D + TQ_D + tid];
  }
  if (tid < TQ_MAX_GROUP) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  RunState rs;
#pragma unroll
  for (int g = 0; g < TQ_MAX_GROUP; ++g) rs.acc[g] = 0.f;
  __syncthreads();
  const float qjl = kQjlNum / TQ_D;
  const int s_begin = split * a.split_len, s_end = min(s_begin + a.split_len, len);
  for (int start = s_begin; start < s_end; start += kSplit) {
    const int n_tok = min(kSplit, s_end - start);
    for (int tt = tid; tt < n_tok; tt += kThreads) {
      const int t = start + tt;
      uint4 planes[4];
      for (int p = 0; p < a.kbits; ++p)
        planes[p] = *reinterpret_cast<const uint4*>(a.kidx + ((bh * a.kbits + p) * a.cap + t) * 16);
      const uint4 sg = *reinterpret_cast<const uint4*>(a.ksgn + (bh * a.cap + t) * 16);
      const float xn = a.kxn[bh * a.cap + t], rn = a.krn[bh * a.cap + t];
      float mse[TQ_MAX_GROUP], qj[TQ_MAX_GROUP];
#pragma unroll
      for (int g = 0; g < TQ_MAX_GROUP; ++g) mse[g] = qj[g] = 0.f;
      for (int w = 0; w < 4; ++w) {
        uint32_t pw[4];
        for (int p = 0; p < 4; ++p) {
          const uint4 u = planes[p];
          pw[p] = w == 0 ? u.x : w == 1 ? u.y : w == 2 ? u.z : u.w;
        }
        const uint32_t sw = w == 0 ? sg.x : w == 1 ? sg.y : w == 2 ? sg.z : sg.w;
        for (int bit = 0; bit < 32; ++bit) {
          const int j = w * 32 + bit;
          int q = 0;
          for (int p = 0; p < a.kbits; ++p) q |= ((pw[p] >> bit) & 1) << p;
          const float c = a.kl.c[q];
          const float s = ((sw >> bit) & 1) ? 1.f : -1.f;
#pragma unroll
          for (int g = 0; g < TQ_MAX_GROUP; ++g) {
            if (g < a.G) {
              mse[g] = fmaf(qr[g][j], c, mse[g]);
              qj[g] = fmaf(qs[g][j], s, qj[g]);
            }
          }
        }
      }
#pragma unroll
      for (int g = 0; g < TQ_MAX_GROUP; ++g)
        if (g < a.G) sc[g][tt] = a.scale * (xn * mse[g] + rn * qjl * qj[g]);
    }
    __syncthreads();
    fold_chunk(a, sc, n_tok, start, false, bh, s_m, s_l, s_corr, rs);
  }
  write_record(a, bh, split, s_m, s_l, rs);
}

// ---------------------------------------------------------------- 2b. asymmetric split decode
__global__ void __launch_bounds__(kThreads) decode_asym_kernel(DecodeArgs a) {
  __shared__ float qf[TQ_MAX_GROUP][TQ_D];
  __shared__ float sc[TQ_MAX_GROUP][kSplit];
  __shared__ float s_m[TQ_MAX_GROUP], s_l[TQ_MAX_GROUP], s_corr[TQ_MAX_GROUP];
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long bh = (long long)b * a.Hkv + kvh;
  const int tid = threadIdx.x;
  const bool tail = split >= a.nsplit_main;
  int len = tail ? a.tail_lens[b] : a.seq_lens[b];
  const int cap = tail ? a.tail_cap : a.cap;
  if (len > cap) {
    if (tid == 0 && (split == 0 || split == a.nsplit_main) && kvh == 0)
      atomicOr(&g_tq_flags, TQ_FLAG_LEN_OVERFLOW);
    len = cap;
  }
  const int span = tail ? kSplit : a.split_len;
  const int s_begin = (tail ? split - a.nsplit_main : split) * span;
  const int s_end = min(s_begin + span, len);
  for (int g = 0; g < a.G; ++g)
    qf[g][tid] = load_elem(a.q, a.q_dtype, ((long long)b * a.Hq + kvh * a.G + g) * TQ_D + tid);
  if (tid < TQ_MAX_GROUP) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  RunState rs;
#pragma unroll
  for (int g = 0; g < TQ_MAX_GROUP; ++g) rs.acc[g] = 0.f;
  __syncthreads();
  const __half* K = tail ? a.ktail : a.kf16;
  for (int start = s_begin; start < s_end; start += kSplit) {
    const int n_tok = min(kSplit, s_end - start);
    for (int tt = tid; tt < n_tok; tt += kThreads) {
      const int t = start + tt;
      const uint4* row = reinterpret_cast<const uint4*>(K + ((long long)bh * cap + t) * TQ_D);
      float dot[TQ_MAX_GROUP];
#pragma unroll
      for (int g = 0; g < TQ_MAX_GROUP; ++g) dot[g] = 0.f;
      for (int c = 0; c < TQ_D / 8; ++c) {
        const uint4 u = row[c];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          const int j = c * 8 + 2 * e;
#pragma unroll
          for (int g = 0; g < TQ_MAX_GROUP; ++g)
            if (g < a.G) dot[g] = fmaf(qf[g][j], f.x, fmaf(qf[g][j + 1], f.y, dot[g]));
        }
      }
#pragma unroll
      for (int g = 0; g < TQ_MAX_GROUP; ++g)
        if (g < a.G) sc[g][tt] = a.scale * dot[g];
    }
    __syncthreads();
    fold_chunk(a, sc, n_tok, start, tail, bh, s_m, s_l, s_corr, rs);
  }
  write_record(a, bh, split, s_m, s_l, rs);
}

// ---------------------------------------------------------------- 3. merge
// One CTA of 512 threads per (batch, query head): the splits are combined four ways in
// parallel (log-sum-exp weights), then out = Πᵀ·acc / L with the product split over k.
constexpr int kMergeThreads = 512;
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const float* part, int Hq, int Hkv,
                                                              int G, int nsplit_main, int nsplit,
                                                              const float* pi, void* out,
                                                              int out_dtype) {
  __shared__ float accR[4][TQ_D], accP[4][TQ_D], accs[TQ_D], prod[4][TQ_D];
  __shared__ float s_M, s_L[4];
  const int row = blockIdx.x;  // b * Hq + h
  const int b = row / Hq, h = row % Hq;
  const int kvh = h / G, g = h % G;
  const long long bh = (long long)b * Hkv + kvh;
  const int tid = threadIdx.x, j = tid & 127, q = tid >> 7;
  const float* recs = part + (bh * nsplit * G + g) * kRec;   // split s at recs + s*G*kRec
  if (tid < 32) {
    float M = -INFINITY;
    for (int sp = tid; sp < nsplit; sp += 32) M = fmaxf(M, recs[(long long)sp * G * kRec]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (tid == 0) s_M = M;
  }
  __syncthreads();
  const float M = s_M;
  float L = 0.f, aR = 0.f, aP = 0.f;
  if (M > -INFINITY) {
    for (int sp = q; sp < nsplit; sp += 4) {
      const float* rec = recs + (long long)sp * G * kRec;
      const float l = rec[1];
      if (!(l > 0.f)) continue;
      const float w = expf(rec[0] - M);
      L += w * l;
      if (sp < nsplit_main) aR += w * rec[2 + j];
      else aP += w * rec[2 + j];
    }
  }
  accR[q][j] = aR;
  accP[q][j] = aP;
  if (j == 0) s_L[q] = L;
  __syncthreads();
  if (tid < TQ_D) accs[j] = (accR[0][j] + accR[1][j]) + (accR[2][j] + accR[3][j]);
  __syncthreads();
  float tp[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) tp[k] = __ldg(&pi[(32 * q + k) * TQ_D + j]);
  float r = 0.f;
#pragma unroll
  for (int k = 0; k < 32; ++k) r = fmaf(tp[k], accs[32 * q + k], r);
  prod[q][j] = r;
  __syncthreads();
  if (tid < TQ_D) {
    const float Lt = (s_L[0] + s_L[1]) + (s_L[2] + s_L[3]);
    float o = 0.f;
    if (Lt > 0.f) {
      const float rot = (prod[0][j] + prod[1][j]) + (prod[2][j] + prod[3][j]);
      const float pl = (accP[0][j] + accP[1][j]) + (accP[2][j] + accP[3][j]);
      o = (rot + pl) / Lt;
    }
    store_elem(out, out_dtype, (long long)row * TQ_D + j, o);
  }
}

tq_status check_prod_cache(const tq_prod_cache& k) {
  if (!k.idx || !k.sgn || !k.xnorm || !k.rnorm) return TQ_ERR_INVALID_ARG;
  if (!aligned16(k.idx) || !aligned16(k.sgn) || !aligned16(k.xnorm) || !aligned16(k.rnorm))
    return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

tq_status check_mse_cache(const tq_mse_cache& v) {
  if (!v.idx || !v.xnorm) return TQ_ERR_INVALID_ARG;
  if (!aligned16(v.idx) || !aligned16(v.xnorm)) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

}  // namespace

extern "C" size_t tq_decode_workspace_bytes(const tq_attn_desc* desc) {
  Plan p;
  if (!desc) return 0;
  if (plan(desc, desc->tail_capacity > 0, &p) != TQ_OK) return 0;
  return p.bytes;
}

namespace {

// Inputs of a decode step that the plain decode call does not have.
struct StepIn {
  const void* k_new;
  const void* v_new;
  tq_dtype kv_dtype;
  int32_t* lens_out;
};

// The appends of a decode step (the caches' pointers and the codecs' constants).
tq::AppendKV append_args(const StepIn& in, const tq_attn_desc* desc, const tq_codec* kc,
                         const tq_codec* vc, const tq_prod_cache& k, const tq_mse_cache& v,
                         const tq_rowmap& kmap, const tq_rowmap& vmap, const int32_t* pos,
                         const DecodeArgs& a) {
  tq::AppendKV ap{};
  ap.k_new = in.k_new; ap.v_new = in.v_new; ap.dtype = in.kv_dtype;
  ap.pos = pos; ap.lens_out = in.lens_out;
  ap.Hkv = desc->kv_heads; ap.cap = desc->capacity;
  ap.kidx = k.idx; ap.ksgn = k.sgn; ap.kxn = k.xnorm; ap.krn = k.rnorm;
  ap.vidx = v.idx; ap.vxn = v.xnorm;
  ap.kpiT = kc->d_piT; ap.kmT = kc->d_mT; ap.vpiT = vc->d_piT;
  ap.klv = a.kl; ap.vlv = a.vl;
  ap.kbits = kc->ibits; ap.vbits = vc->ibits; ap.v_nibbles = vc->ibits == 4;
  ap.shared_pi = kc->pi_digest == vc->pi_digest;
  ap.kmap = kmap; ap.vmap = vmap;
  return ap;
}

// Attended lengths of a decode step on the CUDA-core path: pos + 1.
__global__ void step_lens_kernel(const int32_t* pos, int n, int32_t* lens, int32_t* lens_out) {
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < n; b += gridDim.x * blockDim.x) {
    const int32_t l = pos[b] + 1;
    lens[b] = l;
    if (lens_out) lens_out[b] = l;
  }
}

// Symmetric decode attention, optionally preceded by a decode step's append (step != null:
// seq_lens holds the append positions and pos + 1 tokens are attended).
tq_status run_decode(const tq_attn_desc* desc, const tq_codec* kc, const tq_codec* vc,
                     const void* q, tq_prod_cache k, tq_mse_cache v, const int32_t* seq_lens,
                     void* out, void* workspace, size_t workspace_bytes, tq_stream_t stream_,
                     const StepIn* step, int qps = 1, int causal = 0) {
  Plan p;
  tq_status st = plan(desc, false, &p);
  if (st != TQ_OK) return st;
  if ((st = tq_check_codec(kc, TQ_PROD)) != TQ_OK) return st;
  if ((st = tq_check_codec(vc, TQ_MSE)) != TQ_OK) return st;
  if ((st = check_prod_cache(k)) != TQ_OK) return st;
  if ((st = check_mse_cache(v)) != TQ_OK) return st;
  tq_rowmap kmap, vmap;
  if ((st = tq_rowmap_of(k.pages, desc->capacity, &kmap)) != TQ_OK) return st;
  if ((st = tq_rowmap_of(v.pages, desc->capacity, &vmap)) != TQ_OK) return st;
  if (!q || !seq_lens || !out || !workspace) return TQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < p.bytes)
    return TQ_ERR_INVALID_ARG;
  if (step) {
    if (!step->k_new || !step->v_new || !aligned16(step->k_new) || !aligned16(step->v_new))
      return TQ_ERR_INVALID_ARG;
    if (step->kv_dtype != TQ_F32 && step->kv_dtype != TQ_F16 && step->kv_dtype != TQ_BF16)
      return TQ_ERR_UNSUPPORTED;
    if (step->lens_out && static_cast<const void*>(step->lens_out) == seq_lens)
      return TQ_ERR_INVALID_ARG;
  }
  if (desc->batch == 0) return TQ_OK;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  DecodeArgs a{};
  a.B = desc->batch; a.Hq = desc->q_heads; a.Hkv = desc->kv_heads; a.G = p.G;
  a.cap = desc->capacity; a.tail_cap = 0;
  a.nsplit_main = p.nsplit_main; a.nsplit = p.nsplit; a.split_len = p.split_len;
  a.scale = desc->softmax_scale > 0.f ? desc->softmax_scale : 1.0f / sqrtf((float)TQ_D);
  a.qv = reinterpret_cast<const float*>(ws + p.q_off);
  a.kidx = k.idx; a.ksgn = k.sgn; a.kxn = k.xnorm; a.krn = k.rnorm;
  a.kbits = kc->ibits; a.kl = tq_make_levels(kc);
  a.vidx = v.idx; a.vxn = v.xnorm; a.vbits = vc->ibits; a.vl = tq_make_levels(vc);
  a.seq_lens = seq_lens;
  a.part = reinterpret_cast<float*>(ws + p.part_off);
  const int rows = desc->batch * desc->q_heads;
  const bool tc = tq_tc_decode_supported(kc->ibits, vc->ibits, p.G, p.nsplit);
  if (!tc && qps > 1) return TQ_ERR_UNSUPPORTED;   // query rows sharing a cache row: tcgen05 path
  if (!tc && (kmap.table || vmap.table)) return TQ_ERR_UNSUPPORTED;   // paged: tcgen05 path
  if (tc) {
    tq_mma_launch m{};
    m.qps = qps;
    m.causal = causal;
    m.B = a.B; m.Hq = a.Hq; m.Hkv = a.Hkv; m.G = a.G; m.cap = a.cap;
    m.nsplit = p.nsplit; m.split_len = p.split_len;
    m.scale_log2 = a.scale * 1.4426950408889634f;
    m.q = q; m.q_dtype = desc->q_dtype; m.piT = kc->d_piT; m.sT = kc->d_sT;
    m.u = kc->d_u; m.w = kc->d_w; m.smax = kc->smax;
    m.qfrag = ws + p.q_off;
    m.kidx = k.idx; m.ksgn = k.sgn; m.kxn = k.xnorm; m.krn = k.rnorm;
    m.kmap = kmap; m.vmap = vmap;
    m.kbits = kc->ibits; m.kd = tq_decompose_levels(kc);
    m.vidx = v.idx; m.vxn = v.xnorm; m.vbits = vc->ibits;
    if (vc->ibits < 4) m.vd = tq_decompose_levels(vc);
    m.lut = vc->d_lut;
    m.vc_unscale = vc->ibits == 4 ? 1.f / vc->lut_scale : 1.f;
    m.seq_lens = seq_lens;
    m.part = a.part;
    m.pi = vc->d_pi;
    m.vpiT = vc->d_piT;
    m.out = out;
    m.out_dtype = desc->out_dtype;
    m.counters = reinterpret_cast<int*>(ws + p.ctr_off);
    m.max_len = desc->max_seq_len;
    tq_tc_operand_scales(m.kd, &m.s_idx, &m.s_sgn);
    if (!step) return tq_launch_decode_tc(m, stream);   // query operand, split decode + merge
    m.app = append_args(*step, desc, kc, vc, k, v, kmap, vmap, seq_lens, a);
    m.len_add = 1;
    if (tq_step_prologue_fits(desc->batch, desc->kv_heads, m.app.shared_pi ? 1 : 2)) {
      // the appends and the query operand in one prologue launch, then the split decode; the
      // split grid reads the appended token only after the prologue has completed
      m.fresh = 1;
      return tq_launch_decode_step_tc(m, stream);
    }
    // many (batch, KV head) units: the appends as one launch, then the operand kernel and the
    // split decode (the cache is final when the split grid starts)
    m.fresh = 0;
    if ((st = tq_launch_append_kv(m.app, desc->batch, stream)) != TQ_OK) return st;
    return tq_launch_decode_tc(m, stream);
  }
  if (step) {
    // CUDA-core path: the appends, then attention over pos + 1 tokens
    if ((st = tq_launch_append_kv(append_args(*step, desc, kc, vc, k, v, kmap, vmap, seq_lens, a),
                                  desc->batch, stream)) != TQ_OK)
      return st;
    int32_t* lens = reinterpret_cast<int32_t*>(ws + p.lens_off);
    step_lens_kernel<<<(desc->batch + 255) / 256, 256, 0, stream>>>(seq_lens, desc->batch, lens,
                                                                    nullptr);
    a.seq_lens = lens;
  }
  query_prep_kernel<<<rows, kPrepThreads, 0, stream>>>(q, desc->q_dtype, kc->d_piT, kc->d_sT,
                                                   reinterpret_cast<float*>(ws + p.q_off));
  decode_kernel<<<dim3(p.nsplit_main, desc->kv_heads, desc->batch), kThreads, 0, stream>>>(a);
  merge_kernel<<<rows, kMergeThreads, 0, stream>>>(a.part, a.Hq, a.Hkv, a.G, p.nsplit_main, p.nsplit,
                                              vc->d_pi, out, desc->out_dtype);
  return tq_cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" tq_status tq_decode_attention(const tq_attn_desc* desc, const tq_codec* kc,
                                         const tq_codec* vc, const void* q, tq_prod_cache k,
                                         tq_mse_cache v, const int32_t* seq_lens, void* out,
                                         void* workspace, size_t workspace_bytes,
                                         tq_stream_t stream) {
  return run_decode(desc, kc, vc, q, k, v, seq_lens, out, workspace, workspace_bytes, stream,
                    nullptr);
}

extern "C" size_t tq_prefill_workspace_bytes(const tq_attn_desc* desc, int32_t n_queries) {
  if (!desc || n_queries <= 0 || (long long)desc->batch * n_queries > (1 << 30)) return 0;
  tq_attn_desc rows = *desc;
  rows.batch = desc->batch * n_queries;
  return tq_decode_workspace_bytes(&rows);
}

extern "C" tq_status tq_prefill_attention(const tq_attn_desc* desc, int32_t n_queries,
                                          int32_t causal, const tq_codec* kc, const tq_codec* vc,
                                          const void* q, tq_prod_cache k, tq_mse_cache v,
                                          const int32_t* seq_lens, void* out, void* workspace,
                                          size_t workspace_bytes, tq_stream_t stream) {
  if (!desc || n_queries <= 0 || (causal != 0 && causal != 1)) return TQ_ERR_INVALID_ARG;
  if ((long long)desc->batch * n_queries > (1 << 30)) return TQ_ERR_INVALID_ARG;
  tq_attn_desc rows = *desc;
  rows.batch = desc->batch * n_queries;
  return run_decode(&rows, kc, vc, q, k, v, seq_lens, out, workspace, workspace_bytes, stream,
                    nullptr, n_queries, causal);
}

extern "C" tq_status tq_decode_step(const tq_attn_desc* desc, const tq_codec* kc,
                                    const tq_codec* vc, const void* q, const void* k_new,
                                    const void* v_new, tq_dtype kv_dtype, tq_prod_cache k,
                                    tq_mse_cache v, const int32_t* pos, int32_t* lens_out,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    tq_stream_t stream) {
  const StepIn in{k_new, v_new, kv_dtype, lens_out};
  return run_decode(desc, kc, vc, q, k, v, pos, out, workspace, workspace_bytes, stream, &in);
}

extern "C" tq_status tq_decode_attention_asym(const tq_attn_desc* desc, const tq_codec* vc,
                                              const void* q, const uint16_t* k_f16,
                                              tq_mse_cache v, const int32_t* seq_lens,
                                              const uint16_t* k_tail, const uint16_t* v_tail,
                                              const int32_t* tail_lens, void* out,
                                              void* workspace, size_t workspace_bytes,
                                              tq_stream_t stream_) {
  Plan p;
  tq_status st = plan(desc, true, &p);
  if (st != TQ_OK) return st;
  if ((st = tq_check_codec(vc, TQ_MSE)) != TQ_OK) return st;
  if ((st = check_mse_cache(v)) != TQ_OK) return st;
  if (v.pages) return TQ_ERR_UNSUPPORTED;   // the asymmetric path takes flat value caches
  if (!q || !k_f16 || !seq_lens || !out || !workspace) return TQ_ERR_INVALID_ARG;
  if (desc->tail_capacity > 0 && (!k_tail || !v_tail || !tail_lens)) return TQ_ERR_INVALID_ARG;
  if (!aligned16(k_f16) || (k_tail && !aligned16(k_tail)) || (v_tail && !aligned16(v_tail)))
    return TQ_ERR_INVALID_ARG;
  if (desc->tail_capacity % 8) return TQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < p.bytes)
    return TQ_ERR_INVALID_ARG;
  if (desc->batch == 0) return TQ_OK;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  char* ws = static_cast<char*>(workspace);
  DecodeArgs a{};
  a.B = desc->batch; a.Hq = desc->q_heads; a.Hkv = desc->kv_heads; a.G = p.G;
  a.cap = desc->capacity; a.tail_cap = desc->tail_capacity;
  a.nsplit_main = p.nsplit_main; a.nsplit = p.nsplit; a.split_len = p.split_len;
  a.scale = desc->softmax_scale > 0.f ? desc->softmax_scale : 1.0f / sqrtf((float)TQ_D);
  a.q = q; a.q_dtype = desc->q_dtype;
  a.kf16 = reinterpret_cast<const __half*>(k_f16);
  a.ktail = reinterpret_cast<const __half*>(k_tail);
  a.vtail = reinterpret_cast<const __half*>(v_tail);
  a.tail_lens = tail_lens;
  a.vidx = v.idx; a.vxn = v.xnorm; a.vbits = vc->ibits; a.vl = tq_make_levels(vc);
  a.seq_lens = seq_lens;
  a.part = reinterpret_cast<float*>(ws + p.part_off);
  const int rows = desc->batch * desc->q_heads;
  if (tq_asym_tc_supported(vc->ibits, p.G, p.split_len, kSplit)) {
    tq_asym_launch m{};
    m.B = a.B; m.Hq = a.Hq; m.Hkv = a.Hkv; m.G = a.G; m.cap = a.cap; m.tail_cap = a.tail_cap;
    m.nsplit_main = p.nsplit_main; m.nsplit = p.nsplit; m.split_len = p.split_len;
    m.tail_split = kSplit;
    m.scale_log2 = a.scale * 1.4426950408889634f;
    m.q = q; m.q_dtype = desc->q_dtype;
    m.kf16 = a.kf16; m.ktail = a.ktail; m.vtail = a.vtail; m.tail_lens = tail_lens;
    m.vidx = v.idx; m.vxn = v.xnorm; m.vbits = vc->ibits;
    if (vc->ibits < 4) m.vd = tq_decompose_levels(vc);
    m.lut = vc->d_lut;
    m.vc_unscale = vc->ibits == 4 ? 1.f / vc->lut_scale : 1.f;
    m.seq_lens = seq_lens;
    m.part = a.part;
    const long long units = (long long)desc->batch * desc->kv_heads;
    if ((st = tq_asym_encode_rows(&m.kmap, k_f16, units * desc->capacity)) != TQ_OK) return st;
    if ((st = tq_asym_encode_rows(&m.ktmap, k_tail, units * desc->tail_capacity)) != TQ_OK) return st;
    if ((st = tq_asym_encode_rows(&m.vtmap, v_tail, units * desc->tail_capacity)) != TQ_OK) return st;
    st = tq_launch_decode_asym_tc(m, stream);   // split decode (mma.sync), then the merge
    if (st != TQ_OK) return st;
  } else {
    decode_asym_kernel<<<dim3(p.nsplit, desc->kv_heads, desc->batch), kThreads, 0, stream>>>(a);
  }
  merge_kernel<<<rows, kMergeThreads, 0, stream>>>(a.part, a.Hq, a.Hkv, a.G, p.nsplit_main, p.nsplit,
                                              vc->d_pi, out, desc->out_dtype);
  return tq_cuda_status(cudaGetLastError());
}
