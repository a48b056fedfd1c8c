// Decode attention without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call us: an inference runtime's
// plugin interface that hands a plugin only its input and output buffers and forbids
// allocation inside its enqueue call, a host process whose device memory is owned and
// budgeted by another framework's pool, or a latency-critical loop that must not touch the
// allocator because cudaMalloc/cudaFree can synchronise the device.  This entry point
// serves them: it runs the ordinary decode-attention path with its scratch (per-query
// vectors and per-split partial results) placed in a fixed, statically sized array of
// device memory that the library owns.
//
// The array is a file-scope __device__ object, so every GPU that loads the library holds
// it (kScratchBytes) until the process exits.  Host code may not use the array's name as a
// device address (on the host it is only a stand-in symbol), so the device address is
// looked up once per device with cudaGetSymbolAddress and cached.  The cached address
// belongs to the device's primary context: after cudaDeviceReset it is stale, as are the
// codecs created before the reset, and the library must not be used on that device again.
#include <mutex>

#include "tq_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;   // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on first use).
tq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return TQ_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TQ_OK;
}

}  // namespace

extern "C" size_t tq_decode_noalloc_scratch_bytes(void) { return kScratchBytes; }

extern "C" tq_status tq_decode_attention_noalloc(const tq_attn_desc* desc, const tq_codec* kc,
                                                 const tq_codec* vc, const void* q,
                                                 tq_prod_cache k, tq_mse_cache v,
                                                 const int32_t* seq_lens, void* out,
                                                 tq_stream_t stream) {
  if (!desc) return TQ_ERR_INVALID_ARG;
  const size_t need = tq_decode_workspace_bytes(desc);
  if (need == 0)  // invalid descriptor: let the ordinary entry point report why
    return tq_decode_attention(desc, kc, vc, q, k, v, seq_lens, out, nullptr, 0, stream);
  if (need > kScratchBytes) return TQ_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  tq_status st = scratch_address(&scratch);
  if (st != TQ_OK) return st;
  // The array keeps the previous call's contents; the decode path clears its split tickets
  // itself at the start of every call, so nothing needs resetting here.
  return tq_decode_attention(desc, kc, vc, q, k, v, seq_lens, out, scratch, kScratchBytes, stream);
}
