// kv_noalloc.cu -- dense decode attention for callers that cannot allocate
// device memory.
//
// kv_dense_decode_attn needs a caller-provided workspace for its split-K
// partial results whenever a row is split over several CTAs.  Some callers
// have no way to provide one: a plugin or custom operator invoked by a host
// framework that hands it only its input and output buffers and owns every
// allocation itself, or a latency-critical loop where a cudaMalloc would
// synchronise the device.  kv_dense_decode_attn_noalloc serves them with a
// fixed scratch array that lives in this library's device image instead.
// Every call on a device shares that one array, so calls that overlap on the
// GPU (on different streams, or from several host threads) race on it.
#include <atomic>
#include <mutex>

#include "kv_internal.cuh"
#include "kv_launch.h"

namespace {

// Split-K partials (per split and query head: 128 outputs plus a running max
// and sum, fp32).  Every GPU that loads this library holds the array until
// the process exits.
constexpr size_t kNoallocScratchBytes = 1u << 20;  // 1 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of the scratch array on the current device, looked up once
// per device (host code only holds a stand-in symbol, never usable as a
// device pointer).
void *scratch_address(int dev) {
  void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void *addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
    cudaGetLastError();
    return nullptr;
  }
  g_scratch_addr[dev].store(addr, std::memory_order_release);
  return addr;
}

}  // namespace

extern "C" int kv_dense_decode_attn_noalloc(const kv_shape *shape, const void *q,
                                            const void *k_cache, const void *v_cache,
                                            const int32_t *block_table,
                                            const int32_t *context_lens, float scale,
                                            float *out, void *stream) {
  KV_API_RANGE();
  if (!shape) return KV_ERR_INVALID_ARG;
  // size check first: a shape whose partials do not fit is refused before any
  // other work (kv_attn_workspace_bytes returns 0 for an invalid shape, and
  // the call below then reports the shape error itself)
  const size_t need = kv_attn_workspace_bytes(shape, 0);
  if (need > kNoallocScratchBytes) return KV_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  void *scratch = scratch_address(dev);
  if (!scratch) return KV_ERR_CUDA;
  // Nothing in the scratch has to start at zero: every partial a call reads
  // was written earlier in the same call.
  return kv_dense_decode_attn(shape, q, k_cache, v_cache, block_table, context_lens, scale, out,
                              scratch, kNoallocScratchBytes, stream);
}
