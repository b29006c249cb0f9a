// kv_probe.cu -- reads across the host link that are not K/V:
//  * the streaming-read bandwidth probe, the denominator of the roofline for
//    K/V that the GPU reads in place from pinned host memory;
//  * the staging of one decode step's inputs (q, context lengths) from mapped
//    host memory into device buffers.
//
// DirectKV (No Buffer, No Bottleneck: Efficient Zero-Copy KV Cache Offloading
// for Long-Context LLMs), observation 4: long-context access through the
// host link is bound by its sustained bandwidth, so that bandwidth, measured,
// is what host-resident attention is compared against.
#include <algorithm>

#include "kv_internal.cuh"
#include "kv_launch.h"

namespace kvs {
namespace {

// Every thread streams 16-byte loads (L in flight per iteration) over a
// grid-stride range and folds them with XOR, so the loads cannot be elided;
// one word per thread block is written.
template <int L>
__global__ void __launch_bounds__(1024)
    stream_read_kernel(const uint4 *src, size_t n16, unsigned long long *sink) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint4 acc = make_uint4(0u, 0u, 0u, 0u);
  for (; i + (L - 1) * stride < n16; i += L * stride) {
    uint4 v[L];
#pragma unroll
    for (int u = 0; u < L; ++u) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < L; ++u) {
      acc.x ^= v[u].x;
      acc.y ^= v[u].y;
      acc.z ^= v[u].z;
      acc.w ^= v[u].w;
    }
  }
  for (; i < n16; i += stride) {
    const uint4 a = src[i];
    acc.x ^= a.x; acc.y ^= a.y; acc.z ^= a.z; acc.w ^= a.w;
  }
  unsigned long long v = ((unsigned long long)(acc.x ^ acc.z) << 32) | (acc.y ^ acc.w);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v ^= __shfl_xor_sync(0xFFFFFFFFu, v, off);
  __shared__ unsigned long long red[32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long r = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r ^= red[w];
    sink[blockIdx.x] = r;
  }
}

// One decode step's inputs, mapped host -> device: each thread loads its
// context lengths and 16-byte chunks of q from host memory before waiting
// for the previous kernel in the stream (the host wrote them before the
// call), so the host-link latency overlaps that kernel's tail; after the wait
// (the previous step may still read the device copies) it stores them.  It
// never releases its dependents early: the next kernels may read q before
// their own wait, so they must start only once these stores are complete
// and visible, which the end of this grid guarantees.
constexpr int kStageThreads = 256;
constexpr int kStageChunks = 4;  // 16-byte chunks of q per thread
__global__ void __launch_bounds__(kStageThreads)
    stage_inputs_kernel(const uint4 *q_src, uint4 *q_dst, long long n16,
                        const int32_t *ctx_src, int32_t *ctx_dst,
                        int B) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nt = (long long)gridDim.x * blockDim.x;
  uint4 v[kStageChunks];
#pragma unroll
  for (int c = 0; c < kStageChunks; ++c) {
    const long long i = t + c * nt;
    if (i < n16) v[c] = q_src[i];
  }
  int32_t len = 0;
  if (t < B) len = ctx_src[t];
  pdl_wait();
#pragma unroll
  for (int c = 0; c < kStageChunks; ++c) {
    const long long i = t + c * nt;
    if (i < n16) q_dst[i] = v[c];
  }
  if (t < B) ctx_dst[t] = len;
}

}  // namespace

cudaError_t launch_stage_inputs(const void *q_src, void *q_dst, size_t q_bytes,
                                const int32_t *ctx_src, int32_t *ctx_dst, int B,
                                cudaStream_t st) {
  const long long n16 = (long long)(q_bytes / 16);
  const long long per_cta = (long long)kStageThreads * kStageChunks;
  long long blocks = (n16 + per_cta - 1) / per_cta;
  blocks = std::max(blocks, ((long long)B + kStageThreads - 1) / kStageThreads);
  blocks = std::max(blocks, 1LL);
  return launch_pdl(stage_inputs_kernel, dim3((unsigned)blocks), dim3(kStageThreads), 0, st,
                    static_cast<const uint4 *>(q_src), static_cast<uint4 *>(q_dst), n16, ctx_src,
                    ctx_dst, B);
}
}  // namespace kvs

static int probe_common(const void *src, size_t bytes, unsigned long long *sink, int blocks,
                        int threads, int loads, void *stream) {
  using namespace kvs;
  if (!src || !sink || ((uintptr_t)src & 15u) || ((uintptr_t)sink & 7u) || bytes < 16 ||
      (bytes & 15u) || blocks < 1 || (threads != 128 && threads != 256 && threads != 512 &&
                                      threads != 1024) ||
      (loads != 4 && loads != 8 && loads != 16))
    return KV_ERR_INVALID_ARG;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, src) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  const void *dsrc = src;
  if (at.type == cudaMemoryTypeHost) {
    if (!at.devicePointer) return KV_ERR_LOCATION;
    dsrc = at.devicePointer;
  } else if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) {
    return KV_ERR_LOCATION;
  }
  const uint4 *s16 = static_cast<const uint4 *>(dsrc);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (loads) {
    case 4: stream_read_kernel<4><<<blocks, threads, 0, st>>>(s16, bytes / 16, sink); break;
    case 8: stream_read_kernel<8><<<blocks, threads, 0, st>>>(s16, bytes / 16, sink); break;
    default: stream_read_kernel<16><<<blocks, threads, 0, st>>>(s16, bytes / 16, sink); break;
  }
  return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

extern "C" int kv_stream_read_probe(const void *src, size_t bytes, unsigned long long *sink,
                                    int32_t sink_words, void *stream) {
  KV_API_RANGE();
  if (sink_words < 1) return KV_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  return probe_common(src, bytes, sink, std::min(sms * 4, (int)sink_words), 512, 4, stream);
}

extern "C" int kv_stream_read_probe_shape(const void *src, size_t bytes,
                                          unsigned long long *sink, int32_t blocks,
                                          int32_t threads, int32_t loads_in_flight,
                                          void *stream) {
  KV_API_RANGE();
  return probe_common(src, bytes, sink, blocks, threads, loads_in_flight, stream);
}
