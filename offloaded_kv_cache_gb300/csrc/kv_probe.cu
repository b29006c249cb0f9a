// kv_probe.cu -- streaming-read bandwidth probe: the denominator of the
// roofline for K/V that the GPU reads in place from pinned host memory.
//
// DirectKV (No Buffer, No Bottleneck: Efficient Zero-Copy KV Cache Offloading
// for Long-Context LLMs), observation 4: long-context access through the
// host link is bound by its sustained bandwidth, so that bandwidth, measured,
// is what host-resident attention is compared against.
#include "kv_internal.cuh"

namespace kvs {
namespace {

// Every thread streams 16-byte loads (four in flight per iteration) over a
// grid-stride range and folds them with XOR, so the loads cannot be elided;
// one word per thread block is written.
__global__ void __launch_bounds__(512)
    stream_read_kernel(const uint4 *__restrict__ src, size_t n16, unsigned long long *sink) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint4 acc = make_uint4(0u, 0u, 0u, 0u);
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    acc.x ^= a.x ^ b.x ^ c.x ^ d.x;
    acc.y ^= a.y ^ b.y ^ c.y ^ d.y;
    acc.z ^= a.z ^ b.z ^ c.z ^ d.z;
    acc.w ^= a.w ^ b.w ^ c.w ^ d.w;
  }
  for (; i < n16; i += stride) {
    const uint4 a = src[i];
    acc.x ^= a.x; acc.y ^= a.y; acc.z ^= a.z; acc.w ^= a.w;
  }
  unsigned long long v = ((unsigned long long)(acc.x ^ acc.z) << 32) | (acc.y ^ acc.w);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v ^= __shfl_xor_sync(0xFFFFFFFFu, v, off);
  __shared__ unsigned long long red[16];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long r = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r ^= red[w];
    sink[blockIdx.x] = r;
  }
}

}  // namespace
}  // namespace kvs

extern "C" int kv_stream_read_probe(const void *src, size_t bytes, unsigned long long *sink,
                                    int32_t sink_words, void *stream) {
  using namespace kvs;
  if (!src || !sink || ((uintptr_t)src & 15u) || ((uintptr_t)sink & 7u) || bytes < 16 ||
      (bytes & 15u) || sink_words < 1)
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
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  int blocks = sms * 4;
  if (blocks > sink_words) blocks = sink_words;
  stream_read_kernel<<<blocks, 512, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(dsrc), bytes / 16, sink);
  return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}
