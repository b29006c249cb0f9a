// kv_append.cu -- decode append: one new token per sequence is written into
// the paged K/V cache (HBM or pinned host memory) and the channel-wise
// min/max of the page it lands in is brought up to date in place.
//
// KVDrive (A Holistic Multi-Tier KV Cache Management System for Long-Context
// LLM Inference), section 2.1: every decode step appends the new key and value
// vectors to the cache; section 2.2: the page index is the channel-wise key
// minimum and maximum.  DirectKV (No Buffer, No Bottleneck), core method 4:
// with the cache in pinned host memory, decode appends the new token there.
//
// The token of sequence b goes to position len = context_lens[b] (its length
// before the append): page len / ps, slot t = len % ps.  For t > 0 the page's
// min/max over t tokens is already in the table, so the new entry is
// min(old, k) / max(old, k) channel by channel (taken in IEEE totalOrder, as
// the build does); for t == 0 the page starts with this token and
// min = max = k.  Either way the entry equals a fresh build over t + 1 tokens.
#include <algorithm>

#include "kv_internal.cuh"
#include "kv_launch.h"

namespace kvs {
namespace {

// One CTA per sequence, so every read of context_lens[b] happens before the
// one write of context_lens_out[b] and the two may alias.  Threads walk the
// (kv head, 16-byte chunk) items of the new rows, one item each when the CTA
// is large enough.
template <class T>
__global__ void __launch_bounds__(1024)
    append_kernel(const T *k_new, const T *v_new, T *k_cache,
                  T *v_cache, const int32_t *bt, const int32_t *ctx, int32_t *ctx_out, T *mm,
                  int Hkv, int ps, int maxP, long long nphys, int *status) {
  pdl_wait();
  constexpr int C = kHeadDim * (int)sizeof(T) / 16;  // 16-byte chunks per row
  const int b = blockIdx.x;
  const int len = ctx[b];
  const bool len_ok = len >= 0 && (long long)len < (long long)maxP * ps;
  const int p = len_ok ? len / ps : 0, t = len_ok ? len % ps : 0;
  const long long phys = len_ok ? (long long)bt[(long long)b * maxP + p] : -1;
  const bool ok = len_ok && phys >= 0 && phys < nphys;
  __syncthreads();  // context_lens[b] is read everywhere before it is written
  if (threadIdx.x == 0) {
    if (!ok) flag_error(status, KV_ERR_BOUNDS);
    if (ctx_out) ctx_out[b] = ok ? len + 1 : len;
  }
  if (!ok) return;
  pdl_trigger();
  const uint4 *kn = reinterpret_cast<const uint4 *>(k_new) + (long long)b * Hkv * C;
  const uint4 *vn = reinterpret_cast<const uint4 *>(v_new) + (long long)b * Hkv * C;
  uint4 *kc = reinterpret_cast<uint4 *>(k_cache);
  uint4 *vc = reinterpret_cast<uint4 *>(v_cache);
  uint4 *tab = reinterpret_cast<uint4 *>(mm);
  for (int i = threadIdx.x; i < Hkv * C; i += blockDim.x) {
    const int kvh = i / C, c = i % C;
    const uint4 k = kn[i];
    const uint4 v = vn[i];
    const long long row = ((phys * Hkv + kvh) * ps + t) * C + c;
    kc[row] = k;
    vc[row] = v;
    if (!mm) continue;
    uint4 *e = tab + (phys * Hkv + kvh) * 2 * C + c;  // [min | max] rows of this page
    uint4 lo = k, hi = k;
    if (t > 0) {
      const uint4 omn = e[0], omx = e[C];
      if constexpr (sizeof(T) == 2) {
        const uint4 kk = make_uint4(key16x2(k.x), key16x2(k.y), key16x2(k.z), key16x2(k.w));
        lo = make_uint4(unkey16x2(__vminu2(kk.x, key16x2(omn.x))),
                        unkey16x2(__vminu2(kk.y, key16x2(omn.y))),
                        unkey16x2(__vminu2(kk.z, key16x2(omn.z))),
                        unkey16x2(__vminu2(kk.w, key16x2(omn.w))));
        hi = make_uint4(unkey16x2(__vmaxu2(kk.x, key16x2(omx.x))),
                        unkey16x2(__vmaxu2(kk.y, key16x2(omx.y))),
                        unkey16x2(__vmaxu2(kk.z, key16x2(omx.z))),
                        unkey16x2(__vmaxu2(kk.w, key16x2(omx.w))));
      } else {
        const uint4 kk = make_uint4(key32(k.x), key32(k.y), key32(k.z), key32(k.w));
        lo = make_uint4(unkey32(min(kk.x, key32(omn.x))), unkey32(min(kk.y, key32(omn.y))),
                        unkey32(min(kk.z, key32(omn.z))), unkey32(min(kk.w, key32(omn.w))));
        hi = make_uint4(unkey32(max(kk.x, key32(omx.x))), unkey32(max(kk.y, key32(omx.y))),
                        unkey32(max(kk.z, key32(omx.z))), unkey32(max(kk.w, key32(omx.w))));
      }
    }
    e[0] = lo;
    e[C] = hi;
  }
}

}  // namespace

cudaError_t launch_append(int dtype, const void *k_new, const void *v_new, void *k_cache,
                          void *v_cache, const int32_t *bt, const int32_t *ctx,
                          int32_t *ctx_out, void *minmax, int B, int Hkv, int ps, int maxP,
                          long long nphys, int *status, cudaStream_t st) {
  const int items = Hkv * kHeadDim * (dtype == KV_F32 ? 4 : 2) / 16;
  const dim3 grid(B), block(std::min(1024, std::max(64, (items + 31) / 32 * 32)));
  switch (dtype) {
    case KV_F32:
      return launch_pdl(append_kernel<float>, grid, block, 0, st,
                        static_cast<const float *>(k_new), static_cast<const float *>(v_new),
                        static_cast<float *>(k_cache), static_cast<float *>(v_cache), bt, ctx,
                        ctx_out, static_cast<float *>(minmax), Hkv, ps, maxP, nphys, status);
    case KV_F16:
      return launch_pdl(append_kernel<__half>, grid, block, 0, st,
                        static_cast<const __half *>(k_new), static_cast<const __half *>(v_new),
                        static_cast<__half *>(k_cache), static_cast<__half *>(v_cache), bt, ctx,
                        ctx_out, static_cast<__half *>(minmax), Hkv, ps, maxP, nphys, status);
    default:
      return launch_pdl(append_kernel<__nv_bfloat16>, grid, block, 0, st,
                        static_cast<const __nv_bfloat16 *>(k_new),
                        static_cast<const __nv_bfloat16 *>(v_new),
                        static_cast<__nv_bfloat16 *>(k_cache),
                        static_cast<__nv_bfloat16 *>(v_cache), bt, ctx, ctx_out,
                        static_cast<__nv_bfloat16 *>(minmax), Hkv, ps, maxP, nphys, status);
  }
}

}  // namespace kvs
