// kv_union.cuh -- the union of the pages one GQA head chunk selected, as a
// block-wide device function: the body of the union kernel, and one of the
// two roles of the page window's combined update + union launch.
//
// Quest-style selection is per query head (KVDrive, section 2.2); the heads
// of a GQA group read the same kv head, so the attention walks the union of
// their selections once and masks per head.
#pragma once

#include "kv_internal.cuh"

namespace kvs {

// Union of the pages the gc heads of group `grp` (kv head grp / nchunk, head
// chunk grp % nchunk) of sequence b selected, into list slot b * groups + grp:
// head bits per page by shared atomics into `words` (one byte per page, four
// pages a word; (maxP + 3) / 4 words of shared memory), then each thread owns
// a run of consecutive words, counts its union pages and, after one block
// scan, writes them in page order.  `wsum` holds THREADS / 32 words of shared
// memory.  Calls pdl_trigger once the selection has been read.
template <int THREADS>
__device__ __forceinline__ void union_group(const int32_t *idx,
                                            const int32_t *ctx, int Hq, int G,
                                            int gc, int ps, int maxP, int K, int umax,
                                            int32_t *upages,
                                            uint32_t *umasks,
                                            int32_t *ucount, int *status, int grp,
                                            int b, int groups, uint32_t *words, uint32_t *wsum) {
  constexpr int WARPS = THREADS / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nchunk = G / gc;
  const int kvh = grp / nchunk, chunk = grp % nchunk;
  const int head0 = kvh * G + chunk * gc;
  const long long gbase = (long long)b * groups + grp;
  // the first selections load together with the context length
  constexpr int kSpec = 4;
  int32_t sel[kSpec];
#pragma unroll
  for (int u = 0; u < kSpec; ++u) {
    const int i = tid + u * THREADS;
    sel[u] = i < gc * K ? idx[((long long)b * Hq + head0 + i / K) * K + i % K] : -1;
  }
  const int len = ctx[b];
  if (len < 1 || len > maxP * ps) {
    if (tid == 0) {
      flag_error(status, KV_ERR_BOUNDS);
      ucount[gbase] = 0;
    }
    pdl_trigger();
    return;
  }
  const int P = (len + ps - 1) / ps;
  const int nw = (P + 3) / 4;
  for (int i = tid; i < nw; i += THREADS) words[i] = 0u;
  __syncthreads();
  auto mark = [&](int i, int p) {
    if (p < 0) return;
    if (p >= P) {
      flag_error(status, KV_ERR_BOUNDS);
      return;
    }
    atomicOr(&words[p >> 2], (1u << (i / K)) << ((p & 3) * 8));
  };
#pragma unroll
  for (int u = 0; u < kSpec; ++u) mark(tid + u * THREADS, sel[u]);
  for (int i = tid + kSpec * THREADS; i < gc * K; i += THREADS)
    mark(i, idx[((long long)b * Hq + head0 + i / K) * K + i % K]);
  __syncthreads();
  pdl_trigger();
  const int per = (nw + THREADS - 1) / THREADS;  // words per thread
  const int lo = min(nw, tid * per), hi = min(nw, lo + per);
  uint32_t n = 0;
  for (int i = lo; i < hi; ++i) {
    uint32_t t = words[i];
    t |= t >> 4;
    t |= t >> 2;
    t |= t >> 1;
    n += __popc(t & 0x01010101u);  // pages of the word some head selected
  }
  uint32_t ni = n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, ni, off);
    if (lane >= off) ni += t;
  }
  if (lane == 31) wsum[warp] = ni;
  __syncthreads();
  const uint32_t ws = lane < WARPS ? wsum[lane] : 0u;
  uint32_t pos = __reduce_add_sync(0xFFFFFFFFu, lane < warp ? ws : 0u) + ni - n;
  const uint32_t tot = __reduce_add_sync(0xFFFFFFFFu, ws);
  for (int i = lo; i < hi; ++i) {
    const uint32_t w = words[i];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t m = (w >> (8 * e)) & 0xFFu;
      if (m != 0u) {
        if (pos < (uint32_t)umax) {
          upages[gbase * umax + pos] = 4 * i + e;
          umasks[gbase * umax + pos] = m;
        }
        ++pos;
      }
    }
  }
  if (tid == 0) ucount[gbase] = (int)min(tot, (uint32_t)umax);
}

}  // namespace kvs
