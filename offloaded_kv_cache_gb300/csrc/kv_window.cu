// kv_window.cu -- the GPU-resident window of critical pages.
//
// KVDrive (A Holistic Multi-Tier KV Cache Management System for Long-Context
// LLM Inference), section 5.1 "Sliding window with lookahead eviction": the
// GPU keeps recently critical KV entries; each decode step fetches from host
// memory only the critical entries the window lacks, and evicts the entries
// with the lowest attention score of the current step.  Section 3, Finding 1
// sizes the window in multiples of the per-step budget; section 6.3: with
// most critical entries served from the window, attention stays on the GPU.
//
// One group per (sequence b, kv head) owns C slots of the cache arrays
// [B*C][Hkv][ps][d]: slot s of group (b, kvh) is page b*C + s, kv head kvh,
// so the attention kernel addresses the window exactly like a K/V cache.
//   window_step_kernel  one CTA per group: need set, hits, lookahead
//                       eviction, slot assignment, fetch bits, stats; and,
//                       in the same launch, one CTA per head chunk building
//                       the attention's union lists;
// then the window instantiation of the sparse attention reads the hits from
// the window and the fetched pages from the (host) cache, and stores each
// fetched page's valid tokens into its slot as it goes.
#include <algorithm>

#include "kv_select.cuh"
#include "kv_launch.h"
#include "kv_union.cuh"

namespace kvs {
namespace {

// one CTA per group and few groups: a wide CTA shortens every pass
// (1024 threads measured faster than 512 and 256)
constexpr int kWinThreads = 1024;
constexpr int kWinWarps = kWinThreads / 32;

__device__ __forceinline__ uint32_t win_score_key(float s) {
  return key32(__float_as_uint(s + 0.0f));  // -0.0 ranks with +0.0
}

// Slot keys: a needed page's slot (a hit) 0, a free slot 1, else the eviction
// candidate's key ~key(score), at least ~key(+inf) = 0x007FFFFF, so that the
// largest keys are the lowest scores and hits and free slots never rank
// among the candidates.
constexpr uint32_t kSlotHit = 0u, kSlotFree = 1u;

// Consecutive pages a thread owns in the page passes: 4, 8, 16 or 32 (so
// that a fetch-bit word is shared by whole lanes), else a multiple of 32.
__device__ __forceinline__ int page_run(int P) {
  const int per = (P + kWinThreads - 1) / kWinThreads;
  if (per <= 4) return 4;
  if (per <= 32) return 1 << (32 - __clz(per - 1));
  return (per + 31) & ~31;
}

// The window update of group g = (b, kv head), one CTA.  Shared memory at
// wsm: need[maxP] bytes (0 none, 1 miss, 2 hit), then skey[C] (slot keys),
// then aux[C] (each slot's page until the eviction, then the freed slots in
// ascending order).
__device__ __forceinline__ void update_group(const int32_t *indices,
                                             const float *scores,
                                             const int32_t *ctx, int Hq, int Hkv,
                                             int ps, int maxP, int K, int C, int32_t *slot_page,
                                             int32_t *page_slot, uint32_t *fetch_bits,
                                             int32_t *stats, int *status, long long g,
                                             uint8_t *wsm) {
  uint8_t *need = wsm;
  uint32_t *skey = reinterpret_cast<uint32_t *>(wsm + ((maxP + 15) & ~15));
  int32_t *aux = reinterpret_cast<int32_t *>(skey + C);
  __shared__ RadixScratch sc;
  __shared__ uint32_t wred[9][kWinWarps];  // per-warp partials; row 8: the freed scan
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = (int)(g / Hkv), kvh = (int)(g % Hkv);
  const int G = Hq / Hkv;
  int32_t *sp = slot_page + g * C;
  int32_t *pslot = page_slot + g * maxP;
  const int W = (maxP + 31) / 32;  // fetch-bit words per group
  uint32_t *fbits = fetch_bits + g * W;
  // the first selections and slot pages load together with the context length
  const int32_t *sel = indices + ((long long)b * Hq + (long long)kvh * G) * K;
  constexpr int kSpec = 4;
  int32_t sel_r[kSpec], sp_r[kSpec];
#pragma unroll
  for (int u = 0; u < kSpec; ++u) {
    const int i = tid + u * kWinThreads;
    sel_r[u] = i < G * K ? sel[i] : -1;
    sp_r[u] = i < C ? sp[i] : -1;
  }
  const int len = ctx[b];
  if (len < 1 || len > maxP * ps) {
    if (tid == 0) flag_error(status, KV_ERR_BOUNDS);
    for (int w = tid; w < W; w += kWinThreads) fbits[w] = 0u;
    return;
  }
  const int P = (len + ps - 1) / ps;

  // need set of the group's G query heads
  for (int i = tid; i < (maxP + 3) / 4; i += kWinThreads) reinterpret_cast<uint32_t *>(need)[i] = 0u;
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kSpec; ++u)
    if (sel_r[u] >= 0 && sel_r[u] < P) need[sel_r[u]] = 1;
  for (int i = tid + kSpec * kWinThreads; i < G * K; i += kWinThreads) {
    const int p = sel[i];
    if (p >= 0 && p < P) need[p] = 1;
  }
  __syncthreads();

  // classify the slots: free, hit (need -> 2), or an eviction candidate
  uint32_t hit = 0, fre = 0, cand = 0, cmin = 0xFFFFFFFFu, cmax = 0u;
  for (int s = tid, u = 0; s < C; s += kWinThreads, ++u) {
    int p = 0;
#pragma unroll
    for (int v = 0; v < kSpec; ++v)
      if (u == v) p = sp_r[v];  // static register indexing
    if (u >= kSpec) p = sp[s];
    uint32_t key;
    if (p < 0 || p >= maxP) {
      key = kSlotFree;
      ++fre;
    } else if (p < P && need[p]) {
      need[p] = 2;
      key = kSlotHit;
      ++hit;
    } else {
      float m = -INFINITY;  // stale pages (at or past P) go first
      if (p < P) {
        for (int h = 0; h < G; ++h)
          m = fmaxf(m, scores[((long long)b * Hq + (long long)kvh * G + h) * maxP + p]);
      }
      key = ~win_score_key(m);
      ++cand;
      cmin = min(cmin, key);
      cmax = max(cmax, key);
    }
    skey[s] = key;
    aux[s] = p;
  }
  __syncthreads();  // need[] is final

  // one pass over this thread's pages: needed, misses (scanned), fetches
  const int per = page_run(P);
  const int lo = min(P, tid * per), hi = min(P, lo + per);
  uint32_t nn = 0, nm = 0, nf = 0;
  for (int p = lo; p < hi; p += 4) {  // need[] is zero past P
    const uint32_t w4 = *reinterpret_cast<const uint32_t *>(need + p);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t v = (w4 >> (8 * e)) & 255u;
      nn += v != 0u;
      nm += v == 1u;
      nf += v == 1u || (v == 2u && p + e == P - 1);
    }
  }
  uint32_t mi = nm;  // inclusive scan of the misses over the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, mi, off);
    if (lane >= off) mi += t;
  }
  {
    const uint32_t v0 = __reduce_add_sync(0xFFFFFFFFu, nn);
    const uint32_t v1 = __reduce_add_sync(0xFFFFFFFFu, nf);
    const uint32_t v2 = __reduce_add_sync(0xFFFFFFFFu, hit);
    const uint32_t v3 = __reduce_add_sync(0xFFFFFFFFu, fre);
    const uint32_t v4 = __reduce_add_sync(0xFFFFFFFFu, cand);
    const uint32_t v5 = __reduce_min_sync(0xFFFFFFFFu, cmin);
    const uint32_t v6 = __reduce_max_sync(0xFFFFFFFFu, cmax);
    if (lane == 31) {
      wred[0][warp] = mi;
      wred[1][warp] = v0; wred[2][warp] = v1; wred[3][warp] = v2;
      wred[4][warp] = v3; wred[5][warp] = v4; wred[6][warp] = v5; wred[7][warp] = v6;
    }
  }
  __syncthreads();
  const bool wl = lane < kWinWarps;
  const uint32_t wmiss = wl ? wred[0][lane] : 0u;
  int miss_b = (int)(__reduce_add_sync(0xFFFFFFFFu, lane < warp ? wmiss : 0u) + mi - nm);
  const int n_need = (int)__reduce_add_sync(0xFFFFFFFFu, wl ? wred[1][lane] : 0u);
  const int n_fetch = (int)__reduce_add_sync(0xFFFFFFFFu, wl ? wred[2][lane] : 0u);
  const int n_hit = (int)__reduce_add_sync(0xFFFFFFFFu, wl ? wred[3][lane] : 0u);
  const int n_free = (int)__reduce_add_sync(0xFFFFFFFFu, wl ? wred[4][lane] : 0u);
  const int n_cand = (int)__reduce_add_sync(0xFFFFFFFFu, wl ? wred[5][lane] : 0u);
  cmin = __reduce_min_sync(0xFFFFFFFFu, wl ? wred[6][lane] : 0xFFFFFFFFu);
  cmax = __reduce_max_sync(0xFFFFFFFFu, wl ? wred[7][lane] : 0u);
  const int n_miss = n_need - n_hit;
  const int n_evict = max(0, n_miss - n_free);
  if (n_need > C || n_evict > n_cand) {  // the host checks C; never reached
    if (tid == 0) flag_error(status, KV_ERR_BOUNDS);
    for (int w = tid; w < W; w += kWinThreads) fbits[w] = 0u;
    return;
  }

  // lookahead eviction: the n_evict lowest-scored candidates (the largest
  // keys, all in [cmin, cmax]), ties to the lower slot; their pages leave
  // the map and their slots become free
  if (n_evict > 0) {
    auto key_at = [&](int s) -> uint32_t { return skey[s]; };
    const RadixSel sel = radix_select_top<kWinThreads>(key_at, C, n_evict, cmin, cmax, sc);
    radix_emit<kWinThreads>(key_at, C, sel, sc, [&](int, int s) {
      pslot[aux[s]] = -1;
      sp[s] = -1;
      skey[s] = kSlotFree;
    });
    __syncthreads();
  }
  pdl_trigger();

  // freed slots (free or evicted) in ascending order into aux[]
  {
    const int cper = (C + kWinThreads - 1) / kWinThreads;
    const int clo = min(C, tid * cper), chi = min(C, clo + cper);
    uint32_t nfr = 0;
    for (int s = clo; s < chi; ++s) nfr += skey[s] == kSlotFree;
    uint32_t fi = nfr;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, fi, off);
      if (lane >= off) fi += t;
    }
    if (lane == 31) wred[8][warp] = fi;
    __syncthreads();
    int pos = (int)(__reduce_add_sync(0xFFFFFFFFu, lane < warp && wl ? wred[8][lane] : 0u) + fi -
                    nfr);
    for (int s = clo; s < chi; ++s)
      if (skey[s] == kSlotFree) aux[pos++] = s;
  }
  __syncthreads();

  // misses in ascending page order take the freed slots in ascending order;
  // the fetch bits mark the misses and a hit on the growing last page (the
  // attention reads those from the cache and refreshes their slots)
  for (int w = (P + 31) / 32 + tid; w < W; w += kWinThreads) fbits[w] = 0u;
  {
    const int plo = tid * per;  // unclipped: the fetch-bit word of this run
    uint32_t bits = 0u;         // this run's fetch bits (per <= 32), or one word's
    for (int p = lo; p < hi; p += 4) {
      const uint32_t w4 = *reinterpret_cast<const uint32_t *>(need + p);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t v = (w4 >> (8 * e)) & 255u;
        const int q = p + e;
        if (v == 1u) {
          const int slot = aux[miss_b++];
          sp[slot] = q;
          pslot[q] = slot;
        }
        if (v == 1u || (v == 2u && q == P - 1)) bits |= 1u << (q & 31);
      }
      if (per > 32 && ((p + 4) & 31) == 0) {  // a run of whole words
        fbits[(p >> 5)] = bits;
        bits = 0u;
      }
    }
    if (per <= 32) {
      // the lanes of one word OR their bits; its first lane writes it
      for (int off = 1; off < 32 / per; off <<= 1) bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, off);
      if (plo < P && (plo & 31) == 0) fbits[plo >> 5] = bits;
    } else if (hi > lo && (((hi + 3) & ~3) & 31) != 0) {
      fbits[(hi - 1) >> 5] = bits;  // the run's last word, not yet written
    }
  }
  if (tid == 0 && stats) {
    stats[g * 4 + 0] = n_need;
    stats[g * 4 + 1] = n_hit;
    stats[g * 4 + 2] = n_fetch;
    stats[g * 4 + 3] = n_evict;
  }
}

// One launch, two roles: CTAs [0, n_update) run the window update of group
// blockIdx.x; the others build the union lists of the attention's head
// chunks (u = blockIdx.x - n_update: sequence u / groups, chunk group
// u % groups).  Both only read the selection and they write disjoint
// outputs, so they run side by side instead of one after the other.
__global__ void __launch_bounds__(kWinThreads)
    window_step_kernel(const int32_t *indices, const float *scores,
                       const int32_t *ctx, int Hq, int Hkv, int ps, int maxP, int K,
                       int C, int32_t *slot_page, int32_t *page_slot, uint32_t *fetch_bits,
                       int32_t *stats, int *status, int n_update, int G, int gc, int umax,
                       int groups, int32_t *upages, uint32_t *umasks, int32_t *ucount) {
  pdl_wait();
  extern __shared__ uint8_t wsm[];
  if ((int)blockIdx.x < n_update) {
    update_group(indices, scores, ctx, Hq, Hkv, ps, maxP, K, C, slot_page, page_slot, fetch_bits,
                 stats, status, (long long)blockIdx.x, wsm);
  } else {
    __shared__ uint32_t uwsum[kWinWarps];
    const int u = (int)blockIdx.x - n_update;
    union_group<kWinThreads>(indices, ctx, Hq, G, gc, ps, maxP, K, umax, upages, umasks, ucount,
                             status, u % groups, u / groups, groups,
                             reinterpret_cast<uint32_t *>(wsm), uwsum);
  }
}

__global__ void fill_kernel(int32_t *p, long long n, int32_t v) {
  pdl_wait();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    p[i] = v;
}

}  // namespace

size_t window_update_smem(int maxP, int C) {
  return (size_t)((maxP + 15) & ~15) + (size_t)C * 8;
}

cudaError_t launch_window_step(const int32_t *indices, const float *scores, const int32_t *ctx,
                               int B, int Hq, int Hkv, int ps, int maxP, int K, int C,
                               int32_t *slot_page, int32_t *page_slot, uint32_t *fetch_bits,
                               int32_t *stats, int gc, int umax, int32_t *upages,
                               uint32_t *umasks, int32_t *ucount, int *status, cudaStream_t st) {
  const size_t smem = std::max(window_update_smem(maxP, C), (size_t)((maxP + 3) / 4) * 4);
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && (dev < 0 || dev >= 64 || !attr_done[dev])) {
    cudaError_t e = cudaFuncSetAttribute(window_step_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  const int G = Hq / Hkv;
  const int groups = Hkv * (G / gc);
  const int n_update = B * Hkv;
  const unsigned blocks = (unsigned)(n_update + B * groups);
  return launch_pdl(window_step_kernel, dim3(blocks), dim3(kWinThreads), smem, st, indices,
                    scores, ctx, Hq, Hkv, ps, maxP, K, C, slot_page, page_slot, fetch_bits, stats,
                    status, n_update, G, gc, umax, groups, upages, umasks, ucount);
}

cudaError_t launch_fill(int32_t *p, long long n, int32_t v, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)std::min<long long>((n + 255) / 256, 4096);
  return launch_pdl(fill_kernel, dim3(blocks), dim3(256), 0, st, p, n, v);
}

}  // namespace kvs
