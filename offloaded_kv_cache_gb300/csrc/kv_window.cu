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
//   window_update_kernel  one CTA per group: need set, hits, lookahead
//                         eviction, slot assignment, fetch list, stats;
//   window_fetch_kernel   copies the fetch list's pages (K and V, the valid
//                         tokens) from the (host) cache into their slots;
// then the sparse attention runs over the window (page_slot override).
#include <algorithm>

#include "kv_select.cuh"

namespace kvs {
namespace {

// one CTA per group and few groups: a wide CTA shortens every pass
constexpr int kWinThreads = 1024;
constexpr int kWinWarps = kWinThreads / 32;

__device__ __forceinline__ uint32_t win_score_key(float s) {
  return key32(__float_as_uint(s + 0.0f));  // -0.0 ranks with +0.0
}

// Dynamic shared memory: need[maxP] bytes (0 none, 1 miss, 2 hit), then
// ekey[C] (eviction keys), then freed[C] (slots in ascending order).
__global__ void __launch_bounds__(kWinThreads)
    window_update_kernel(const int32_t *__restrict__ indices, const float *__restrict__ scores,
                         const int32_t *__restrict__ ctx, int Hq, int Hkv, int ps, int maxP,
                         int K, int C, int32_t *slot_page, int32_t *page_slot,
                         int32_t *fetch_page, int32_t *fetch_slot, int32_t *fetch_count,
                         int32_t *stats, int *status) {
  pdl_wait();
  extern __shared__ uint8_t wsm[];
  uint8_t *need = wsm;
  uint32_t *ekey = reinterpret_cast<uint32_t *>(wsm + ((maxP + 15) & ~15));
  int32_t *freed = reinterpret_cast<int32_t *>(ekey + C);
  __shared__ RadixScratch sc;
  __shared__ int s_hit, s_free, s_cand, s_need;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long g = blockIdx.x;
  const int b = (int)(g / Hkv), kvh = (int)(g % Hkv);
  const int G = Hq / Hkv;
  int32_t *sp = slot_page + g * C;
  int32_t *pslot = page_slot + g * maxP;
  const int len = ctx[b];
  if (len < 1 || len > maxP * ps) {
    if (tid == 0) {
      flag_error(status, KV_ERR_BOUNDS);
      fetch_count[g] = 0;
    }
    return;
  }
  const int P = (len + ps - 1) / ps;

  // need set of the group's G query heads
  for (int i = tid; i < (maxP + 3) / 4; i += kWinThreads) reinterpret_cast<uint32_t *>(need)[i] = 0u;
  if (tid == 0) s_hit = s_free = s_cand = s_need = 0;
  __syncthreads();
  for (int i = tid; i < G * K; i += kWinThreads) {
    const int p = indices[((long long)b * Hq + (long long)kvh * G) * K + i];
    if (p >= 0 && p < P) need[p] = 1;
  }
  __syncthreads();

  // classify the slots: free, hit (need -> 2), or an eviction candidate
  // keyed by ~score so that the radix select's "largest" is the lowest score
  int hit = 0, fre = 0, cand = 0;
  for (int s = tid; s < C; s += kWinThreads) {
    const int p = sp[s];
    uint32_t key = 0u;  // not a candidate: below every candidate's key
    if (p < 0 || p >= maxP) {
      ++fre;
    } else if (p < P && need[p]) {
      need[p] = 2;
      ++hit;
    } else {
      float m = -INFINITY;  // stale pages (at or past P) go first
      if (p < P) {
        for (int h = 0; h < G; ++h)
          m = fmaxf(m, scores[((long long)b * Hq + (long long)kvh * G + h) * maxP + p]);
      }
      key = ~win_score_key(m);
      ++cand;
    }
    ekey[s] = key;
  }
  if (hit) atomicAdd(&s_hit, hit);
  if (fre) atomicAdd(&s_free, fre);
  if (cand) atomicAdd(&s_cand, cand);
  __syncthreads();
  int nn = 0;
  for (int p = tid; p < P; p += kWinThreads) nn += need[p] != 0;
  if (nn) atomicAdd(&s_need, nn);
  __syncthreads();
  const int n_need = s_need, n_hit = s_hit, n_free = s_free, n_cand = s_cand;
  const int n_miss = n_need - n_hit;
  const int n_evict = max(0, n_miss - n_free);
  if (n_need > C || n_evict > n_cand) {  // the host checks C; never reached
    if (tid == 0) {
      flag_error(status, KV_ERR_BOUNDS);
      fetch_count[g] = 0;
    }
    return;
  }

  // lookahead eviction: the n_evict lowest-scored candidates, ties to the
  // lower slot; their pages leave the map and their slots become free
  auto key_at = [&](int s) -> uint32_t { return ekey[s]; };
  if (n_evict > 0) {
    const RadixSel sel = radix_select_top<kWinThreads>(key_at, C, n_evict, sc);
    radix_emit<kWinThreads>(key_at, C, sel, sc, [&](long long, int s) {
      pslot[sp[s]] = -1;
      sp[s] = -1;
    });
    __syncthreads();
  }
  pdl_trigger();

  // freed slots (free or evicted) in ascending order
  {
    const int seg = ((C + kWinWarps - 1) / kWinWarps + 31) / 32 * 32;
    const int lo = warp * seg, hi = min(C, lo + seg);
    unsigned long long cnt = 0;
    for (int s0 = lo; s0 < hi; s0 += 32) {
      const int s = s0 + lane;
      cnt += __popc(__ballot_sync(0xFFFFFFFFu, s < hi && sp[s] < 0));
    }
    unsigned long long tot;
    unsigned long long pos = warp_bases64<kWinWarps>(cnt, sc.wsum, &tot);
    for (int s0 = lo; s0 < hi; s0 += 32) {
      const int s = s0 + lane;
      const bool f = s < hi && sp[s] < 0;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, f);
      if (f) freed[pos + __popc(bal & ((1u << lane) - 1u))] = s;
      pos += __popc(bal);
    }
  }
  __syncthreads();

  // misses in ascending page order take the freed slots in ascending order;
  // the fetch list holds the misses and a hit on the growing last page
  {
    const int seg = ((P + kWinWarps - 1) / kWinWarps + 31) / 32 * 32;
    const int lo = warp * seg, hi = min(P, lo + seg);
    unsigned long long cnt = 0;  // misses (low half), fetches (high half)
    for (int p0 = lo; p0 < hi; p0 += 32) {
      const int p = p0 + lane;
      const int nd = p < hi ? need[p] : 0;
      cnt += __popc(__ballot_sync(0xFFFFFFFFu, nd == 1));
      cnt += (unsigned long long)__popc(
                 __ballot_sync(0xFFFFFFFFu, nd == 1 || (nd == 2 && p == P - 1)))
             << 32;
    }
    unsigned long long tot;
    unsigned long long base = warp_bases64<kWinWarps>(cnt, sc.wsum, &tot);
    long long mb = (long long)(base & 0xFFFFFFFFull), fb = (long long)(base >> 32);
    const unsigned lt = (1u << lane) - 1u;
    for (int p0 = lo; p0 < hi; p0 += 32) {
      const int p = p0 + lane;
      const int nd = p < hi ? need[p] : 0;
      const bool miss = nd == 1, fetch = miss || (nd == 2 && p == P - 1);
      const unsigned mbal = __ballot_sync(0xFFFFFFFFu, miss);
      const unsigned fbal = __ballot_sync(0xFFFFFFFFu, fetch);
      if (fetch) {
        int slot;
        if (miss) {
          slot = freed[mb + __popc(mbal & lt)];
          sp[slot] = p;
          pslot[p] = slot;
        } else {
          slot = pslot[p];
        }
        const long long f = fb + __popc(fbal & lt);
        fetch_page[g * C + f] = p;
        fetch_slot[g * C + f] = slot;
      }
      mb += __popc(mbal);
      fb += __popc(fbal);
    }
    if (tid == 0) {
      fetch_count[g] = (int)(tot >> 32);
      if (stats) {
        stats[g * 4 + 0] = n_need;
        stats[g * 4 + 1] = n_hit;
        stats[g * 4 + 2] = (int)(tot >> 32);
        stats[g * 4 + 3] = n_evict;
      }
    }
  }
}

// Copies each fetch-list page of each group: the page's valid tokens of one
// kv head, K then V, from the (host-mapped) cache into the window slot.  CTAs
// stride over the entries of their group; each thread moves 16-byte chunks,
// several loads in flight.
template <int CH>  // 16-byte chunks per row
__global__ void __launch_bounds__(256)
    window_fetch_kernel(const uint4 *__restrict__ k_src, const uint4 *__restrict__ v_src,
                        uint4 *__restrict__ k_win, uint4 *__restrict__ v_win,
                        const int32_t *__restrict__ bt, const int32_t *__restrict__ ctx,
                        const int32_t *__restrict__ fetch_page,
                        const int32_t *__restrict__ fetch_slot,
                        const int32_t *__restrict__ fetch_count, int Hkv, int ps, int maxP,
                        int C, long long nphys, int *status) {
  pdl_wait();
  const long long g = blockIdx.y;
  const int b = (int)(g / Hkv), kvh = (int)(g % Hkv);
  const int count = fetch_count[g];
  const int len = ctx[b];
  for (int e = blockIdx.x; e < count; e += gridDim.x) {
    const int p = fetch_page[g * C + e];
    const int slot = fetch_slot[g * C + e];
    if (p < 0 || p * ps >= len || slot < 0 || slot >= C) {
      if (threadIdx.x == 0) flag_error(status, KV_ERR_BOUNDS);
      continue;
    }
    const long long phys = bt[(long long)b * maxP + p];
    if (phys < 0 || phys >= nphys) {
      if (threadIdx.x == 0) flag_error(status, KV_ERR_BOUNDS);
      continue;
    }
    const int n = min(ps, len - p * ps) * CH;  // chunks of the valid rows
    const long long src = (phys * Hkv + kvh) * ps * CH;
    const long long dst = (((long long)b * C + slot) * Hkv + kvh) * ps * CH;
    int i = threadIdx.x;
    for (; i + 256 < n; i += 512) {
      const uint4 k0 = k_src[src + i], k1 = k_src[src + i + 256];
      const uint4 v0 = v_src[src + i], v1 = v_src[src + i + 256];
      k_win[dst + i] = k0;
      k_win[dst + i + 256] = k1;
      v_win[dst + i] = v0;
      v_win[dst + i + 256] = v1;
    }
    for (; i < n; i += 256) {
      k_win[dst + i] = k_src[src + i];
      v_win[dst + i] = v_src[src + i];
    }
  }
  pdl_trigger();
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

cudaError_t launch_window_update(const int32_t *indices, const float *scores, const int32_t *ctx,
                                 int B, int Hq, int Hkv, int ps, int maxP, int K, int C,
                                 int32_t *slot_page, int32_t *page_slot, int32_t *fetch_page,
                                 int32_t *fetch_slot, int32_t *fetch_count, int32_t *stats,
                                 int *status, cudaStream_t st) {
  const size_t smem = window_update_smem(maxP, C);
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && (dev < 0 || dev >= 64 || !attr_done[dev])) {
    cudaError_t e = cudaFuncSetAttribute(window_update_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  return launch_pdl(window_update_kernel, dim3((unsigned)((long long)B * Hkv)), dim3(kWinThreads),
                    smem, st, indices, scores, ctx, Hq, Hkv, ps, maxP, K, C, slot_page, page_slot,
                    fetch_page, fetch_slot, fetch_count, stats, status);
}

cudaError_t launch_window_fetch(int dtype, const void *k_src, const void *v_src, void *k_win,
                                void *v_win, const int32_t *bt, const int32_t *ctx,
                                const int32_t *fetch_page, const int32_t *fetch_slot,
                                const int32_t *fetch_count, int B, int Hkv, int ps, int maxP,
                                int C, long long nphys, int blocks_per_group, int *status,
                                cudaStream_t st) {
  const dim3 grid((unsigned)blocks_per_group, (unsigned)((long long)B * Hkv));
  auto kern = dtype == KV_F32 ? window_fetch_kernel<32> : window_fetch_kernel<16>;
  return launch_pdl(kern, grid, dim3(256), 0, st, static_cast<const uint4 *>(k_src),
                    static_cast<const uint4 *>(v_src), static_cast<uint4 *>(k_win),
                    static_cast<uint4 *>(v_win), bt, ctx, fetch_page, fetch_slot, fetch_count,
                    Hkv, ps, maxP, C, nphys, status);
}

cudaError_t launch_fill(int32_t *p, long long n, int32_t v, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)std::min<long long>((n + 255) / 256, 4096);
  return launch_pdl(fill_kernel, dim3(blocks), dim3(256), 0, st, p, n, v);
}

}  // namespace kvs
