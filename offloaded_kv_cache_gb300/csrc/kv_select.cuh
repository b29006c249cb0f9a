// kv_select.cuh -- block-wide selection helpers for the page window's
// eviction: a radix select of the k largest 32-bit keys (ties to the lower
// index) and the in-order compaction of the selected indices.  (The top-K
// kernel keeps its own specialised copy of the same select.)
#pragma once
#include "kv_internal.cuh"

namespace kvs {

// Threshold of a radix select: the selected keys are those whose masked
// value beats `prefix`, plus the first krem in index order of those equal to
// it (when the last pass took its whole bin, krem is their count).
struct RadixSel {
  uint32_t prefix, pmask;
  int krem;
};

// Shared scratch of the helpers below (one per block).
struct RadixScratch {
  uint32_t hist[2][256];
  unsigned long long wsum[32];
  uint32_t digit;
  int krem, all;
};

// The k (1 <= k <= n) largest of key_at(0 .. n-1), given that those k keys
// lie in [lo, hi] and no key exceeds hi (lo = 0, hi = ~0u when nothing is
// known).  8 bits per pass from the highest bit where lo and hi differ: the
// bits above it are common to every key that can be selected.  Each pass
// builds a shared-memory histogram (double-buffered, so two block barriers
// per pass) whose threshold digit one warp finds with a shuffle scan; stops
// early once every key of the threshold bin is taken.
// THREADS: 256, 512 or 1024 (the block size).
template <int THREADS, class KeyAt>
__device__ __forceinline__ RadixSel radix_select_top(KeyAt key_at, int n, int k, uint32_t lo,
                                                     uint32_t hi, RadixScratch &sc) {
  static_assert(THREADS % 256 == 0 && THREADS <= 1024, "256, 512 or 1024 threads");
  const int tid = threadIdx.x;
  const uint32_t diff = lo ^ hi;
  const int top = diff ? 31 - __clz(diff) : -1;
  RadixSel r;
  r.pmask = top >= 31 ? 0u : (0xFFFFFFFFu << (top + 1));
  r.prefix = hi & r.pmask;
  r.krem = k;
  if (tid < 256) sc.hist[0][tid] = 0;
  __syncthreads();
  int pass = 0;
#pragma unroll 1
  for (int hb = top; hb >= 0; hb -= 8, ++pass) {
    const int lb = max(hb - 7, 0);
    const uint32_t dmask = (1u << (hb - lb + 1)) - 1u;
    uint32_t *h = sc.hist[pass & 1];
    if (tid < 256) sc.hist[(pass + 1) & 1][tid] = 0;  // the next pass's histogram
    for (int i = tid; i < n; i += THREADS) {
      const uint32_t key = key_at(i);
      if ((key & r.pmask) == r.prefix) atomicAdd(&h[(key >> lb) & dmask], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits 255-8l .. 248-8l, scanned from the top
      int c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = (int)h[255 - 8 * tid - j];
        sum += c[j];
      }
      int incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (tid >= off) incl += t;
      }
      int above = incl - sum;
      if (above < r.krem && r.krem <= incl) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (above + c[j] >= r.krem) {
            sc.digit = (uint32_t)(255 - 8 * tid - j);
            sc.krem = r.krem - above;
            sc.all = (above + c[j] == r.krem) ? 1 : 0;
            break;
          }
          above += c[j];
        }
      }
    }
    __syncthreads();
    r.prefix |= sc.digit << lb;
    r.pmask |= dmask << lb;
    r.krem = sc.krem;
    if (sc.all) break;  // every key with this prefix is selected
  }
  return r;
}

// Calls emit(pos, i) for every selected index i, pos = its rank in index
// order (0 .. k-1).  Each thread owns a run of consecutive indices, counts
// its keys above and at the threshold, and after one block scan of those
// counts emits its selected indices in order.  One block barrier.
template <int THREADS, class KeyAt, class Emit>
__device__ __forceinline__ void radix_emit(KeyAt key_at, int n, const RadixSel &r,
                                           RadixScratch &sc, Emit emit) {
  constexpr int WARPS = THREADS / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per = (n + THREADS - 1) / THREADS;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  uint32_t gt_n = 0, eq_n = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = key_at(i) & r.pmask;
    gt_n += key > r.prefix;
    eq_n += key == r.prefix;
  }
  uint32_t gi = gt_n, ei = eq_n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t tg = __shfl_up_sync(0xFFFFFFFFu, gi, off);
    const uint32_t te = __shfl_up_sync(0xFFFFFFFFu, ei, off);
    if (lane >= off) {
      gi += tg;
      ei += te;
    }
  }
  if (lane == 31) sc.wsum[warp] = ((unsigned long long)ei << 32) | gi;
  __syncthreads();
  const unsigned long long t = lane < WARPS ? sc.wsum[lane] : 0ull;
  const bool before = lane < warp;
  int gt_b = (int)(__reduce_add_sync(0xFFFFFFFFu, before ? (uint32_t)t : 0u) + gi - gt_n);
  int eq_b = (int)(__reduce_add_sync(0xFFFFFFFFu, before ? (uint32_t)(t >> 32) : 0u) + ei - eq_n);
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = key_at(i) & r.pmask;
    const bool is_gt = key > r.prefix, is_eq = key == r.prefix;
    if (is_gt || (is_eq && eq_b < r.krem)) emit(gt_b + min(eq_b, r.krem), i);
    gt_b += is_gt;
    eq_b += is_eq;
  }
}

}  // namespace kvs
