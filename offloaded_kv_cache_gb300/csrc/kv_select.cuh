// kv_select.cuh -- block-wide selection helpers shared by the top-K page
// selection and the page window's eviction: a radix select of the k largest
// 32-bit keys (ties to the lower index) and the in-order compaction of the
// selected indices.
#pragma once
#include "kv_internal.cuh"

namespace kvs {

// Exclusive prefix sum over the warps of the block of one 64-bit value per
// warp (lane 0's argument counts); returns the warp's base, *total the sum.
// Two block barriers; `wsum` holds one slot per warp.
template <int WARPS>
__device__ __forceinline__ unsigned long long warp_bases64(unsigned long long v,
                                                           unsigned long long *wsum,
                                                           unsigned long long *total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) wsum[warp] = v;
  __syncthreads();
  unsigned long long base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) {
    const unsigned long long t = wsum[w];
    base += w < warp ? t : 0ull;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return base;
}

// Threshold of a radix select: the selected keys are those whose masked
// value beats `prefix`, plus -- all of them when all_taken, else the first
// krem in index order -- those equal to it.
struct RadixSel {
  uint32_t prefix, pmask;
  int krem;
  bool all_taken;
};

// Shared scratch of the helpers below (one per block).
struct RadixScratch {
  uint32_t hist[256];
  unsigned long long wsum[32];
  uint32_t digit;
  int krem, all;
};

// The k (1 <= k <= n) largest of key_at(0 .. n-1), 8 bits per pass from the
// top: a shared-memory histogram whose threshold digit one warp finds with a
// shuffle scan; stops early once every key of the threshold bin is taken.
// THREADS: 256, 512 or 1024 (the block size).
template <int THREADS, class KeyAt>
__device__ __forceinline__ RadixSel radix_select_top(KeyAt key_at, int n, int k,
                                                     RadixScratch &sc) {
  static_assert(THREADS % 256 == 0 && THREADS <= 1024, "256, 512 or 1024 threads");
  const int tid = threadIdx.x;
  RadixSel r{0u, 0u, k, false};
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) sc.hist[tid] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += THREADS) {
      const uint32_t key = key_at(i);
      if ((key & r.pmask) == r.prefix) atomicAdd(&sc.hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits 255-8l .. 248-8l, scanned from the top
      int c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = (int)sc.hist[255 - 8 * tid - j];
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
    r.prefix |= sc.digit << shift;
    r.pmask |= 255u << shift;
    r.krem = sc.krem;
    if (sc.all) {
      r.all_taken = true;  // every key with this prefix is selected
      break;
    }
  }
  return r;
}

// Calls emit(pos, i) for every selected index i, pos = its rank in index
// order (0 .. k-1).  The indices are split into one contiguous segment per
// warp; each warp walks its segment 32 at a time and places its selected
// indices with ballots after one block scan of the per-warp counts.
template <int THREADS, class KeyAt, class Emit>
__device__ __forceinline__ void radix_emit(KeyAt key_at, int n, const RadixSel &r,
                                           RadixScratch &sc, Emit emit) {
  constexpr int WARPS = THREADS / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = ((n + WARPS - 1) / WARPS + 31) / 32 * 32;  // indices per warp
  const int lo = warp * seg, hi = min(n, lo + seg);
  uint32_t gt_n = 0, eq_n = 0;
  for (int i0 = lo; i0 < hi; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < hi ? key_at(i) & r.pmask : 0u;
    gt_n += __popc(__ballot_sync(0xFFFFFFFFu, i < hi && key > r.prefix));
    eq_n += __popc(__ballot_sync(0xFFFFFFFFu, i < hi && key == r.prefix));
  }
  unsigned long long tot;
  const unsigned long long base =
      warp_bases64<WARPS>(((unsigned long long)eq_n << 32) | gt_n, sc.wsum, &tot);
  long long gt_b = (long long)(base & 0xFFFFFFFFull);
  long long eq_b = (long long)(base >> 32);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int i0 = lo; i0 < hi; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < hi ? key_at(i) & r.pmask : 0u;
    const unsigned gtb = __ballot_sync(0xFFFFFFFFu, i < hi && key > r.prefix);
    const unsigned eqb = __ballot_sync(0xFFFFFFFFu, i < hi && key == r.prefix);
    const long long my_gt = gt_b + __popc(gtb & lt_mask);
    const long long my_eq = eq_b + __popc(eqb & lt_mask);
    const bool is_gt = (gtb >> lane) & 1u, is_eq = (eqb >> lane) & 1u;
    const bool sel = is_gt || (is_eq && (r.all_taken || my_eq < r.krem));
    if (sel) emit(my_gt + (r.all_taken ? my_eq : min(my_eq, (long long)r.krem)), i);
    gt_b += __popc(gtb);
    eq_b += __popc(eqb);
  }
}

}  // namespace kvs
