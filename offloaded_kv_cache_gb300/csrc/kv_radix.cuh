// kv_radix.cuh -- block-wide radix select of the K largest 32-bit keys of a
// row, and the pass that emits the selected positions in ascending order.
// Used by the top-K kernel and by the fused selection kernel.
//
// KVDrive: A Holistic Multi-Tier KV Cache Management System for Long-Context
// LLM Inference, section 2.2: only the Top-K most important blocks are
// retrieved.  Equal keys at the threshold go to the lower position.
#pragma once

#include "kv_internal.cuh"

namespace kvs {

__device__ __forceinline__ uint32_t score_key(float s) {
  // +0.0f folds -0.0 into +0.0 so that equal scores compare equal
  return key32(__float_as_uint(s + 0.0f));
}

// Key of a forced page: above every score's key (+inf maps to 0xFF800000;
// 0xFFFFFFFF is a NaN's key, and scores are never NaN).
constexpr uint32_t kForcedKey = 0xFFFFFFFFu;

// Shared state of one select (the caller provides it in shared memory).
template <int THREADS>
struct RadixSmem {
  uint32_t hist[2][256];
  uint32_t wmin[THREADS / 32], wmax[THREADS / 32];
  unsigned long long wsum[THREADS / 32];
  uint32_t digit;
  int krem, all;
};

// Block-wide minimum and maximum of the threads' kmin / kmax.  Every thread
// gets both.  One block barrier.
template <int THREADS>
__device__ __forceinline__ void block_minmax(RadixSmem<THREADS> &sm, uint32_t &kmin,
                                             uint32_t &kmax) {
  constexpr int W = THREADS / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  if (lane == 0) {
    sm.wmin[warp] = kmin;
    sm.wmax[warp] = kmax;
  }
  __syncthreads();
  kmin = __reduce_min_sync(0xFFFFFFFFu, lane < W ? sm.wmin[lane] : 0xFFFFFFFFu);
  kmax = __reduce_max_sync(0xFFFFFFFFu, lane < W ? sm.wmax[lane] : 0u);
}

// The keff-th largest key of key_at(p), p < P, as a (prefix, pmask) pair: the
// selected keys are those whose masked bits exceed prefix, then the first
// krem (in position order) equal to it.  8 bits per pass, starting at the
// highest bit where kmin and kmax differ (the bits above it are common to
// every key, so a pass spent on them would select nothing), stopping as soon
// as every key of the threshold bin is taken.  Double-buffered histograms:
// two block barriers a pass.  sm.hist[0] must be zero, and visible to every
// thread, on entry.  THREADS >= 32.
template <int THREADS, class KeyAt>
__device__ __forceinline__ void radix_threshold(RadixSmem<THREADS> &sm, KeyAt key_at, int P,
                                                int keff, uint32_t kmin, uint32_t kmax,
                                                uint32_t &prefix, uint32_t &pmask, int &krem) {
  const int tid = threadIdx.x;
  const uint32_t diff = kmin ^ kmax;
  const int top = diff ? 31 - __clz(diff) : -1;
  pmask = top >= 31 ? 0u : (0xFFFFFFFFu << (top + 1));
  prefix = kmin & pmask;
  krem = keff;
  int pass = 0;
#pragma unroll 1
  for (int hb = top; hb >= 0; hb -= 8, ++pass) {
    const int lb = max(hb - 7, 0);
    const uint32_t dmask = (1u << (hb - lb + 1)) - 1u;
    uint32_t *h = sm.hist[pass & 1];
    for (int i = tid; i < 256; i += THREADS) sm.hist[(pass + 1) & 1][i] = 0;  // the next pass's
    for (int p = tid; p < P; p += THREADS) {
      const uint32_t k = key_at(p);
      if ((k & pmask) == prefix) atomicAdd(&h[(k >> lb) & dmask], 1u);
    }
    __syncthreads();
    if (tid < 32) {
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
      if (above < krem && krem <= incl) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (above + c[j] >= krem) {
            sm.digit = (uint32_t)(255 - 8 * tid - j);
            sm.krem = krem - above;
            sm.all = (above + c[j] == krem) ? 1 : 0;
            break;
          }
          above += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= sm.digit << lb;
    pmask |= dmask << lb;
    krem = sm.krem;
    if (sm.all) break;
  }
}

// The selected positions in ascending order: emit(rank, p) for each.  Each
// thread owns a run of consecutive positions (a multiple of 4, so that keys
// held in shared memory load 16 bytes at a time), counts its keys above and
// at the threshold, and after one block scan of those counts emits its
// selected positions in order.  skeys: the keys in shared memory (16-byte
// aligned), or nullptr to read them through key_at.  One block barrier.
template <int THREADS, class KeyAt, class Emit>
__device__ __forceinline__ void radix_emit(RadixSmem<THREADS> &sm, KeyAt key_at,
                                           const uint32_t *skeys, int P, uint32_t prefix,
                                           uint32_t pmask, int krem, Emit emit) {
  constexpr int W = THREADS / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per = ((P + THREADS - 1) / THREADS + 3) & ~3;
  const int lo = min(P, tid * per), hi = min(P, lo + per);
  auto load4 = [&](int p, uint32_t(&kk)[4]) {
    if (skeys != nullptr && p + 4 <= hi) {
      const uint4 v = *reinterpret_cast<const uint4 *>(skeys + p);
      kk[0] = v.x; kk[1] = v.y; kk[2] = v.z; kk[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) kk[e] = p + e < hi ? key_at(p + e) : 0u;
    }
  };
  uint32_t gt_n = 0, eq_n = 0;
  for (int p = lo; p < hi; p += 4) {
    uint32_t kk[4];
    load4(p, kk);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t k = kk[e] & pmask;
      const bool in = p + e < hi;
      gt_n += in && k > prefix;
      eq_n += in && k == prefix;
    }
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
  if (lane == 31) sm.wsum[warp] = ((unsigned long long)ei << 32) | gi;
  __syncthreads();
  const unsigned long long t = lane < W ? sm.wsum[lane] : 0ull;
  const bool before = lane < warp;
  int gt_b = (int)(__reduce_add_sync(0xFFFFFFFFu, before ? (uint32_t)t : 0u) + gi - gt_n);
  int eq_b =
      (int)(__reduce_add_sync(0xFFFFFFFFu, before ? (uint32_t)(t >> 32) : 0u) + ei - eq_n);
  for (int p = lo; p < hi; p += 4) {
    uint32_t kk[4];
    load4(p, kk);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t k = kk[e] & pmask;
      const bool in = p + e < hi;
      const bool is_gt = in && k > prefix, is_eq = in && k == prefix;
      if (is_gt || (is_eq && eq_b < krem)) emit(gt_b + min(eq_b, krem), p + e);
      gt_b += is_gt;
      eq_b += is_eq;
    }
  }
}

}  // namespace kvs
