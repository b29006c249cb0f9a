// kv_topk.cu -- top-K page selection, the per-group union of selected pages,
// and the split-K combine of partial attention results.
//
// KVDrive: A Holistic Multi-Tier KV Cache Management System for Long-Context
// LLM Inference, section 2.2: for each query only the Top-K most important
// blocks are retrieved.  Ties go to the lower page index; pages come out
// ascending.
#include "kv_internal.cuh"
#include "kv_launch.h"
#include "kv_union.cuh"

namespace kvs {
namespace {


__device__ __forceinline__ uint32_t score_key(float s) {
  // +0.0f folds -0.0 into +0.0 so that equal scores compare equal
  return key32(__float_as_uint(s + 0.0f));
}

// Key of a forced page: above every score's key (+inf maps to 0xFF800000;
// 0xFFFFFFFF is a NaN's key, and scores are never NaN).
constexpr uint32_t kForcedKey = 0xFFFFFFFFu;

// One CTA per (b, h) row.  Radix select of the K-th largest key, 8 bits per
// pass from the highest bit where the row's keys differ (the bits above it
// are common to every key, so a pass spent on them would select nothing):
// a shared-memory histogram, double-buffered so that a pass needs two block
// barriers, whose threshold digit one warp finds with a shuffle scan;
// stopping early once every key of the threshold bin is taken.  The output
// pass gives each thread a run of consecutive pages, counts its keys above
// and at the threshold, and after one block scan of those counts places the
// selected pages in page order.  Equal keys at the threshold go to the lower
// page index.  (kv_select.cuh holds a generic select for other kernels.)
// Forced pages (the pages holding the first sink_tokens tokens and the last
// local_tokens tokens of the row) take a key above every score's, so they are
// selected first, lower index first among themselves.
template <int kTopkThreads>
__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float *scores, const int32_t *ctx, int Hq, int ps,
                int maxP, int K, int keys_in_smem, int sink_tokens, int local_tokens,
                int32_t *out, int *status) {
  pdl_wait();
  constexpr int kTopkWarps = kTopkThreads / 32;
  extern __shared__ uint32_t skeys[];
  __shared__ uint32_t hist[2][256];
  __shared__ uint32_t wmin[kTopkWarps], wmax[kTopkWarps];
  __shared__ uint32_t s_digit;
  __shared__ int s_krem, s_all;
  __shared__ unsigned long long wsum[kTopkWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long row = blockIdx.x;
  const int b = (int)(row / Hq);
  int32_t *orow = out + row * K;
  const float *srow = scores + row * maxP;
  // the row's first scores load together with the context length (every
  // one of the row's maxP entries is allocated); entries past the row's
  // pages are masked once the length is known
  constexpr int kSpec = 4;
  float spec[kSpec];
#pragma unroll
  for (int u = 0; u < kSpec; ++u) {
    const int p = tid + u * kTopkThreads;
    spec[u] = p < maxP ? srow[p] : 0.f;
  }
  const int len = ctx[b];
  if (len < 1 || len > maxP * ps) {
    if (tid == 0) flag_error(status, KV_ERR_BOUNDS);
    for (int i = tid; i < K; i += kTopkThreads) orow[i] = -1;
    return;
  }
  const int P = (len + ps - 1) / ps;
  const int keff = min(K, P);
  if (keff == P) {
    for (int i = tid; i < K; i += kTopkThreads) orow[i] = i < P ? i : -1;
    return;
  }
  const int f_sink = sink_tokens > 0 ? min(P, (sink_tokens + ps - 1) / ps) : 0;
  const int f_local = local_tokens > 0 ? max(0, len - local_tokens) / ps : P;
  auto raw_key = [&](int p) -> uint32_t {
    return (p < f_sink || p >= f_local) ? kForcedKey : score_key(srow[p]);
  };
  auto key_at = [&](int p) -> uint32_t { return keys_in_smem ? skeys[p] : raw_key(p); };

  // keys (into shared memory when they fit), their minimum and maximum
  if (tid < 256) hist[0][tid] = 0;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
  for (int u = 0; u < kSpec; ++u) {
    const int p = tid + u * kTopkThreads;
    if (p < P) {
      const uint32_t k = (p < f_sink || p >= f_local) ? kForcedKey : score_key(spec[u]);
      if (keys_in_smem) skeys[p] = k;
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
  }
  for (int p = tid + kSpec * kTopkThreads; p < P; p += kTopkThreads) {
    const uint32_t k = raw_key(p);
    if (keys_in_smem) skeys[p] = k;
    kmin = min(kmin, k);
    kmax = max(kmax, k);
  }
  kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  if (lane == 0) { wmin[warp] = kmin; wmax[warp] = kmax; }
  __syncthreads();
  kmin = __reduce_min_sync(0xFFFFFFFFu, lane < kTopkWarps ? wmin[lane] : 0xFFFFFFFFu);
  kmax = __reduce_max_sync(0xFFFFFFFFu, lane < kTopkWarps ? wmax[lane] : 0u);

  // radix select from the highest bit where the keys differ (the bits above
  // it are common to every key), 8 bits per pass
  const uint32_t diff = kmin ^ kmax;
  const int top = diff ? 31 - __clz(diff) : -1;
  uint32_t pmask = top >= 31 ? 0u : (0xFFFFFFFFu << (top + 1));
  uint32_t prefix = kmin & pmask;
  int krem = keff;
  int pass = 0;
#pragma unroll 1
  for (int hb = top; hb >= 0; hb -= 8, ++pass) {
    const int lb = max(hb - 7, 0);
    const uint32_t dmask = (1u << (hb - lb + 1)) - 1u;
    uint32_t *h = hist[pass & 1];
    if (tid < 256) hist[(pass + 1) & 1][tid] = 0;  // the next pass's histogram
    for (int p = tid; p < P; p += kTopkThreads) {
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
            s_digit = (uint32_t)(255 - 8 * tid - j);
            s_krem = krem - above;
            s_all = (above + c[j] == krem) ? 1 : 0;
            break;
          }
          above += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << lb;
    pmask |= dmask << lb;
    krem = s_krem;
    if (s_all) break;
  }
  pdl_trigger();
  // selected: keys above the threshold, then the first krem equal to it in
  // page order (all of them when the last pass took its whole bin, where
  // krem is their count).  Each thread owns `per` consecutive pages.
  const int per = ((P + kTopkThreads - 1) / kTopkThreads + 3) & ~3;
  const int lo = min(P, tid * per), hi = min(P, lo + per);
  auto load4 = [&](int p, uint32_t (&kk)[4]) {
    if (keys_in_smem && p + 4 <= hi) {
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
    if (lane >= off) { gi += tg; ei += te; }
  }
  if (lane == 31) wsum[warp] = ((unsigned long long)ei << 32) | gi;
  __syncthreads();
  const unsigned long long t = lane < kTopkWarps ? wsum[lane] : 0ull;
  const bool before = lane < warp;
  int gt_b = (int)(__reduce_add_sync(0xFFFFFFFFu, before ? (uint32_t)t : 0u) + gi - gt_n);
  int eq_b = (int)(__reduce_add_sync(0xFFFFFFFFu, before ? (uint32_t)(t >> 32) : 0u) + ei - eq_n);
  for (int p = lo; p < hi; p += 4) {
    uint32_t kk[4];
    load4(p, kk);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t k = kk[e] & pmask;
      const bool in = p + e < hi;
      const bool is_gt = in && k > prefix, is_eq = in && k == prefix;
      if (is_gt || (is_eq && eq_b < krem)) {
        const int pos = gt_b + min(eq_b, krem);
        if (pos < K) orow[pos] = p + e;
      }
      gt_b += is_gt;
      eq_b += is_eq;
    }
  }
  for (int i = keff + tid; i < K; i += kTopkThreads) orow[i] = -1;
}

// ---------------------------------------------------------------------------
// union of the selected pages of the gc heads of one (b, kv head, head chunk)
// ---------------------------------------------------------------------------
// One CTA per group runs union_group (kv_union.cuh).  512 threads (1024
// measured the same, 256 slower on 8192-page rows).
constexpr int kUnionThreads = 512;

__global__ void __launch_bounds__(kUnionThreads)
    union_kernel(const int32_t *idx, const int32_t *ctx, int Hq, int G,
                 int gc, int ps, int maxP, int K, int umax, int32_t *upages,
                 uint32_t *umasks, int32_t *ucount, int *status) {
  pdl_wait();
  extern __shared__ uint32_t words[];  // one byte of head bits per page, 4 pages a word
  __shared__ uint32_t wsum[kUnionThreads / 32];
  union_group<kUnionThreads>(idx, ctx, Hq, G, gc, ps, maxP, K, umax, upages, umasks, ucount,
                             status, blockIdx.x, blockIdx.y, gridDim.x, words, wsum);
}

// ---------------------------------------------------------------------------
// split-K combine: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s
// ---------------------------------------------------------------------------
// One CTA per (b, q head), one thread per output channel.  Every warp finds M
// and the weight sum itself, lane s holding split s, 32 splits a round, so
// the split maxima and weights load together, once, and no block barrier
// waits on them; the first kPre partial outputs of the channel load before
// that, all in flight at once (16 up to 16 splits, else 64: the 57 splits of
// the 128k-token rows), the rest with independent loads after it.

template <int kPre>
__global__ void __launch_bounds__(kHeadDim)
    combine_kernel(const float *part_o, const float *part_ml, float *out, int S, long long rows) {
  pdl_wait();
  constexpr int R = (kPre + 31) / 32;  // rounds of 32 splits whose values stay in registers
  const long long r = blockIdx.x;
  const int c = threadIdx.x, lane = c & 31;
  const float *po = part_o + r * kHeadDim + c;
  const long long stride = rows * kHeadDim;
  // all the first 32 R splits need, loaded at once: this channel's first kPre
  // partial outputs, and split 32 q + lane's maximum and weight per round q
  float pre[kPre], mr[R], lr[R];
#pragma unroll
  for (int s = 0; s < kPre; ++s) pre[s] = s < S ? po[s * stride] : 0.f;
#pragma unroll
  for (int q = 0; q < R; ++q) {
    const int s = 32 * q + lane;
    mr[q] = s < S ? part_ml[(s * rows + r) * 2] : -INFINITY;
    lr[q] = s < S ? part_ml[(s * rows + r) * 2 + 1] : 0.f;
  }
  float M = -INFINITY;
#pragma unroll
  for (int q = 0; q < R; ++q) M = fmaxf(M, mr[q]);
  for (int s = 32 * R + lane; s < S; s += 32) M = fmaxf(M, part_ml[(s * rows + r) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
  auto weight = [M](float m) { return (M == -INFINITY || m == -INFINITY) ? 0.f : ex2(m - M); };
  float l = 0.f, o = 0.f, fr[R];
#pragma unroll
  for (int q = 0; q < R; ++q) {
    fr[q] = weight(mr[q]);
    l = fmaf(fr[q], lr[q], l);
  }
#pragma unroll
  for (int s = 0; s < kPre; ++s) {
    const float ft = __shfl_sync(0xFFFFFFFFu, fr[s / 32], s % 32);
    if (s < S) o = fmaf(ft, pre[s], o);
  }
  // splits kPre .. 32 R - 1 (only when kPre = 16): weights in round R - 1
  for (int s = kPre; s < min(S, 32 * R); ++s)
    o = fmaf(__shfl_sync(0xFFFFFFFFu, fr[R - 1], s & 31), po[s * stride], o);
  for (int s0 = 32 * R; s0 < S; s0 += 32) {
    const int s = s0 + lane;
    float f = 0.f;
    if (s < S) {
      f = weight(part_ml[(s * rows + r) * 2]);
      l = fmaf(f, part_ml[(s * rows + r) * 2 + 1], l);
    }
    const int n = min(32, S - s0);
    for (int t = 0; t < n; ++t) o = fmaf(__shfl_sync(0xFFFFFFFFu, f, t), po[(s0 + t) * stride], o);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, off);
  pdl_trigger();
  out[r * kHeadDim + c] = l > 0.f ? o / l : 0.f;
}

}  // namespace

cudaError_t launch_topk(const float *scores, const int32_t *ctx, int B, int Hq, int ps, int maxP,
                        int k, int sink_tokens, int local_tokens, int32_t *indices, int *status,
                        cudaStream_t st) {
  // keys cached in shared memory, within the default 48 KB per block
  constexpr size_t kMaxSmemKeys = 11264;
  const int in_smem = (size_t)maxP <= kMaxSmemKeys ? 1 : 0;
  const size_t smem = in_smem ? (size_t)maxP * 4 : 0;
  // long rows with few of them get wider CTAs: the histogram and output
  // passes are latency-bound loops over the row
  // (1024 threads on 2048-page rows measured slower: 6.68 against 6.48 us)
  constexpr long long kSms = 152;  // GB300
  const long long rows = (long long)B * Hq;
  const int threads = (maxP >= 4096 && rows < 2 * kSms) ? 1024 : 256;
  auto kern = threads == 1024 ? topk_kernel<1024> : topk_kernel<256>;
  return launch_pdl(kern, dim3((unsigned)rows), dim3(threads), smem, st,
                    scores, ctx, Hq, ps, maxP, k, in_smem, sink_tokens, local_tokens, indices,
                    status);
}

cudaError_t launch_union(const int32_t *indices, const int32_t *ctx, int B, int Hq, int Hkv,
                         int gc, int ps, int maxP, int k, int umax, int32_t *upages,
                         uint32_t *umasks, int32_t *ucount, int *status, cudaStream_t st) {
  const int G = Hq / Hkv;
  const size_t smem = (size_t)((maxP + 3) / 4) * 4;
  static int attr_done[64] = {0};  // raise the dynamic shared memory cap once per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && (dev < 0 || dev >= 64 || !attr_done[dev])) {
    cudaError_t e =
        cudaFuncSetAttribute(union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  dim3 grid(Hkv * (G / gc), B);
  return launch_pdl(union_kernel, grid, dim3(kUnionThreads), smem, st, indices, ctx, Hq, G, gc, ps,
                    maxP, k, umax, upages, umasks, ucount, status);
}

cudaError_t launch_combine(const float *part_o, const float *part_ml, float *out, int S, int B,
                           int Hq, cudaStream_t st) {
  const long long rows = (long long)B * Hq;
  auto kern = S <= 16 ? combine_kernel<16> : combine_kernel<64>;
  return launch_pdl(kern, dim3((unsigned)rows), dim3(kHeadDim), 0, st, part_o, part_ml, out, S,
                    rows);
}

}  // namespace kvs
