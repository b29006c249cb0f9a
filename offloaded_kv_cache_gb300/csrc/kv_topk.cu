// kv_topk.cu -- top-K page selection, the per-group union of selected pages,
// and the split-K combine of partial attention results.
//
// KVDrive: A Holistic Multi-Tier KV Cache Management System for Long-Context
// LLM Inference, section 2.2: for each query only the Top-K most important
// blocks are retrieved.  Ties go to the lower page index; pages come out
// ascending.
#include "kv_internal.cuh"
#include "kv_launch.h"
#include "kv_radix.cuh"
#include "kv_union.cuh"

namespace kvs {
namespace {


// One CTA per (b, h) row: the radix select of kv_radix.cuh over the row's
// keys (in shared memory when they fit), then its selected pages in page
// order.  (kv_select.cuh holds a generic select for other kernels.)  Forced
// pages (the pages holding the first sink_tokens tokens and the last
// local_tokens tokens of the row) take a key above every score's, so they are
// selected first, lower index first among themselves.
template <int kTopkThreads>
__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float *scores, const int32_t *ctx, int Hq, int ps,
                int maxP, int K, int keys_in_smem, int sink_tokens, int local_tokens,
                int32_t *out, int *status) {
  pdl_wait();
  extern __shared__ uint32_t skeys[];
  __shared__ RadixSmem<kTopkThreads> rs;
  const int tid = threadIdx.x;
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
  if (tid < 256) rs.hist[0][tid] = 0;
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
  block_minmax<kTopkThreads>(rs, kmin, kmax);
  uint32_t prefix, pmask;
  int krem;
  radix_threshold<kTopkThreads>(rs, key_at, P, keff, kmin, kmax, prefix, pmask, krem);
  pdl_trigger();
  radix_emit<kTopkThreads>(rs, key_at, keys_in_smem ? skeys : nullptr, P, prefix, pmask, krem,
                           [&](int pos, int p) {
                             if (pos < K) orow[pos] = p;
                           });
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

// ---------------------------------------------------------------------------
// split combine of the attention over kv_select_pages' lists
// ---------------------------------------------------------------------------
// The attention kernel records per group g (gmeta[g]) whether its partials
// are the S splits of g (kSplitPerGroup: partial s of row r at s * rows + r)
// or come from the equal chunks of all groups' lists (kSplitSpread): the
// merged partials of CTAs first..last (CTA i's at i * G + head), where with
// tail = 1 the last CTA's share of g is instead nw warp partials in spa_*.
// One CTA per (b, q head), one thread per output channel; the merge is the
// one of combine_kernel over that list of partials.
template <int kPre>
__global__ void __launch_bounds__(kHeadDim)
    combine_lists_kernel(const float *part_o, const float *part_ml, const float *spa_o,
                         const float *spa_ml, const int32_t *gmeta, float *out, int S, int Hq,
                         int Hkv, int nw, int *status) {
  pdl_wait();
  constexpr int R = (kPre + 31) / 32;  // rounds of 32 partials whose values stay in registers
  const int r = blockIdx.x, c = threadIdx.x, lane = c & 31;
  const int G = Hq / Hkv, b = r / Hq, h = r % Hq;
  const int NG = (int)(gridDim.x / Hq) * Hkv;
  const int g = b * Hkv + h / G, hl = h % G;
  const long long ncta = (long long)S * NG;
  // partial k: merged partial k (k < nm) at base + k * stride, else warp
  // partial k - nm of the group's tail in spa_*
  int nm = S, na = 0;
  const long long rows = (long long)NG * G;
  const float *ob = part_o + ((long long)g * G + hl) * kHeadDim + c;  // per group: split k
  const float *mb = part_ml + ((long long)g * G + hl) * 2;
  long long os = rows * kHeadDim, ms = rows * 2;
  const float *tob = spa_o + ((long long)g * nw * G + hl) * kHeadDim + c;
  const float *tmb = spa_ml + ((long long)g * nw * G + hl) * 2;
  auto po = [&](int k) -> const float * {
    return k < nm ? ob + k * os : tob + (long long)(k - nm) * G * kHeadDim;
  };
  auto pml = [&](int k) -> const float * {
    return k < nm ? mb + k * ms : tmb + (long long)(k - nm) * G * 2;
  };
  // the per-group split's first partials load with the record, as in
  // combine_kernel (so that split costs no extra round trip); equal chunks
  // load theirs once the record is read
  const int4 m = ld_issue(reinterpret_cast<const int4 *>(gmeta) + g);
  float pre[kPre], mr[R], lr[R];
  auto load_first = [&](int n) {
#pragma unroll
    for (int s = 0; s < kPre; ++s) pre[s] = s < n ? ld_issue(po(s)) : 0.f;
#pragma unroll
    for (int q = 0; q < R; ++q) {
      const int k = 32 * q + lane;
      mr[q] = k < n ? ld_issue(pml(k)) : -INFINITY;
      lr[q] = k < n ? ld_issue(pml(k) + 1) : 0.f;
    }
  };
  load_first(S);
  if (m.x == kSplitSpread && m.y >= 0 && m.y <= m.z && m.z < ncta && (m.w == 0 || m.w == 1)) {
    // merged partials of CTAs m.y .. (row CTA * G + head)
    ob = part_o + ((long long)m.y * G + hl) * kHeadDim + c;
    mb = part_ml + ((long long)m.y * G + hl) * 2;
    os = (long long)G * kHeadDim;
    ms = (long long)G * 2;
    nm = m.z - m.y + (m.w ? 0 : 1);
    na = m.w ? nw : 0;
    load_first(nm + na);
  } else if (m.x != kSplitPerGroup) {
    if (c == 0) flag_error(status, KV_ERR_BOUNDS);
    out[(long long)r * kHeadDim + c] = 0.f;
    return;
  }
  // from here the merge of combine_kernel, over partials 0 .. n - 1
  const int n = nm + na;
  float M = -INFINITY;
#pragma unroll
  for (int q = 0; q < R; ++q) M = fmaxf(M, mr[q]);
  for (int k = 32 * R + lane; k < n; k += 32) M = fmaxf(M, pml(k)[0]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
  auto weight = [M](float x) { return (M == -INFINITY || x == -INFINITY) ? 0.f : ex2(x - M); };
  float l = 0.f, o = 0.f, fr[R];
#pragma unroll
  for (int q = 0; q < R; ++q) {
    fr[q] = weight(mr[q]);
    l = fmaf(fr[q], lr[q], l);
  }
#pragma unroll
  for (int s = 0; s < kPre; ++s) {
    const float ft = __shfl_sync(0xFFFFFFFFu, fr[s / 32], s % 32);
    if (s < n) o = fmaf(ft, pre[s], o);
  }
  for (int s = kPre; s < min(n, 32 * R); ++s)
    o = fmaf(__shfl_sync(0xFFFFFFFFu, fr[R - 1], s & 31), *po(s), o);
  for (int s0 = 32 * R; s0 < n; s0 += 32) {
    const int k = s0 + lane;
    float f = 0.f;
    if (k < n) {
      f = weight(pml(k)[0]);
      l = fmaf(f, pml(k)[1], l);
    }
    const int cnt = min(32, n - s0);
    for (int t = 0; t < cnt; ++t) o = fmaf(__shfl_sync(0xFFFFFFFFu, f, t), *po(s0 + t), o);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, off);
  pdl_trigger();
  out[(long long)r * kHeadDim + c] = l > 0.f ? o / l : 0.f;
}

cudaError_t launch_combine_lists(const float *part_o, const float *part_ml, const float *spa_o,
                                 const float *spa_ml, const int32_t *gmeta, float *out, int S,
                                 int B, int Hq, int Hkv, int nw, int *status, cudaStream_t st) {
  const long long rows = (long long)B * Hq;
  auto kern = S <= 16 ? combine_lists_kernel<16> : combine_lists_kernel<64>;
  return launch_pdl(kern, dim3((unsigned)rows), dim3(kHeadDim), 0, st, part_o, part_ml, spa_o,
                    spa_ml, gmeta, out, S, Hq, Hkv, nw, status);
}

cudaError_t launch_combine(const float *part_o, const float *part_ml, float *out, int S, int B,
                           int Hq, cudaStream_t st) {
  const long long rows = (long long)B * Hq;
  auto kern = S <= 16 ? combine_kernel<16> : combine_kernel<64>;
  return launch_pdl(kern, dim3((unsigned)rows), dim3(kHeadDim), 0, st, part_o, part_ml, out, S,
                    rows);
}

}  // namespace kvs
