// kv_index.cu -- the Quest index: per-page channel-wise key min/max, and the
// page score q . (min, max) that bounds q . k from above.
//
// KVDrive: A Holistic Multi-Tier KV Cache Management System for Long-Context
// LLM Inference, section 2.2 "Sparse attention": keys are split into blocks
// and a block's importance is estimated by multiplying the query with the
// channel-wise minimum and maximum of its keys.
//
// Both kernels stream their input once with coalesced 16-byte loads; they are
// HBM-bound (or host-link bound for a host-resident K cache in the build).
#include <type_traits>

#include "kv_internal.cuh"
#include "kv_launch.h"

namespace kvs {
namespace {

// ---------------------------------------------------------------------------
// minmax build: one warp per (sequence, logical page, kv head)
// ---------------------------------------------------------------------------
// A page of one kv head is ps rows of d = 128 elements (256 or 512 bytes).
// Lane = (16-byte column chunk, row group); rows are strided by the number of
// row groups.  Values become IEEE totalOrder keys, so an unsigned min/max is
// exact and does not depend on the order of the reduction (-0.0 < +0.0).
template <class T>
__global__ void __launch_bounds__(256)
    minmax_build_kernel(const T *k, const int32_t *bt,
                        const int32_t *ctx, T *mm, int B, int Hkv,
                        int ps, int maxP, long long nphys, int *status) {
  pdl_wait();
  constexpr int C = kHeadDim * (int)sizeof(T) / 16;  // 16-byte chunks per row
  constexpr int RG = 32 / C;                          // row groups per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * 8 + warp;
  if (item >= (long long)B * maxP * Hkv) return;
  const int kvh = (int)(item % Hkv);
  const long long bp = item / Hkv;
  const int p = (int)(bp % maxP);
  const int b = (int)(bp / maxP);
  const int len = ctx[b];
  if (len < 1 || len > maxP * ps) {
    if (p == 0 && kvh == 0 && lane == 0) flag_error(status, KV_ERR_BOUNDS);
    return;
  }
  if (p * ps >= len) return;
  const int n = min(ps, len - p * ps);
  const long long phys = bt[(long long)b * maxP + p];
  if (phys < 0 || phys >= nphys) {
    if (lane == 0) flag_error(status, KV_ERR_BOUNDS);
    return;
  }
  const int chunk = lane % C, rg = lane / C;
  const uint4 *src = reinterpret_cast<const uint4 *>(k) + ((phys * Hkv + kvh) * ps) * C + chunk;
  uint4 lo = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
  uint4 hi = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 8
  for (int r = rg; r < n; r += RG) {
    uint4 x = src[(long long)r * C];
    if constexpr (sizeof(T) == 2) {
      x.x = key16x2(x.x); x.y = key16x2(x.y); x.z = key16x2(x.z); x.w = key16x2(x.w);
      lo.x = __vminu2(lo.x, x.x); lo.y = __vminu2(lo.y, x.y);
      lo.z = __vminu2(lo.z, x.z); lo.w = __vminu2(lo.w, x.w);
      hi.x = __vmaxu2(hi.x, x.x); hi.y = __vmaxu2(hi.y, x.y);
      hi.z = __vmaxu2(hi.z, x.z); hi.w = __vmaxu2(hi.w, x.w);
    } else {
      x.x = key32(x.x); x.y = key32(x.y); x.z = key32(x.z); x.w = key32(x.w);
      lo.x = min(lo.x, x.x); lo.y = min(lo.y, x.y); lo.z = min(lo.z, x.z); lo.w = min(lo.w, x.w);
      hi.x = max(hi.x, x.x); hi.y = max(hi.y, x.y); hi.z = max(hi.z, x.z); hi.w = max(hi.w, x.w);
    }
  }
  pdl_trigger();
  if constexpr (RG == 2) {
    // merge the two row groups (lanes l and l ^ 16 hold the same chunk)
    uint4 lo2, hi2;
    lo2.x = __shfl_xor_sync(0xFFFFFFFFu, lo.x, 16); lo2.y = __shfl_xor_sync(0xFFFFFFFFu, lo.y, 16);
    lo2.z = __shfl_xor_sync(0xFFFFFFFFu, lo.z, 16); lo2.w = __shfl_xor_sync(0xFFFFFFFFu, lo.w, 16);
    hi2.x = __shfl_xor_sync(0xFFFFFFFFu, hi.x, 16); hi2.y = __shfl_xor_sync(0xFFFFFFFFu, hi.y, 16);
    hi2.z = __shfl_xor_sync(0xFFFFFFFFu, hi.z, 16); hi2.w = __shfl_xor_sync(0xFFFFFFFFu, hi.w, 16);
    lo.x = __vminu2(lo.x, lo2.x); lo.y = __vminu2(lo.y, lo2.y);
    lo.z = __vminu2(lo.z, lo2.z); lo.w = __vminu2(lo.w, lo2.w);
    hi.x = __vmaxu2(hi.x, hi2.x); hi.y = __vmaxu2(hi.y, hi2.y);
    hi.z = __vmaxu2(hi.z, hi2.z); hi.w = __vmaxu2(hi.w, hi2.w);
  }
  uint4 *dst = reinterpret_cast<uint4 *>(mm) + ((phys * Hkv + kvh) * 2) * C + chunk;
  if constexpr (sizeof(T) == 2) {
    // row group 0 writes the minimum, row group 1 the maximum
    uint4 kk = rg == 0 ? lo : hi;
    kk.x = unkey16x2(kk.x); kk.y = unkey16x2(kk.y); kk.z = unkey16x2(kk.z); kk.w = unkey16x2(kk.w);
    dst[rg * C] = kk;
  } else {
    lo.x = unkey32(lo.x); lo.y = unkey32(lo.y); lo.z = unkey32(lo.z); lo.w = unkey32(lo.w);
    hi.x = unkey32(hi.x); hi.y = unkey32(hi.y); hi.z = unkey32(hi.z); hi.w = unkey32(hi.w);
    dst[0] = lo;
    dst[C] = hi;
  }
}

// ---------------------------------------------------------------------------
// page score: one warp per page, lane = 4 channels, GS query heads at once
// ---------------------------------------------------------------------------
// Sum over G per-lane partials across the warp with halving exchanges: after
// the call lane l holds the full sum of head l / (32 / G).
template <int G>
__device__ __forceinline__ float reduce_heads(float (&v)[G], int lane) {
  int bit = 16;
#pragma unroll
  for (int n = G; n > 1; n >>= 1, bit >>= 1) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? v[i] : v[i + n / 2];
      const float keep = up ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, bit);
    }
  }
#pragma unroll
  for (; bit >= 1; bit >>= 1) v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], bit);
  return v[0];
}

template <class T>
__device__ __forceinline__ void load4(const T *p, float (&x)[4]) {
  if constexpr (sizeof(T) == 4) {
    const float4 f = *reinterpret_cast<const float4 *>(p);
    x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
  } else {
    const uint2 w = *reinterpret_cast<const uint2 *>(p);
    const float2 a = unpack2(w.x, T()), c = unpack2(w.y, T());
    x[0] = a.x; x[1] = a.y; x[2] = c.x; x[3] = c.y;
  }
}

constexpr int kScoreWarps = 8;
constexpr int kScorePagesPerWarp = 8;

// One warp scores kScorePagesPerWarp pages of one (b, kv head, head chunk):
// the pages' block-table entries arrive in one load, every table load is
// issued before any arithmetic, then each page's GS head sums are reduced.
// MEAN: the table row is the page's mean key and the score is q . mean.
template <class T, int GS, bool MEAN>
__global__ void __launch_bounds__(32 * kScoreWarps)
    page_score_kernel(const T *q, const T *mm,
                      const int32_t *bt, const int32_t *ctx,
                      float *scores, int Hq, int Hkv, int ps, int maxP,
                      long long nphys, int nchunk, int *status) {
  pdl_wait();
  constexpr int PPW = kScorePagesPerWarp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int kvh = blockIdx.y / nchunk, chunk = blockIdx.y % nchunk;
  const int G = Hq / Hkv;
  const int head0 = kvh * G + chunk * GS;
  const int len = ctx[b];
  if (len < 1 || len > maxP * ps) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) flag_error(status, KV_ERR_BOUNDS);
    return;
  }
  const int P = (len + ps - 1) / ps;
  const int p0 = (blockIdx.x * kScoreWarps + warp) * PPW;  // this warp's first page
  if (p0 >= maxP) return;

  constexpr int kSpan = 32 / GS;     // lanes per head after the reduction
  const int my_head = lane / kSpan;  // the head whose total this lane ends with
  const bool writer = (lane % kSpan) == 0;
  float *srow = scores + ((long long)b * Hq + head0 + my_head) * maxP;

  // block-table entries of the warp's pages (lane i < PPW holds page p0 + i)
  long long my_phys = -1;
  if (lane < PPW && p0 + lane < P) {
    const long long ph = bt[(long long)b * maxP + p0 + lane];
    if (ph >= 0 && ph < nphys) my_phys = ph;
    else flag_error(status, KV_ERR_BOUNDS);
  }
  constexpr int kRows = MEAN ? 1 : 2;  // table rows per (page, kv head)
  float mn[PPW][4], mx[PPW][MEAN ? 1 : 4];
#pragma unroll
  for (int i = 0; i < PPW; ++i) {
    const long long phys = __shfl_sync(0xFFFFFFFFu, my_phys, i);
    if (phys >= 0) {
      const T *row = mm + ((phys * Hkv + kvh) * kRows) * kHeadDim + 4 * lane;
      load4(row, mn[i]);
      if constexpr (!MEAN) load4(row + kHeadDim, mx[i]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) mn[i][e] = 0.f;
      if constexpr (!MEAN) {
#pragma unroll
        for (int e = 0; e < 4; ++e) mx[i][e] = 0.f;
      }
    }
  }
  float qf[GS][4];
#pragma unroll
  for (int g = 0; g < GS; ++g) load4(q + ((long long)b * Hq + head0 + g) * kHeadDim + 4 * lane, qf[g]);

#pragma unroll
  for (int i = 0; i < PPW; ++i) {
    const int p = p0 + i;
    if (p >= maxP) break;
    const long long phys = __shfl_sync(0xFFFFFFFFu, my_phys, i);
    if (phys < 0) {  // past the row's last page, or a bad entry
      if (writer) srow[p] = -INFINITY;
      continue;
    }
    float part[GS];
#pragma unroll
    for (int g = 0; g < GS; ++g) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // max(q*mn, q*mx) == q * (q >= 0 ? mx : mn) because mx >= mn
        float bound;
        if constexpr (MEAN) bound = mn[i][e];
        else bound = qf[g][e] >= 0.f ? mx[i][e] : mn[i][e];
        s = fmaf(qf[g][e], bound, s);
      }
      part[g] = s;
    }
    const float tot = reduce_heads<GS>(part, lane);
    if (writer) srow[p] = tot;
  }
}

// ---------------------------------------------------------------------------
// page score as a tensor-core contraction (16-bit data, 4 or 8 heads)
// ---------------------------------------------------------------------------
// max(q*mn, q*mx) == min(q, 0)*mn + max(q, 0)*mx, so over a group's GS heads
// the scores of 16 pages are S[page][head] = T[page][0..256) . C[0..256)[head]
// with T a page's [min | max] row (the table's own layout) and C the
// [q- | q+] coefficients -- a 16 x 8 x 256 mma.sync contraction.  Products of
// two 16-bit values are exact in fp32; sums accumulate in fp32.
//
// k order: lane (gid, tig) loads 16-byte chunks ch = tig + 4 i (i = 0..7) of
// rows gid and gid + 8; chunk i supplies k-steps 2i and 2i + 1, whose slots
// (2tig, 2tig+1, 2tig+8, 2tig+9) take the chunk's elements 0..3 and 4..7.
// The q coefficients follow the same permutation, so every global load is a
// coalesced 16-byte load straight into an A fragment.
__device__ __forceinline__ void mma_score(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, __nv_bfloat16) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_score(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, __half) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// keep the halves of a packed 16-bit pair whose sign is set (neg) or clear
__device__ __forceinline__ uint32_t sign_part(uint32_t w, bool neg) {
  const uint32_t s = (w >> 15) & 0x00010001u;  // 1 per negative half
  const uint32_t m = (neg ? s : (s ^ 0x00010001u)) * 0xFFFFu;
  return w & m;
}

constexpr int kScoreMmaWarps = 8;

// MEAN: the contraction runs over the 128-long mean row with q itself as the
// coefficients (4 chunks per lane instead of 8).
template <class T, int GS, bool MEAN>
__global__ void __launch_bounds__(32 * kScoreMmaWarps)
    page_score_mma_kernel(const T *q, const T *mm,
                          const int32_t *bt, const int32_t *ctx,
                          float *scores, int Hq, int Hkv, int ps, int maxP,
                          long long nphys, int nchunk, int early_inputs, int *status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int b = blockIdx.z;
  const int kvh = blockIdx.y / nchunk, chunk = blockIdx.y % nchunk;
  const int G = Hq / Hkv;
  const int head0 = kvh * G + chunk * GS;
  // q's coefficients first.  When the previous kernel in the stream is one
  // of the library's (early_inputs), which write neither q nor the block
  // table, they load before the wait for it, overlapping its tail; as the
  // first kernel of a call, after the wait.
  if (!early_inputs) pdl_wait();
  // coefficients of head gid in the same k order: [q- | q+] (min/max) or q (mean)
  constexpr int NCH = MEAN ? 4 : 8;       // 16-byte chunks per lane per row
  uint4 cf[NCH];
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    cf[i] = make_uint4(0u, 0u, 0u, 0u);
    if (gid < GS) {
      const int ch = tig + 4 * i;  // chunk of the coefficient row
      const uint4 w = reinterpret_cast<const uint4 *>(
          q + ((long long)b * Hq + head0 + gid) * kHeadDim)[ch & 15];
      if constexpr (MEAN) {
        cf[i] = w;
      } else {
        const bool neg = ch < 16;
        cf[i] = make_uint4(sign_part(w.x, neg), sign_part(w.y, neg), sign_part(w.z, neg),
                           sign_part(w.w, neg));
      }
    }
  }
  const int p0 = (blockIdx.x * kScoreMmaWarps + warp) * 16;  // this warp's 16 pages
  // the block-table entries too
  long long bt_lane = -1;
  if (lane < 16 && p0 + lane < maxP) bt_lane = bt[(long long)b * maxP + p0 + lane];
  if (early_inputs) pdl_wait();
  // Index rows of the warp's in-range physical pages load together with the
  // context length (their addresses need only the block table); pages past
  // the context are masked once the length is known.  Lanes 0..15 hold the
  // 16 entries; rows gid and gid + 8 are this lane's.
  const long long cand = (lane < 16 && bt_lane >= 0 && bt_lane < nphys) ? bt_lane : -1;
  const long long ph_a = __shfl_sync(0xFFFFFFFFu, cand, gid);
  const long long ph_b = __shfl_sync(0xFFFFFFFFu, cand, gid + 8);
  constexpr int kRowElems = MEAN ? kHeadDim : 2 * kHeadDim;
  uint4 ra[NCH], rb[NCH];
  const uint4 *rowa = reinterpret_cast<const uint4 *>(mm + ((ph_a < 0 ? 0 : ph_a) * Hkv + kvh) * kRowElems);
  const uint4 *rowb = reinterpret_cast<const uint4 *>(mm + ((ph_b < 0 ? 0 : ph_b) * Hkv + kvh) * kRowElems);
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    ra[i] = ph_a >= 0 ? rowa[tig + 4 * i] : make_uint4(0u, 0u, 0u, 0u);
    rb[i] = ph_b >= 0 ? rowb[tig + 4 * i] : make_uint4(0u, 0u, 0u, 0u);
  }
  const int len = ctx[b];
  if (len < 1 || len > maxP * ps) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) flag_error(status, KV_ERR_BOUNDS);
    return;
  }
  const int P = (len + ps - 1) / ps;
  if (p0 >= maxP) return;
  // a page of the context whose block-table entry is out of range
  if (lane < 16 && p0 + lane < P && cand < 0) flag_error(status, KV_ERR_BOUNDS);
  pdl_trigger();
  float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const uint32_t a0[4] = {ra[i].x, rb[i].x, ra[i].y, rb[i].y};
    mma_score(c, a0, cf[i].x, cf[i].y, T());
    const uint32_t a1[4] = {ra[i].z, rb[i].z, ra[i].w, rb[i].w};
    mma_score(c, a1, cf[i].z, cf[i].w, T());
  }
  // c0/c1: page gid, heads 2tig / 2tig+1; c2/c3: page gid + 8
  const int pa = p0 + gid, pb = pa + 8;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int h = 2 * tig + (e & 1);
    const int p = (e < 2) ? pa : pb;
    const bool ok = p < P && ((e < 2) ? ph_a >= 0 : ph_b >= 0);
    if (h < GS && p < maxP)
      scores[((long long)b * Hq + head0 + h) * maxP + p] = ok ? c[e] : -INFINITY;
  }
}

template <class T, bool MEAN>
cudaError_t score_dispatch(const void *q, const void *mm, const int32_t *bt, const int32_t *ctx,
                           float *scores, int B, int Hq, int Hkv, int ps, int maxP,
                           long long nphys, int early_inputs, int *status, cudaStream_t st) {
  const int G = Hq / Hkv;
  const int gs = (G % 8 == 0) ? 8 : (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
  const int nchunk = G / gs;
  if constexpr (sizeof(T) == 2) {
    if (gs >= 4) {  // a tokens-free pages x heads x 256 contraction: tensor cores
      dim3 g((maxP + 16 * kScoreMmaWarps - 1) / (16 * kScoreMmaWarps), Hkv * nchunk, B);
      const T *qq = static_cast<const T *>(q);
      const T *m = static_cast<const T *>(mm);
      auto kern = gs == 8 ? page_score_mma_kernel<T, 8, MEAN> : page_score_mma_kernel<T, 4, MEAN>;
      return launch_pdl(kern, g, dim3(32 * kScoreMmaWarps), 0, st, qq, m, bt, ctx, scores, Hq,
                        Hkv, ps, maxP, nphys, nchunk, early_inputs, status);
    }
  }
  dim3 grid((maxP + kScoreWarps * kScorePagesPerWarp - 1) / (kScoreWarps * kScorePagesPerWarp),
            Hkv * nchunk, B);
  const T *qq = static_cast<const T *>(q);
  const T *m = static_cast<const T *>(mm);
  auto kern = gs == 8   ? page_score_kernel<T, 8, MEAN>
              : gs == 4 ? page_score_kernel<T, 4, MEAN>
              : gs == 2 ? page_score_kernel<T, 2, MEAN>
                        : page_score_kernel<T, 1, MEAN>;
  return launch_pdl(kern, grid, dim3(32 * kScoreWarps), 0, st, qq, m, bt, ctx, scores, Hq, Hkv,
                    ps, maxP, nphys, nchunk, status);
}

}  // namespace

cudaError_t launch_minmax_build(int dtype, const void *k, const int32_t *bt, const int32_t *ctx,
                                void *minmax, int B, int Hkv, int ps, int maxP, long long nphys,
                                int *status, cudaStream_t st) {
  const long long items = (long long)B * maxP * Hkv;
  const unsigned blocks = (unsigned)((items + 7) / 8);
  switch (dtype) {
    case KV_F32:
      return launch_pdl(minmax_build_kernel<float>, dim3(blocks), dim3(256), 0, st,
                        static_cast<const float *>(k), bt, ctx, static_cast<float *>(minmax), B,
                        Hkv, ps, maxP, nphys, status);
    case KV_F16:
      return launch_pdl(minmax_build_kernel<__half>, dim3(blocks), dim3(256), 0, st,
                        static_cast<const __half *>(k), bt, ctx, static_cast<__half *>(minmax), B,
                        Hkv, ps, maxP, nphys, status);
    default:
      return launch_pdl(minmax_build_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, st,
                        static_cast<const __nv_bfloat16 *>(k), bt, ctx,
                        static_cast<__nv_bfloat16 *>(minmax), B, Hkv, ps, maxP, nphys, status);
  }
}

cudaError_t launch_page_score(int dtype, bool mean, const void *q, const void *table,
                              const int32_t *bt, const int32_t *ctx, float *scores, int B, int Hq,
                              int Hkv, int ps, int maxP, long long nphys, int early_inputs,
                              int *status, cudaStream_t st) {
#define KVS_SCORE(T, M)                                                                     \
  score_dispatch<T, M>(q, table, bt, ctx, scores, B, Hq, Hkv, ps, maxP, nphys, early_inputs, \
                       status, st)
  switch (dtype) {
    case KV_F32: return mean ? KVS_SCORE(float, true) : KVS_SCORE(float, false);
    case KV_F16: return mean ? KVS_SCORE(__half, true) : KVS_SCORE(__half, false);
    default: return mean ? KVS_SCORE(__nv_bfloat16, true) : KVS_SCORE(__nv_bfloat16, false);
  }
#undef KVS_SCORE
}

// ---------------------------------------------------------------------------
// mean-key index: per (page, kv head), the mean of the valid keys, rounded
// once (to nearest, ties to even) from the exact mean
// ---------------------------------------------------------------------------
// Same lane layout as the min/max build (lane = 16-byte column chunk x row
// group).  Each lane sums its channels in fp32 from -0.0 (so the sum of
// keys that are all -0.0 stays -0.0, as IEEE addition of the keys gives)
// with an error-free transformation per addition (Knuth's TwoSum: the sum s
// and the exact rounding error of each addition, accumulated in c), and sums
// |k| beside it.  The only inexact step is the accumulation of the errors in
// c, within (n + 2)^2 2^-48 sum|k| of its exact value, so s + c is the exact sum
// to that bound; the candidate -- (s + c) / n rounded to the storage type --
// is the correctly rounded mean when that whole interval lies strictly
// inside the candidate's rounding cell (between the midpoints to its
// neighbours).  That holds for all but a vanishing share of channels (a
// plain fp32 sum's bound, n 2^-24 sum|k|, left a few per cent of the
// channels of N(0,1) keys undecided: the 70B-class build went from 0.17 to
// 2.1 ms); the others (a mean on or next to a midpoint, overflow) are
// recomputed exactly: the channel's keys re-read, summed as integers in
// units of 2^-149 (every fp32, f16 and bf16 value is a whole number of
// them), divided by n by long division, rounded once.
// last_only: one item per (b, kv head), the page holding the row's last
// token -- the refresh after an append.
namespace {

// storage format: significand bits (with the implicit one), and the
// exponent of the smallest spacing in units of 2^-149
template <class T> struct Fmt;
template <> struct Fmt<float> { static constexpr int kP = 24, kTmin = 0; };
template <> struct Fmt<__half> { static constexpr int kP = 11, kTmin = 125; };
template <> struct Fmt<__nv_bfloat16> { static constexpr int kP = 8, kTmin = 16; };

// value of a stored key as (sign, integer magnitude, shift): |k| = mag 2^shift
// units of 2^-149
template <class T>
__device__ __forceinline__ void key_parts(uint32_t bits, uint32_t &neg, uint32_t &mag, int &sh) {
  if constexpr (sizeof(T) == 4) {
    const int e = (bits >> 23) & 0xFF;
    neg = bits >> 31;
    mag = (bits & 0x7FFFFFu) | (e ? 0x800000u : 0u);
    sh = max(e, 1) - 1;
  } else if constexpr (std::is_same<T, __half>::value) {
    const int e = (bits >> 10) & 0x1F;
    neg = (bits >> 15) & 1u;
    mag = (bits & 0x3FFu) | (e ? 0x400u : 0u);
    sh = max(e, 1) + 124;
  } else {
    const int e = (bits >> 7) & 0xFF;
    neg = (bits >> 15) & 1u;
    mag = (bits & 0x7Fu) | (e ? 0x80u : 0u);
    sh = max(e, 1) + 15;
  }
}

// exact integer sums: 9 digits of 32 bits (288 bits; n <= 128 keys below
// 2^128 need 284 bits above 2^-149)
constexpr int kMeanDigits = 9;

__device__ __noinline__ void digits_add(uint32_t *acc, uint32_t mag, int sh) {
  const int i = sh >> 5;
  uint64_t v = (uint64_t)mag << (sh & 31);
  uint64_t carry = 0;
  for (int j = i; j < kMeanDigits; ++j) {
    const uint64_t t = (uint64_t)acc[j] + (v & 0xFFFFFFFFull) + carry;
    acc[j] = (uint32_t)t;
    carry = t >> 32;
    v >>= 32;
    if (v == 0 && carry == 0) break;
  }
}

// 16-bit (or 32-bit) pattern of sign * keep * 2^(t - 149), which is a value of
// the storage type
template <class T>
__device__ __forceinline__ uint32_t pack_value(bool neg, uint32_t keep, int t) {
  float v = 0.f;
  if (keep != 0u) {
    const int k = t - 149;
    const float p2 = k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
    v = (float)keep * p2;  // exact: the product is a value of the type
  }
  if (neg) v = -v;
  if constexpr (sizeof(T) == 4) return __float_as_uint(v);
  else if constexpr (std::is_same<T, __half>::value) return __half_as_ushort(__float2half_rn(v));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// The exact mean of channel c of the page's n keys, correctly rounded (the
// rare path: kept out of line).
template <class T>
__device__ __noinline__ uint32_t exact_mean(const T *page, int c, int n) {
  uint32_t pos[kMeanDigits], negd[kMeanDigits];
  for (int j = 0; j < kMeanDigits; ++j) pos[j] = negd[j] = 0u;
  bool any_pos_zero = false;
  for (int r = 0; r < n; ++r) {
    uint32_t bits;
    if constexpr (sizeof(T) == 4) bits = __float_as_uint(page[(long long)r * kHeadDim + c]);
    else bits = reinterpret_cast<const uint16_t *>(page)[(long long)r * kHeadDim + c];
    uint32_t ng, mag;
    int sh;
    key_parts<T>(bits, ng, mag, sh);
    if (mag == 0u) {
      any_pos_zero |= ng == 0u;
      continue;
    }
    digits_add(ng ? negd : pos, mag, sh);
  }
  // |pos - neg| and its sign
  int cmp = 0;
  for (int j = kMeanDigits - 1; j >= 0 && cmp == 0; --j)
    cmp = pos[j] > negd[j] ? 1 : pos[j] < negd[j] ? -1 : 0;
  if (cmp == 0) {  // an exact zero: -0 only if every key was -0 (none positive)
    bool all_neg_zero = !any_pos_zero;
    for (int r = 0; r < n && all_neg_zero; ++r) {
      uint32_t bits;
      if constexpr (sizeof(T) == 4) bits = __float_as_uint(page[(long long)r * kHeadDim + c]);
      else bits = reinterpret_cast<const uint16_t *>(page)[(long long)r * kHeadDim + c];
      uint32_t ng, mag;
      int sh;
      key_parts<T>(bits, ng, mag, sh);
      all_neg_zero = mag == 0u && ng;
    }
    return pack_value<T>(all_neg_zero, 0u, 0);
  }
  const bool neg = cmp < 0;
  uint32_t *a = neg ? negd : pos;
  const uint32_t *b = neg ? pos : negd;
  uint64_t borrow = 0;
  for (int j = 0; j < kMeanDigits; ++j) {
    const uint64_t t = (uint64_t)a[j] - b[j] - borrow;
    a[j] = (uint32_t)t;
    borrow = (t >> 63) & 1u;
  }
  // quotient by n, remainder
  uint64_t rem = 0;
  for (int j = kMeanDigits - 1; j >= 0; --j) {
    const uint64_t cur = (rem << 32) | a[j];
    a[j] = (uint32_t)(cur / (uint64_t)n);
    rem = cur % (uint64_t)n;
  }
  int bitlen = 0;
  for (int j = kMeanDigits - 1; j >= 0; --j)
    if (a[j]) {
      bitlen = 32 * j + 32 - __clz(a[j]);
      break;
    }
  auto qbit = [&](int i) -> uint32_t { return i < 0 ? 0u : (a[i >> 5] >> (i & 31)) & 1u; };
  const int t = max(Fmt<T>::kTmin, bitlen - Fmt<T>::kP);
  uint32_t keep = 0u;
  for (int i = bitlen - 1; i >= t; --i) keep = (keep << 1) | qbit(i);
  bool up;
  if (t == 0) {  // the spacing is the unit: the remainder decides
    up = 2 * rem > (uint64_t)n || (2 * rem == (uint64_t)n && (keep & 1u));
  } else {
    bool sticky = rem != 0;
    for (int i = t - 2; i >= 0 && !sticky; --i) sticky = qbit(i) != 0u;
    up = qbit(t - 1) && (sticky || (keep & 1u));
  }
  return pack_value<T>(neg, keep + (up ? 1u : 0u), t);
}

template <class T>
__device__ __forceinline__ double stored_value(uint32_t bits) {
  if constexpr (sizeof(T) == 4) return (double)__uint_as_float(bits);
  else if constexpr (std::is_same<T, __half>::value)
    return (double)__half2float(__ushort_as_half((unsigned short)bits));
  else return (double)__uint_as_float(bits << 16);
}

// the adjacent pattern of the type towards +inf (up) or -inf (down)
template <class T>
__device__ __forceinline__ uint32_t neighbour(uint32_t bits, bool up) {
  constexpr uint32_t kSign = sizeof(T) == 4 ? 0x80000000u : 0x8000u;
  if (bits == kSign) return up ? 1u : kSign | 1u;  // -0
  if (bits == 0u) return up ? 1u : kSign | 1u;      // +0
  const bool neg = (bits & kSign) != 0u;
  return (up != neg) ? bits + 1u : bits - 1u;
}

// Knuth's TwoSum: s + x = t + e exactly (round to nearest, no overflow);
// the error's bits are ORed into `inexact` (zero while every addition was
// exact)
__device__ __forceinline__ void two_sum(float &s, float &c, uint32_t &inexact, float x) {
  const float t = s + x;
  const float bp = t - s;
  const float e = (s - (t - bp)) + (x - bp);
  s = t;
  c += e;
  inexact |= __float_as_uint(e);
}

// The mean of one channel from its TwoSum pair (s, c) and sum of magnitudes
// a: the correctly rounded pattern when the error bound settles it, else ~0u
// (the exact path decides).  When no addition rounded (inexact == 0) s is
// the exact sum, and a mean exactly halfway between two values -- frequent
// for sums of a power-of-two count of 16-bit keys -- is settled here too,
// to the even pattern.  Patterns of the type never equal ~0u (it would be a
// NaN of fp32, and 16-bit patterns are below 2^16).
template <class T>
__device__ __forceinline__ uint32_t fast_mean(float s, float c, float a, uint32_t inexact, int n) {
  constexpr uint32_t kSign = sizeof(T) == 4 ? 0x80000000u : 0x8000u;
  if (!isfinite(s) || !isfinite(c) || !isfinite(a)) return ~0u;
  if (a == 0.f) return pack_value<T>(signbit(s), 0u, 0);  // every key is a zero
  if constexpr (sizeof(T) == 2) {
    // A full page (n a power of two), in fp32 only: fp64 arithmetic is slow
    // on this part (the build took 0.86 ms for 1 GiB of keys with it).
    if ((n & (n - 1)) == 0) {
      const float inv = 1.0f / (float)n;  // exact
      auto round16 = [](float x) -> uint32_t {
        if constexpr (std::is_same<T, __half>::value) return __half_as_ushort(__float2half_rn(x));
        else return __bfloat16_as_ushort(__float2bfloat16_rn(x));
      };
      // s exact: s / n is exact too, and its one rounding is the answer (ties
      // to even; a zero keeps the sign of the mean, and keys that cancel give
      // s = +0)
      if (inexact == 0u) return round16(s * inv);
      const uint32_t r = round16(fmaf(c, inv, s * inv));
      const float rv = (float)stored_value<T>(r);
      if (fabsf(rv) < 0x1p120f) {  // n * midpoint below fp32's overflow
        // n * the midpoints: exact (a 16-bit value's neighbours are at most
        // one bit more precise, n a power of two)
        const float lo = n * ((rv + (float)stored_value<T>(neighbour<T>(r, false))) * 0.5f);
        const float hi = n * ((rv + (float)stored_value<T>(neighbour<T>(r, true))) * 0.5f);
        // the bound on (s, c) as below, plus an absolute floor and the
        // roundings of this check's few fp32 operations
        const float err = a * ((float)((n + 2) * (n + 2)) * 0x1p-48f) * (1.0f + 0x1p-10f) +
                          0x1p-149f;
        const float d1 = s - lo, d2 = hi - s;
        const float margin = err + 0x1p-22f * (fabsf(d1) + fabsf(d2) + fabsf(c));
        if (d1 + c > margin && d2 - c > margin) {
          if (rv != 0.f) return r;
          const float t = s + c;  // a zero: the sign of the exact mean
          if (t > margin + 0x1p-22f * fabsf(t)) return pack_value<T>(false, 0u, 0);
          if (t < -(margin + 0x1p-22f * fabsf(t))) return pack_value<T>(true, 0u, 0);
        }
        return ~0u;
      }
    }
  }
  const double sd = (double)s + (double)c;
  const double md = sd / n;
  uint32_t r;
  if constexpr (sizeof(T) == 4) r = __float_as_uint((float)md);
  else if constexpr (std::is_same<T, __half>::value) r = __half_as_ushort(__double2half(md));
  else r = __bfloat16_as_ushort(__double2bfloat16(md));
  if (inexact == 0u) {  // sd is the exact sum, compared exactly below
    if (sd == 0.0) return pack_value<T>(false, 0u, 0);  // non-zero keys cancelling: +0
    const uint32_t dn = neighbour<T>(r, false), up = neighbour<T>(r, true);
    const double rv = stored_value<T>(r);
    const double lo = n * ((rv + stored_value<T>(dn)) * 0.5);
    const double hi = n * ((rv + stored_value<T>(up)) * 0.5);
    uint32_t pick;
    if (sd > lo && sd < hi) pick = r;
    else if (sd == lo) pick = (r & 1u) ? dn : r;  // a tie: the even pattern
    else if (sd == hi) pick = (r & 1u) ? up : r;
    else return ~0u;
    // a zero takes the sign of the exact mean
    if ((pick & ~kSign) == 0u) pick = sd < 0.0 ? kSign : 0u;
    return pick;
  }
  // error bound of (s, c): the n + 1 error terms, each at most 2^-24 of a
  // partial sum, accumulated in fp32 -- (n + 2)^2 2^-48 sum|k| -- with room
  // for this check's roundings (s + c, the products and differences in fp64)
  const double err =
      (double)a * ((double)(n + 2) * (n + 2) * 0x1p-48) * (1.0 + 0x1p-10) + fabs(sd) * 0x1p-50;
  const double rv = stored_value<T>(r);
  const double lo = n * ((rv + stored_value<T>(neighbour<T>(r, false))) * 0.5);
  const double hi = n * ((rv + stored_value<T>(neighbour<T>(r, true))) * 0.5);
  if (!(sd - err > lo && sd + err < hi)) return ~0u;
  if (rv == 0.0) {  // a zero: its sign is the exact mean's, which must be settled
    if (sd > err) return pack_value<T>(false, 0u, 0);
    if (sd < -err) return pack_value<T>(true, 0u, 0);
    return ~0u;
  }
  return r;
}

template <class T>
__global__ void __launch_bounds__(256)
    mean_build_kernel(const T *k, const int32_t *bt,
                      const int32_t *ctx, T *mean, int B, int Hkv,
                      int ps, int maxP, long long nphys, int last_only, int *status) {
  pdl_wait();
  constexpr int C = kHeadDim * (int)sizeof(T) / 16;  // 16-byte chunks per row
  constexpr int RG = 32 / C;                          // row groups per warp
  constexpr int E = 16 / (int)sizeof(T);              // elements per chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * 8 + warp;
  const long long items = (long long)B * (last_only ? 1 : maxP) * Hkv;
  if (item >= items) return;
  const int kvh = (int)(item % Hkv);
  const long long bp = item / Hkv;
  const int b = (int)(last_only ? bp : bp / maxP);
  const int len = ctx[b];
  if (len < 1 || len > maxP * ps) {
    if ((last_only || bp % maxP == 0) && kvh == 0 && lane == 0) flag_error(status, KV_ERR_BOUNDS);
    return;
  }
  const int p = last_only ? (len - 1) / ps : (int)(bp % maxP);
  if (p * ps >= len) return;
  const int n = min(ps, len - p * ps);
  const long long phys = bt[(long long)b * maxP + p];
  if (phys < 0 || phys >= nphys) {
    if (lane == 0) flag_error(status, KV_ERR_BOUNDS);
    return;
  }
  const int chunk = lane % C, rg = lane / C;
  const T *page = k + ((phys * Hkv + kvh) * ps) * kHeadDim;
  const uint4 *src = reinterpret_cast<const uint4 *>(page) + chunk;
  float s[E], c[E], a[E];
  uint32_t inexact[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    s[e] = -0.f;
    c[e] = 0.f;
    a[e] = 0.f;
    inexact[e] = 0u;
  }
#pragma unroll 4
  for (int r = rg; r < n; r += RG) {
    const uint4 x = src[(long long)r * C];
    if constexpr (sizeof(T) == 2) {
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = unpack2(w[j], T());
        two_sum(s[2 * j], c[2 * j], inexact[2 * j], f.x);
        two_sum(s[2 * j + 1], c[2 * j + 1], inexact[2 * j + 1], f.y);
        a[2 * j] += fabsf(f.x);
        a[2 * j + 1] += fabsf(f.y);
      }
    } else {
      const float f[4] = {__uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z),
                          __uint_as_float(x.w)};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        two_sum(s[j], c[j], inexact[j], f[j]);
        a[j] += fabsf(f[j]);
      }
    }
  }
  pdl_trigger();
  if constexpr (RG == 2) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float so = __shfl_xor_sync(0xFFFFFFFFu, s[e], 16);
      const float co = __shfl_xor_sync(0xFFFFFFFFu, c[e], 16);
      inexact[e] |= __shfl_xor_sync(0xFFFFFFFFu, inexact[e], 16);
      two_sum(s[e], c[e], inexact[e], so);
      c[e] += co;
      a[e] += __shfl_xor_sync(0xFFFFFFFFu, a[e], 16);
    }
  }
  if (rg != 0) return;
  uint32_t out[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    out[e] = fast_mean<T>(s[e], c[e], a[e], inexact[e], n);
    if (out[e] == ~0u) out[e] = exact_mean<T>(page, chunk * E + e, n);
  }
  T *dst = mean + (phys * Hkv + kvh) * kHeadDim + chunk * E;
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<uint4 *>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
  } else {
    *reinterpret_cast<uint4 *>(dst) =
        make_uint4(out[0] | (out[1] << 16), out[2] | (out[3] << 16), out[4] | (out[5] << 16),
                   out[6] | (out[7] << 16));
  }
}

}  // namespace

cudaError_t launch_mean_build(int dtype, const void *k, const int32_t *bt, const int32_t *ctx,
                              void *mean, int B, int Hkv, int ps, int maxP, long long nphys,
                              bool last_only, int *status, cudaStream_t st) {
  const long long items = (long long)B * (last_only ? 1 : maxP) * Hkv;
  const unsigned blocks = (unsigned)((items + 7) / 8);
  const int lo = last_only ? 1 : 0;
  switch (dtype) {
    case KV_F32:
      return launch_pdl(mean_build_kernel<float>, dim3(blocks), dim3(256), 0, st,
                        static_cast<const float *>(k), bt, ctx, static_cast<float *>(mean), B,
                        Hkv, ps, maxP, nphys, lo, status);
    case KV_F16:
      return launch_pdl(mean_build_kernel<__half>, dim3(blocks), dim3(256), 0, st,
                        static_cast<const __half *>(k), bt, ctx, static_cast<__half *>(mean), B,
                        Hkv, ps, maxP, nphys, lo, status);
    default:
      return launch_pdl(mean_build_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, st,
                        static_cast<const __nv_bfloat16 *>(k), bt, ctx,
                        static_cast<__nv_bfloat16 *>(mean), B, Hkv, ps, maxP, nphys, lo, status);
  }
}

}  // namespace kvs
