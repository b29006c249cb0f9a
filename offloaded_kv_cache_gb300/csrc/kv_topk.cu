// kv_topk.cu -- top-K page selection, the per-group union of selected pages,
// and the split-K combine of partial attention results.
//
// KVDrive: A Holistic Multi-Tier KV Cache Management System for Long-Context
// LLM Inference, section 2.2: for each query only the Top-K most important
// blocks are retrieved.  Ties go to the lower page index; pages come out
// ascending.
#include "kv_internal.cuh"

namespace kvs {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;

__device__ __forceinline__ uint32_t score_key(float s) {
  // +0.0f folds -0.0 into +0.0 so that equal scores compare equal
  return key32(__float_as_uint(s + 0.0f));
}

// Exclusive prefix count of `flag` over the block in thread order; *total
// receives the block-wide count.  Two block barriers.
__device__ __forceinline__ int block_excl_count(bool flag, int *warp_tot, int *total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned bal = __ballot_sync(0xFFFFFFFFu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(bal);
  __syncthreads();
  int off = 0, tot = 0;
#pragma unroll 8
  for (int w = 0; w < kTopkWarps; ++w) {
    const int t = warp_tot[w];
    off += w < warp ? t : 0;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return off + in_warp;
}

// One CTA per (b, h) row.  Radix select of the K-th largest key, 8 bits per
// pass from the top, over keys cached in shared memory (or re-read from the
// L2-resident score row when the row does not fit); the digit search is one
// warp scanning the 256-bin histogram; the final pass compacts the selected
// pages in index order with ballots.
__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float *__restrict__ scores, const int32_t *__restrict__ ctx, int Hq, int ps,
                int maxP, int K, int keys_in_smem, int32_t *__restrict__ out, int *status) {
  extern __shared__ uint32_t skeys[];
  __shared__ uint32_t hist[256];
  __shared__ int warp_tot[kTopkWarps];
  __shared__ uint32_t s_digit;
  __shared__ int s_krem;
  const int tid = threadIdx.x;
  const long long row = blockIdx.x;
  const int b = (int)(row / Hq);
  int32_t *orow = out + row * K;
  const float *srow = scores + row * maxP;
  const int len = ctx[b];
  if (len < 1 || len > maxP * ps) {
    if (tid == 0) flag_error(status, KV_ERR_BOUNDS);
    for (int i = tid; i < K; i += kTopkThreads) orow[i] = -1;
    return;
  }
  const int P = (len + ps - 1) / ps;
  const int keff = min(K, P);
  if (keff == P) {  // every page is selected
    for (int i = tid; i < K; i += kTopkThreads) orow[i] = i < P ? i : -1;
    return;
  }
  if (keys_in_smem) {
    for (int p = tid; p < P; p += kTopkThreads) skeys[p] = score_key(srow[p]);
    __syncthreads();
  }
  auto key_at = [&](int p) -> uint32_t {
    return keys_in_smem ? skeys[p] : score_key(srow[p]);
  };

  uint32_t prefix = 0, pmask = 0;
  int krem = keff;  // how many of the keys matching `prefix` still have to be taken
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += kTopkThreads) {
      const uint32_t k = key_at(p);
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits 255-8l .. 248-8l, scanned from the top
      int c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = (int)hist[255 - 8 * tid - j];
        sum += c[j];
      }
      int incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (tid >= off) incl += t;
      }
      int above = incl - sum;  // keys whose digit beats this lane's range
      if (above < krem && krem <= incl) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (above + c[j] >= krem) {
            s_digit = (uint32_t)(255 - 8 * tid - j);
            s_krem = krem - above;
            break;
          }
          above += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    pmask |= 255u << shift;
    krem = s_krem;
  }
  // prefix is now the K-th largest key; krem keys equal to it are taken,
  // lowest page index first.
  const uint32_t tau = prefix;
  int eq_carry = 0, sel_carry = 0;
#pragma unroll 1
  for (int base = 0; base < P; base += kTopkThreads) {
    const int p = base + tid;
    const uint32_t k = p < P ? key_at(p) : 0u;
    const bool eq = p < P && k == tau;
    const bool gt = p < P && k > tau;
    int eq_tot, sel_tot;
    const int eq_rank = block_excl_count(eq, warp_tot, &eq_tot);
    const bool sel = gt || (eq && eq_carry + eq_rank < krem);
    const int pos = block_excl_count(sel, warp_tot, &sel_tot);
    if (sel && sel_carry + pos < K) orow[sel_carry + pos] = p;
    eq_carry += eq_tot;
    sel_carry += sel_tot;
  }
  for (int i = keff + tid; i < K; i += kTopkThreads) orow[i] = -1;
}

// ---------------------------------------------------------------------------
// union of the selected pages of the gc heads of one (b, kv head, head chunk)
// ---------------------------------------------------------------------------
constexpr int kUnionThreads = 512;

__global__ void __launch_bounds__(kUnionThreads)
    union_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ ctx, int Hq, int G,
                 int gc, int ps, int maxP, int K, int umax, int32_t *__restrict__ upages,
                 uint32_t *__restrict__ umasks, int32_t *__restrict__ ucount, int *status) {
  extern __shared__ uint32_t words[];  // one byte of head bits per page, 4 pages a word
  __shared__ int warp_tot[kUnionThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = blockIdx.x, b = blockIdx.y;
  const int nchunk = G / gc;
  const int kvh = grp / nchunk, chunk = grp % nchunk;
  const int head0 = kvh * G + chunk * gc;
  const long long gbase = ((long long)b * gridDim.x + grp);
  const int len = ctx[b];
  if (len < 1 || len > maxP * ps) {
    if (tid == 0) {
      flag_error(status, KV_ERR_BOUNDS);
      ucount[gbase] = 0;
    }
    return;
  }
  const int P = (len + ps - 1) / ps;
  const int nw = (P + 3) / 4;
  for (int i = tid; i < nw; i += kUnionThreads) words[i] = 0u;
  __syncthreads();
  for (int i = tid; i < gc * K; i += kUnionThreads) {
    const int g = i / K, j = i % K;
    const int p = idx[((long long)b * Hq + head0 + g) * K + j];
    if (p < 0) continue;
    if (p >= P) {
      flag_error(status, KV_ERR_BOUNDS);
      continue;
    }
    atomicOr(&words[p >> 2], (1u << g) << ((p & 3) * 8));
  }
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < P; base += kUnionThreads) {
    const int p = base + tid;
    const uint32_t m = p < P ? (words[p >> 2] >> ((p & 3) * 8)) & 0xFFu : 0u;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, m != 0u);
    if (lane == 0) warp_tot[warp] = __popc(bal);
    __syncthreads();
    int off = 0, tot = 0;
    for (int w = 0; w < kUnionThreads / 32; ++w) {
      off += w < warp ? warp_tot[w] : 0;
      tot += warp_tot[w];
    }
    __syncthreads();
    const int pos = carry + off + __popc(bal & ((1u << lane) - 1u));
    if (m != 0u && pos < umax) {
      upages[gbase * umax + pos] = p;
      umasks[gbase * umax + pos] = m;
    }
    carry += tot;
  }
  if (tid == 0) ucount[gbase] = min(carry, umax);
}

// ---------------------------------------------------------------------------
// split-K combine: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kHeadDim)
    combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_ml,
                   float *__restrict__ out, int S, long long rows) {
  const long long r = blockIdx.x;
  const int c = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, part_ml[(s * rows + r) * 2]);
  float o = 0.f, l = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float m = part_ml[(s * rows + r) * 2];
      const float w = m == -INFINITY ? 0.f : ex2(m - M);
      o = fmaf(w, part_o[(s * rows + r) * kHeadDim + c], o);
      l = fmaf(w, part_ml[(s * rows + r) * 2 + 1], l);
    }
  }
  out[r * kHeadDim + c] = l > 0.f ? o / l : 0.f;
}

}  // namespace

cudaError_t launch_topk(const float *scores, const int32_t *ctx, int B, int Hq, int ps, int maxP,
                        int k, int32_t *indices, int *status, cudaStream_t st) {
  constexpr size_t kMaxSmemKeys = 48 * 1024 / 4;  // keys cached in shared memory
  const int in_smem = (size_t)maxP <= kMaxSmemKeys ? 1 : 0;
  const size_t smem = in_smem ? (size_t)maxP * 4 : 0;
  topk_kernel<<<(unsigned)((long long)B * Hq), kTopkThreads, smem, st>>>(scores, ctx, Hq, ps, maxP,
                                                                       k, in_smem, indices, status);
  return cudaGetLastError();
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
  union_kernel<<<grid, kUnionThreads, smem, st>>>(indices, ctx, Hq, G, gc, ps, maxP, k, umax,
                                                  upages, umasks, ucount, status);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float *part_o, const float *part_ml, float *out, int S, int B,
                           int Hq, cudaStream_t st) {
  const long long rows = (long long)B * Hq;
  combine_kernel<<<(unsigned)rows, kHeadDim, 0, st>>>(part_o, part_ml, out, S, rows);
  return cudaGetLastError();
}

}  // namespace kvs
