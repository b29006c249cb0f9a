// kv_attn.cuh -- paged decode attention (dense or over selected pages) for
// sm_103a: one producer warp streams K/V pages into a ring of shared-memory
// stages, consumer warps run a streaming softmax over them.
//
// What it computes, per query head h of sequence b:
//   out = sum_t softmax_t(scale * q . k_t) v_t
// over the valid tokens of every page (dense) or of the pages head h selected
// (sparse).  Sources: KVDrive (A Holistic Multi-Tier KV Cache Management
// System for Long-Context LLM Inference), section 2.3 step (3), attention over
// the selected entries; DirectKV (No Buffer, No Bottleneck: Efficient
// Zero-Copy KV Cache Offloading for Long-Context LLMs), core method 2-3: in
// decode the query and the output stay on chip, every K/V tile is scanned
// once, a producer warp prefetches the next tile while consumers compute the
// current one, and the softmax is streamed.
//
// Design on GB300:
//  * CTA = (split, kv head x head chunk, sequence).  All GC query heads of
//    the chunk share one pass over the K/V bytes; in the sparse path the CTA
//    walks the union of their selected pages once and masks per head.
//  * Stage = one 16-token tile of one page of one kv head: K then V, each 16
//    rows x 128 elements, stored as 128-byte slabs in the 128B-swizzled
//    layout, so ldmatrix and 16-byte shared loads are bank-conflict free.  A
//    page of ps tokens is ps / 16 consecutive tiles.
//  * Producer: HBM -> TMA tiled loads (cp.async.bulk.tensor, one 3-D box of
//    every slab of the tile for K and one for V) completing on a full
//    mbarrier with a transaction count; pinned host memory -> 16-byte
//    cp.async issued by the 32 producer lanes (same layout, same barrier).
//    Stage s always belongs to consumer warp s % nw, which arrives on the
//    stage's empty mbarrier when done.  The number of consumer warps nw and
//    of stages are launch parameters: many short (sequence, head) units run
//    as small CTAs, all resident in one wave; long units as deep CTAs.
//  * Consumers: GQA groups of >= 4 heads on 16-bit data use mma.sync
//    m16n8k16 (tokens x heads tile of q.K^T, then V^T . P^T with P split in a
//    high and a low 16-bit part so the weights keep ~16 bits); otherwise
//    CUDA-core FMAs with lanes over (token, slab) for q.k and over channels
//    for p.v.  Max/sum reductions are warp shuffles.
//  * Window instantiations (WIN): K/V are the GPU-resident page window and
//    the pages the window update marked in fetch_bits come from the source
//    cache instead.  The producer fills a window page's stage by TMA and a
//    fetched page's stage by cp.async from the (host-mapped) source; the
//    consumer that used a fetched tile stores its valid rows into the page's
//    window slot.  The host-link reads of the misses so overlap the HBM reads
//    of the hits, and no separate copy pass runs before the attention.
//  * Every mbarrier wait is bounded in wall time; a wait that gives up
//    records KV_ERR_DEVICE_TIMEOUT and the CTA winds down.
#pragma once

#include "kv_internal.cuh"

namespace kvs {

// shared memory before the ring: barriers, q and weights (attn_fixed_header),
// then the page list (a.header_bytes in total, a multiple of 1024)

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, __nv_bfloat16) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, __half) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// (hi, lo) 16-bit pairs with x ~= hi + lo to ~16 significant bits
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t &hi, uint32_t &lo,
                                           __nv_bfloat16) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t &hi, uint32_t &lo,
                                           __half) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

// per-CTA page list: the j-th page of this CTA's share
struct PageRange {
  int lo, n;  // first index into the (dense or union) list, count
};

// ---------------------------------------------------------------------------
// equal chunks of the concatenated union lists (AttnArgs::spread)
// ---------------------------------------------------------------------------
// With every group's list split over the same S CTAs, a group whose union is
// larger than the others' gives its CTAs more pages, and the call ends with
// them: rows of different context lengths in one batch, or GQA groups whose
// heads agree less on their pages.  Instead, CTA i of N can take entries
// [i T / N, (i + 1) T / N) of the groups' lists laid end to end (T entries,
// groups in (sequence, kv head) order).  When every group holds at least
// ceil(T / N) entries, a chunk meets at most two groups: the tail of one
// (segment A) and the head of the next (segment B).
struct SpreadShare {
  bool on;
  int T;                 // entries of all groups
  int gA, offA, lenA;    // segment A: entries offA .. offA + lenA - 1 of group gA
  int gB, lenB;          // segment B (lenB > 0): entries 0 .. lenB - 1 of group gB
};

// Step 1, every thread of the CTA after the PDL wait: the groups' list
// lengths into pre[1 .. ngroups] (shared memory), and the decision, the same
// in every CTA.  a.spread 2 takes equal chunks whenever they are possible; 1
// only when the per-group split's longest CTA holds at least
// a.spread_min_gain bytes more K/V than an equal chunk (the price of the
// prefix sums' round trip before the first load and of the longer combine).
// red: 96 ints of scratch.
__device__ __forceinline__ SpreadShare spread_decide(const AttnArgs &a, long long ncta,
                                                     int page_bytes, int32_t *pre, int *red) {
  const int NG = a.ngroups;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = blockDim.x >> 5;
  const int per = (NG + (int)blockDim.x - 1) / (int)blockDim.x;
  const int g0 = min(NG, t * per), g1 = min(NG, g0 + per);
  int sum = 0, mn = INT_MAX, mx = 0;
  for (int g = g0; g < g1; ++g) {
    const int l = ld_issue(a.context_lens + g / a.Hkv);
    const int cnt = ld_issue(a.union_count + g);
    const bool bad = l < 1 || l > a.maxP * a.ps;  // such a row's list is empty
    const int u = bad ? 0 : min(max(cnt, 0), a.umax);
    pre[g + 1] = u;
    sum += u;
    mn = min(mn, u);
    mx = max(mx, u);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
    mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  }
  if (lane == 0) {
    red[warp] = sum;
    red[32 + warp] = mn;
    red[64 + warp] = mx;
  }
  __syncthreads();
  int T = 0, minU = INT_MAX, maxU = 0;
  for (int w = 0; w < nwarps; ++w) {
    T += red[w];
    minU = min(minU, red[32 + w]);
    maxU = max(maxU, red[64 + w]);
  }
  SpreadShare sh{};
  sh.T = T;
  sh.on = T >= ncta && (long long)minU * ncta >= T;
  if (sh.on && a.spread == 1) {
    const int S = a.num_splits;
    const long long chunk = (T + ncta - 1) / ncta;
    sh.on = ((long long)(maxU + S - 1) / S - chunk) * page_bytes >= a.spread_min_gain;
  }
  return sh;
}

// Step 2, when sh.on: prefix sums of the lengths in pre[0 .. ngroups] and this
// CTA's chunk.  Every thread; red: 32 ints of scratch (reused).
__device__ __forceinline__ void spread_share(const AttnArgs &a, long long cta, long long ncta,
                                             int32_t *pre, int *red, SpreadShare &sh) {
  const int NG = a.ngroups;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = blockDim.x >> 5;
  const int per = (NG + (int)blockDim.x - 1) / (int)blockDim.x;
  const int g0 = min(NG, t * per), g1 = min(NG, g0 + per);
  int sum = 0;
  for (int g = g0; g < g1; ++g) sum += pre[g + 1];
  int inc = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int x = __shfl_up_sync(0xFFFFFFFFu, inc, off);
    if (lane >= off) inc += x;
  }
  __syncthreads();  // every warp has read red[] of step 1
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp && w < nwarps; ++w) base += red[w];
  int run = base + inc - sum;
  if (t == 0) pre[0] = 0;
  for (int g = g0; g < g1; ++g) {
    run += pre[g + 1];
    pre[g + 1] = run;
  }
  __syncthreads();
  const int T = sh.T;
  const long long c0 = cta * T / ncta, c1 = (cta + 1) * T / ncta;
  int lo = 0, hi = NG - 1;  // the group holding entry c0: the last g with pre[g] <= c0
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= c0) lo = mid;
    else hi = mid - 1;
  }
  const long long endA = min(c1, (long long)pre[lo + 1]);
  sh.gA = lo;
  sh.offA = (int)(c0 - pre[lo]);
  sh.lenA = (int)(endA - c0);
  sh.gB = lo + 1;
  sh.lenB = (int)(c1 - endA);
}

// gmeta of group g, written by the CTA whose chunk holds the group's first
// entry: the CTAs first..last whose chunks meet g, and whether the last one
// goes on past g's end (then g is its segment A).  Chunk of entry e: the last
// i with i T / N <= e, that is ((e + 1) N - 1) / T.
__device__ __forceinline__ void spread_meta(const AttnArgs &a, const int32_t *pre, int g,
                                            long long cta, long long ncta, int T) {
  const long long end = pre[g + 1];  // one past g's last entry
  const long long last = (end * ncta - 1) / T;
  const long long next = (last + 1) * T / ncta;  // where that chunk ends
  reinterpret_cast<int4 *>(a.gmeta)[g] =
      make_int4(kSplitSpread, (int)cta, (int)last, next > end ? 1 : 0);
}
// one page of the list, resolved once in the prologue: physical page (-1 when
// the entry is out of range) and (valid tokens | head mask << 8); the window
// instantiations add the source page to fetch (-1: the window slot holds it)
template <bool WIN>
struct PageEnt {
  int phys;
  int info;
};
template <>
struct PageEnt<true> {
  int phys;
  int info;
  int src;
  int pad;
};

template <class T, int GC, bool MMA, bool WIN>
__global__ void __launch_bounds__(kAttnMaxThreads)
    attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv) {
  using Ent = PageEnt<WIN>;
  static_assert(sizeof(Ent) == attn_entry_bytes(WIN), "page-list entry size");
  // the producer's first TMA needs the tensor maps: fetch them while the
  // prologue runs
  if (a.use_tma && threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tv)) : "memory");
  }
  if constexpr (MMA) pdl_wait();
  constexpr int SL = (int)sizeof(T);        // 128-byte slabs per 128-element row
  constexpr int EPS = 128 / (int)sizeof(T); // elements per slab
  constexpr int EPC = 16 / (int)sizeof(T);  // elements per 16-byte chunk
  constexpr int TP = 32 / SL;               // tokens per CUDA-core pass
  constexpr int QSTR = EPS + 4;             // padded q slab stride (floats)

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + kMaxStages;
  float *q_s = reinterpret_cast<float *>(smem + 256);  // CUDA core: [GC][SL][QSTR]
  float *pbuf = q_s + GC * SL * QSTR;                  // CUDA core: [warps][GC][TP]
  Ent *plist = reinterpret_cast<Ent *>(smem + attn_fixed_header(SL, GC, MMA));
  uint8_t *stages = smem + a.header_bytes;

  constexpr int TT = kTileTokens;            // tokens per tile (stage)
  constexpr int slab_bytes = TT * 128;
  constexpr int kv_off = TT * 128 * SL;      // V follows K inside a stage
  constexpr int stage_bytes = 2 * kv_off;
  const int ps = a.ps;
  const int UPP = ps / TT;                   // tiles per page
  const int NS = a.nstages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, grp = blockIdx.y, b = blockIdx.z;
  const int kvh = grp / a.nchunk, chunk = grp % a.nchunk;
  const int head0 = kvh * a.G + chunk * GC;

  if constexpr (!MMA) {
    // CUDA-core path: the barriers before waiting for the previous kernel in
    // the stream, and, when that kernel is known to be one of the library's
    // (a.early_inputs), q in shared memory and the block table too, so that
    // they overlap that kernel's tail (OPT-6.7B dense 46.7 -> 46.0 us for q;
    // the block table below, 46.33 -> 46.20 us).
    if (threadIdx.x == 0) {
      for (int s = 0; s < a.nstages; ++s) {
        mbar_init(smem_u32(&full[s]), a.use_tma && !WIN ? 1u : 32u);
        mbar_init(smem_u32(&empty[s]), 1u);
      }
      fence_mbar_init();
    }
    if (!a.early_inputs) pdl_wait();
    for (int i = threadIdx.x; i < GC * kHeadDim; i += blockDim.x) {
      const int g = i / kHeadDim, c = i % kHeadDim;
      const T *qrow = static_cast<const T *>(a.q) + ((long long)b * a.Hq + head0 + g) * kHeadDim;
      q_s[(g * SL + c / EPS) * QSTR + (c % EPS)] = Elem<T>::to_f32(qrow[c]);
    }
    // A dense CTA with the whole row (one split) lists pages [0, P), P <= maxP:
    // their block-table entries load here too, into the entries the same
    // thread resolves below.
    if (!WIN && a.union_pages == nullptr && a.num_splits == 1) {
      for (int j = threadIdx.x; j < min(a.maxP, kMaxListPages); j += blockDim.x)
        plist[j].phys = a.block_table[(long long)b * a.maxP + j];
    }
    if (a.early_inputs) pdl_wait();
  }
  const bool sparse = a.union_pages != nullptr;
  const long long gidx = (long long)b * gridDim.y + grp;
  // (launch plans use 128 or 160 threads; the page list needs at least 128)
  if (blockDim.x < 128) {
    if (threadIdx.x == 0) flag_error(a.status, KV_ERR_BOUNDS);
    return;
  }

  // ---- this CTA's share of the page list ---------------------------------
  // Sparse: split s of S takes union entries s, s + S, s + 2S, ... (still in
  // page order), so its entries load together with the length and the union
  // count instead of after them (a contiguous share needs the count first).
  // Dense: a contiguous range of pages.  kSpec entries per thread cover
  // kMaxListPages with the smallest CTA (128 threads).
  constexpr int kSpec = (kMaxListPages + 127) / 128;
  const int S = a.num_splits;
  int32_t sp_page[kSpec];
  uint32_t sp_mask[kSpec];
  PageRange rng;
  // equal chunks of all groups' lists (spread): segment A of group (bA, kvhA)
  // is entries 0 .. segB - 1 of this CTA's list, segment B of (bB, kvhB) the
  // rest; the split per group has one segment, this CTA's own group
  bool spread = false;
  int segB = INT_MAX, gA = (int)gidx;
  int bA = b, kvhA = kvh, bB = b, kvhB = kvh;
  const int len = ld_issue(a.context_lens + b);  // in flight with the entries below
  if (sparse) {
#pragma unroll
    for (int u = 0; u < kSpec; ++u) {
      const int j = threadIdx.x + u * blockDim.x;
      const long long e = split + (long long)j * S;
      sp_page[u] = -1;
      sp_mask[u] = 0u;
      if (j < kMaxListPages && e < a.umax) {
        sp_page[u] = ld_issue(a.union_pages + gidx * a.umax + e);
        sp_mask[u] = ld_issue(a.union_masks + gidx * a.umax + e);
      }
    }
  }
  if constexpr (MMA && !WIN) {
    if (a.spread) {
      // the groups' lengths load together with the entries above (the split
      // per group's), so keeping that split costs no extra round trip
      const long long ncta = (long long)gridDim.x * a.ngroups;
      const long long cta = (long long)split * a.ngroups + gidx;
      int32_t *pre = reinterpret_cast<int32_t *>(stages);  // the idle ring
      int *red = pre + ((a.ngroups + 1 + 31) & ~31);
      SpreadShare sh = spread_decide(a, ncta, (int)(2 * ps * kHeadDim * sizeof(T)), pre, red);
      spread = sh.on;
      if (spread) {
        spread_share(a, cta, ncta, pre, red, sh);
        if (threadIdx.x == 0) {
          if (sh.offA == 0) spread_meta(a, pre, sh.gA, cta, ncta, sh.T);
          if (sh.lenB > 0) spread_meta(a, pre, sh.gB, cta, ncta, sh.T);
        }
        const int n = sh.lenA + sh.lenB;  // at most ceil(T / N) <= kMaxListPages
#pragma unroll
        for (int u = 0; u < kSpec; ++u) {
          const int j = threadIdx.x + u * blockDim.x;
          sp_page[u] = -1;
          sp_mask[u] = 0u;
          if (j < n && j < kMaxListPages) {
            const long long e = j < sh.lenA ? (long long)sh.gA * a.umax + sh.offA + j
                                            : (long long)sh.gB * a.umax + (j - sh.lenA);
            sp_page[u] = a.union_pages[e];
            sp_mask[u] = a.union_masks[e];
          }
        }
        rng.lo = 0;
        rng.n = min(n, kMaxListPages);
        gA = sh.gA;
        bA = bB = gA / a.Hkv;
        kvhA = kvhB = gA % a.Hkv;
        if (sh.lenB > 0) {
          segB = sh.lenA;
          bB = sh.gB / a.Hkv;
          kvhB = sh.gB % a.Hkv;
        }
      } else if (split == 0 && threadIdx.x == 0) {
        reinterpret_cast<int4 *>(a.gmeta)[gidx] = make_int4(kSplitPerGroup, 0, 0, 0);
      }
      // the ring that held the lengths is next written by TMA
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
  }
  const bool bad_len = len < 1 || len > a.maxP * ps;
  const int P = bad_len ? 0 : (len + ps - 1) / ps;
  if (spread) {
    // rng set above
  } else if (sparse) {
    const int total = bad_len ? 0 : min(a.union_count[gidx], a.umax);
    rng.lo = split;
    rng.n = total > split ? min((total - split + S - 1) / S, kMaxListPages) : 0;
  } else {
    const int per = (P + S - 1) / S;
    rng.lo = min(P, split * per);
    rng.n = max(0, min(min(P, rng.lo + per) - rng.lo, kMaxListPages));
  }
  const int ntiles = rng.n * UPP;
  if (bad_len && split == 0 && threadIdx.x == 0 && chunk == 0) flag_error(a.status, KV_ERR_BOUNDS);

  if (MMA && threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), a.use_tma && !WIN ? 1u : 32u);
      mbar_init(smem_u32(&empty[s]), 1u);
    }
    fence_mbar_init();
  }
  // Resolve this CTA's page list once (block table, union list, valid tokens,
  // head masks), all threads in parallel, so no tile waits on a dependent
  // global load later.
#pragma unroll
  for (int u = 0; u < kSpec; ++u) {
    const int j = threadIdx.x + u * blockDim.x;
    if (j >= rng.n) break;
    if constexpr (!WIN) {
      if (sparse && a.union_resolved) {
        // the fused selection's entries: physical page, valid tokens | mask << 8
        const int ph = sp_page[u];
        Ent ent{};
        ent.phys = -1;
        if (ph >= 0 && ph < a.nphys) {
          ent.phys = ph;
          ent.info = (int)sp_mask[u];
        } else {
          flag_error(a.status, KV_ERR_BOUNDS);
        }
        plist[j] = ent;
        continue;
      }
    }
    int p;
    uint32_t mask;
    if (sparse) {
      p = sp_page[u];
      mask = sp_mask[u];
    } else {
      p = rng.lo + j;
      mask = (1u << GC) - 1u;
    }
    Ent ent{};
    ent.phys = -1;
    if constexpr (WIN) ent.src = -1;
    if (p >= 0 && p < P) {
      long long ph;
      if constexpr (WIN) {  // the page's slot in the window (page b*C + slot)
        const long long gk = (long long)b * a.Hkv + kvh;
        const int sl = a.page_slot[gk * a.maxP + p];
        ph = (sl >= 0 && sl < a.cache_C) ? (long long)b * a.cache_C + sl : -1;
        if (ph >= 0 && ((a.fetch_bits[gk * a.fetch_words + (p >> 5)] >> (p & 31)) & 1u)) {
          const long long sp = a.block_table[(long long)b * a.maxP + p];
          if (sp >= 0 && sp < a.src_nphys) ent.src = (int)sp;
          else ph = -1;
        }
      } else if (!MMA && !sparse && a.num_splits == 1) {
        ph = plist[j].phys;  // loaded above (p == j)
      } else {
        ph = a.block_table[(long long)b * a.maxP + p];
      }
      if (ph >= 0 && ph < a.nphys) {
        ent.phys = (int)ph;
        ent.info = min(ps, len - p * ps) | (int)(mask << 8);
      }
    }
    if (ent.phys < 0) flag_error(a.status, KV_ERR_BOUNDS);
    plist[j] = ent;
  }
  __syncthreads();

  if (warp == 0) {
    // ======================= producer =====================================
    int issued = 0;
    bool ok = true;
    if constexpr (WIN) {
      // all 32 lanes: a fetched page by cp.async from the source (each lane
      // arrives when its copies land), a window page by TMA (lane 0 arms the
      // transaction count, the other lanes arrive at once)
      const char *kbase = static_cast<const char *>(a.src_k);
      const char *vbase = static_cast<const char *>(a.src_v);
      constexpr int chunks = TT * SL * 8;  // 16-byte chunks per K (or V) tile
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(smem_u32(&empty[s]), ((j / NS) - 1) & 1, a.wait_limit_ns)) {
          if (lane == 0) flag_error(a.status, KV_ERR_DEVICE_TIMEOUT);
          ok = false;
          break;
        }
        const Ent ent = plist[j / UPP];
        issued = j + 1;
        if (j == a.debug_skip_page) continue;
        const uint32_t fb = smem_u32(&full[s]);
        const uint32_t dst = smem_u32(stages + (size_t)s * stage_bytes);
        if (ent.src >= 0) {
          const size_t src0 =
              ((size_t)(((long long)ent.src * a.Hkv + kvh) * ps) + (size_t)(j % UPP) * TT) *
              (SL * 128);
          for (int i = lane; i < chunks; i += 32) {
            const int row = i / (SL * 8), rem = i % (SL * 8);
            const uint32_t d = dst + (rem >> 3) * slab_bytes + swz(row, rem & 7);
            const size_t off = src0 + (size_t)row * (SL * 128) + rem * 16;
            cp_async16(d, kbase + off);
            cp_async16(d + kv_off, vbase + off);
          }
          cp_async_arrive_noinc(fb);
        } else if (lane == 0) {
          const long long phys = max(ent.phys, 0);
          const int row0 = (int)((phys * a.Hkv + kvh) * ps) + (j % UPP) * TT;
          mbar_arrive_expect_tx(fb, (uint32_t)stage_bytes);
          tma_load_3d(dst, &tk, 0, row0, 0, fb);  // every slab of the K tile
          tma_load_3d(dst + kv_off, &tv, 0, row0, 0, fb);
        } else {
          mbar_arrive(fb);
        }
      }
    } else if (a.use_tma) {
      if (lane == 0) {
        for (int j = 0; j < ntiles; ++j) {
          const int s = j % NS;
          if (j >= NS && !mbar_wait(smem_u32(&empty[s]), ((j / NS) - 1) & 1, a.wait_limit_ns)) {
            flag_error(a.status, KV_ERR_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          // a bad entry still fills its stage (from page 0); the consumer skips it
          const long long phys = max(plist[j / UPP].phys, 0);
          issued = j + 1;
          if (j == a.debug_skip_page) continue;
          const uint32_t fb = smem_u32(&full[s]);
          const uint32_t dst = smem_u32(stages + (size_t)s * stage_bytes);
          const int kh = j / UPP < segB ? kvhA : kvhB;
          const int row0 = (int)((phys * a.Hkv + kh) * ps) + (j % UPP) * TT;
          mbar_arrive_expect_tx(fb, (uint32_t)stage_bytes);
          tma_load_3d(dst, &tk, 0, row0, 0, fb);  // every slab of the K tile
          tma_load_3d(dst + kv_off, &tv, 0, row0, 0, fb);
        }
      }
    } else {
      const char *kbase = static_cast<const char *>(a.k);
      const char *vbase = static_cast<const char *>(a.v);
      constexpr int chunks = TT * SL * 8;  // 16-byte chunks per K (or V) tile
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(smem_u32(&empty[s]), ((j / NS) - 1) & 1, a.wait_limit_ns)) {
          if (lane == 0) flag_error(a.status, KV_ERR_DEVICE_TIMEOUT);
          ok = false;
          break;
        }
        const long long phys = max(plist[j / UPP].phys, 0);
        issued = j + 1;
        if (j == a.debug_skip_page) continue;
        const int kh = j / UPP < segB ? kvhA : kvhB;
        const size_t src0 =
            ((size_t)((phys * a.Hkv + kh) * ps) + (size_t)(j % UPP) * TT) * (SL * 128);
        const uint32_t dst = smem_u32(stages + (size_t)s * stage_bytes);
        for (int i = lane; i < chunks; i += 32) {
          const int row = i / (SL * 8), rem = i % (SL * 8);
          const int h = rem >> 3, c = rem & 7;
          const size_t off = src0 + (size_t)row * (SL * 128) + rem * 16;
          const uint32_t d = dst + h * slab_bytes + swz(row, c);
          cp_async16(d, kbase + off);
          cp_async16(d + kv_off, vbase + off);
        }
        cp_async_arrive_noinc(smem_u32(&full[s]));
      }
    }
    (void)ok;
    // Drain: wait (bounded) until the last fill of every stage has landed, so
    // no asynchronous copy targets this CTA's shared memory after it moves on.
    if (lane == 0 || !a.use_tma || WIN) {
      for (int s = 0; s < NS && s < issued; ++s) {
        int jl = s + ((issued - 1 - s) / NS) * NS;  // last page issued into stage s
        if (jl == a.debug_skip_page) jl -= NS;
        if (jl < 0) continue;
        if (!mbar_wait(smem_u32(&full[s]), (jl / NS) & 1, a.wait_limit_ns))
          flag_error(a.status, KV_ERR_DEVICE_TIMEOUT);
      }
      // and, whatever the waits saw, none of this lane's cp.async is in flight
      if (WIN || !a.use_tma) cp_async_wait_all();
    }
    __syncwarp();
  }

  // ======================= consumers ======================================
  const int cw = warp - 1;
  float m_run[MMA ? 2 : GC], l_run[MMA ? 2 : GC];
  float acc[MMA ? 8 : GC][4];
#pragma unroll
  for (int i = 0; i < (MMA ? 2 : GC); ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < (MMA ? 8 : GC); ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  const int gid = lane >> 2, tig = lane & 3;
  if (warp > 0) {
    uint32_t qb[8][2];
    // q as the B operand (k = channel, n = head): b0 = channels 16j+2tig..+1,
    // b1 = channels 16j+8+2tig..+1 of head gid; heads >= GC are zero.
    auto load_q = [&](int bq, int h0q) {
#pragma unroll
      for (int j8 = 0; j8 < 8; ++j8) {
        qb[j8][0] = qb[j8][1] = 0u;
        if (gid < GC) {
          const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
              static_cast<const T *>(a.q) + ((long long)bq * a.Hq + h0q + gid) * kHeadDim);
          qb[j8][0] = qrow[(16 * j8 + 2 * tig) >> 1];
          qb[j8][1] = qrow[(16 * j8 + 8 + 2 * tig) >> 1];
        }
      }
    };
    // spread: this warp's state for segment A goes out as one of the group's
    // nw warp partials, and the warp starts segment B afresh
    const int jB = segB == INT_MAX ? INT_MAX : segB * UPP;  // first tile of segment B
    bool in_b = false;
    auto finish_a = [&]() {
      if constexpr (MMA) {
        float l0 = l_run[0], l1 = l_run[1];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
          l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
        }
        const long long slot = ((long long)gA * a.nw + cw) * GC;
        float *po = a.spa_o + slot * kHeadDim;
        float *pml = a.spa_ml + slot * 2;
        const int h0 = 2 * tig, h1 = h0 + 1;
        if (gid == 0) {
          if (h0 < GC) { pml[2 * h0] = m_run[0]; pml[2 * h0 + 1] = l0; }
          if (h1 < GC) { pml[2 * h1] = m_run[1]; pml[2 * h1 + 1] = l1; }
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int d0 = 16 * mt + gid, d1 = d0 + 8;
          if (h0 < GC) { po[h0 * kHeadDim + d0] = acc[mt][0]; po[h0 * kHeadDim + d1] = acc[mt][2]; }
          if (h1 < GC) { po[h1 * kHeadDim + d0] = acc[mt][1]; po[h1 * kHeadDim + d1] = acc[mt][3]; }
          acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
        }
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
      }
      in_b = true;
    };
    if constexpr (MMA) load_q(bA, kvhA * a.G + chunk * GC);
    const float sl = a.scale_log2;
#pragma unroll 1
    for (int j = cw; j < ntiles; j += a.nw) {
      if (j >= jB && !in_b) {
        finish_a();
        if constexpr (MMA) load_q(bB, kvhB * a.G);
      }
      const int s = j % NS;
      if (!mbar_wait(smem_u32(&full[s]), (j / NS) & 1, a.wait_limit_ns)) {
        if (lane == 0) flag_error(a.status, KV_ERR_DEVICE_TIMEOUT);
        break;
      }
      const Ent ent = plist[j / UPP];
      const uint32_t msk = (uint32_t)ent.info >> 8;
      // valid tokens of this tile (0 for a bad entry)
      const int nv = ent.phys >= 0 ? max(0, min(TT, (ent.info & 0xFF) - (j % UPP) * TT)) : 0;
      uint8_t *st = stages + (size_t)s * stage_bytes;
      if constexpr (MMA) {
        const uint32_t kb = smem_u32(st), vb = kb + kv_off;
        if (nv > 0 && nv < TT) {
          // zero the V rows past the last valid token (P is 0 there, but
          // 0 * NaN would not be)
          for (int i = lane; i < (TT - nv) * SL * 8; i += 32) {
            const int row = nv + i / (SL * 8), rem = i % (SL * 8);
            *reinterpret_cast<uint4 *>(st + kv_off + (rem >> 3) * slab_bytes + swz(row, rem & 7)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
#pragma unroll 1
        for (int sub = 0; sub * 16 < nv; ++sub) {
          float c[4] = {0.f, 0.f, 0.f, 0.f};
          {
            const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int tok = sub * 16 + r;
#pragma unroll
            for (int j8 = 0; j8 < 8; ++j8) {
              const int ch = 2 * j8 + (lane >> 4);
              uint32_t af[4];
              ldsm_x4(kb + (ch >> 3) * slab_bytes + swz(tok, ch & 7), af);
              mma16816(c, af, qb[j8][0], qb[j8][1], T());
            }
          }
          const int t0 = sub * 16 + gid, t1 = t0 + 8;
          const bool v0 = t0 < nv, v1 = t1 < nv;
          const bool s0 = (msk >> (2 * tig)) & 1u, s1 = (msk >> (2 * tig + 1)) & 1u;
          const float z00 = (v0 && s0) ? c[0] * sl : -INFINITY;
          const float z01 = (v0 && s1) ? c[1] * sl : -INFINITY;
          const float z10 = (v1 && s0) ? c[2] * sl : -INFINITY;
          const float z11 = (v1 && s1) ? c[3] * sl : -INFINITY;
          float tm0 = fmaxf(z00, z10), tm1 = fmaxf(z01, z11);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            tm0 = fmaxf(tm0, __shfl_xor_sync(0xFFFFFFFFu, tm0, off));
            tm1 = fmaxf(tm1, __shfl_xor_sync(0xFFFFFFFFu, tm1, off));
          }
          const float mn0 = fmaxf(m_run[0], tm0), mn1 = fmaxf(m_run[1], tm1);
          const float bs0 = mn0 == -INFINITY ? 0.f : mn0;
          const float bs1 = mn1 == -INFINITY ? 0.f : mn1;
          const float al0 = ex2(m_run[0] - bs0), al1 = ex2(m_run[1] - bs1);
          const float p00 = ex2(z00 - bs0), p10 = ex2(z10 - bs0);
          const float p01 = ex2(z01 - bs1), p11 = ex2(z11 - bs1);
          l_run[0] = fmaf(l_run[0], al0, p00 + p10);
          l_run[1] = fmaf(l_run[1], al1, p01 + p11);
          m_run[0] = mn0;
          m_run[1] = mn1;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            acc[mt][0] *= al0; acc[mt][2] *= al0;
            acc[mt][1] *= al1; acc[mt][3] *= al1;
          }
          // P^T as the B operand (k = token, n = head) via 8x8 transposes
          uint32_t x0h, x0l, x1h, x1l;
          split_pack(p00, p01, x0h, x0l, T());
          split_pack(p10, p11, x1h, x1l, T());
          const uint32_t bh0 = movm_t(x0h), bh1 = movm_t(x1h);
          const uint32_t bl0 = movm_t(x0l), bl1 = movm_t(x1l);
          {
            const int mi = lane >> 3;
            const int tok = sub * 16 + (lane & 7) + (mi >> 1) * 8;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              const int ch = 2 * mt + (mi & 1);
              uint32_t af[4];
              ldsm_x4_t(vb + (ch >> 3) * slab_bytes + swz(tok, ch & 7), af);
              mma16816(acc[mt], af, bh0, bh1, T());
              mma16816(acc[mt], af, bl0, bl1, T());
            }
          }
        }
        if (nv > 0 && nv < TT) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      } else {
        // ---- CUDA-core consumer ----
        const int tt = lane / SL, hh = lane % SL;
        float *pb = pbuf + cw * GC * TP;  // cw < kMaxConsumerWarps
        // this lane's 4 output channels 4*lane .. 4*lane+3 inside a V row
        const int vslab = (4 * lane * SL) / 128;
        const int vbyte = (4 * lane * SL) % 128;
        const uint8_t *kst = st;
        const uint8_t *vst = st + kv_off + vslab * slab_bytes;
#pragma unroll 1
        for (int pass = 0; pass * TP < nv; ++pass) {
          const int t = pass * TP + tt;
          float dot[GC];
#pragma unroll
          for (int g = 0; g < GC; ++g) dot[g] = 0.f;
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const int lc = (c8 + hh * (8 / SL)) & 7;
            const uint4 kw = *reinterpret_cast<const uint4 *>(kst + hh * slab_bytes + swz(t, lc));
            float kf[EPC];
            if constexpr (SL == 2) {
              const float2 f0 = unpack2(kw.x, T()), f1 = unpack2(kw.y, T());
              const float2 f2 = unpack2(kw.z, T()), f3 = unpack2(kw.w, T());
              kf[0] = f0.x; kf[1] = f0.y; kf[2] = f1.x; kf[3] = f1.y;
              kf[4] = f2.x; kf[5] = f2.y; kf[6] = f3.x; kf[7] = f3.y;
            } else {
              kf[0] = __uint_as_float(kw.x); kf[1] = __uint_as_float(kw.y);
              kf[2] = __uint_as_float(kw.z); kf[3] = __uint_as_float(kw.w);
            }
#pragma unroll
            for (int g = 0; g < GC; ++g) {
              const float4 *qp =
                  reinterpret_cast<const float4 *>(q_s + (g * SL + hh) * QSTR + lc * EPC);
#pragma unroll
              for (int e4 = 0; e4 < EPC / 4; ++e4) {
                const float4 qv = qp[e4];
                dot[g] = fmaf(qv.x, kf[4 * e4 + 0], dot[g]);
                dot[g] = fmaf(qv.y, kf[4 * e4 + 1], dot[g]);
                dot[g] = fmaf(qv.z, kf[4 * e4 + 2], dot[g]);
                dot[g] = fmaf(qv.w, kf[4 * e4 + 3], dot[g]);
              }
            }
          }
          const bool valid = t < nv;
#pragma unroll
          for (int g = 0; g < GC; ++g) {
#pragma unroll
            for (int off = 1; off < SL; off <<= 1)
              dot[g] += __shfl_xor_sync(0xFFFFFFFFu, dot[g], off);
            const float z = (valid && ((msk >> g) & 1u)) ? dot[g] * sl : -INFINITY;
            float tm = z;
#pragma unroll
            for (int off = SL; off < 32; off <<= 1)
              tm = fmaxf(tm, __shfl_xor_sync(0xFFFFFFFFu, tm, off));
            const float mn = fmaxf(m_run[g], tm);
            const float bs = mn == -INFINITY ? 0.f : mn;
            const float al = ex2(m_run[g] - bs);
            const float pz = ex2(z - bs);
            l_run[g] = fmaf(l_run[g], al, hh == 0 ? pz : 0.f);
            acc[g][0] *= al; acc[g][1] *= al; acc[g][2] *= al; acc[g][3] *= al;
            m_run[g] = mn;
            if (hh == 0) pb[g * TP + tt] = pz;
          }
          __syncwarp();
          const int ntok = min(TP, nv - pass * TP);
#pragma unroll 4
          for (int tk2 = 0; tk2 < ntok; ++tk2) {
            const int row = pass * TP + tk2;
            float vv[4];
            if constexpr (SL == 2) {
              const int chk = vbyte >> 4;
              const uint2 w = *reinterpret_cast<const uint2 *>(vst + swz(row, chk) + (vbyte & 15));
              const float2 f0 = unpack2(w.x, T()), f1 = unpack2(w.y, T());
              vv[0] = f0.x; vv[1] = f0.y; vv[2] = f1.x; vv[3] = f1.y;
            } else {
              const float4 w = *reinterpret_cast<const float4 *>(vst + swz(row, vbyte >> 4));
              vv[0] = w.x; vv[1] = w.y; vv[2] = w.z; vv[3] = w.w;
            }
#pragma unroll
            for (int g = 0; g < GC; ++g) {
              const float pz = pb[g * TP + tk2];
              acc[g][0] = fmaf(pz, vv[0], acc[g][0]);
              acc[g][1] = fmaf(pz, vv[1], acc[g][1]);
              acc[g][2] = fmaf(pz, vv[2], acc[g][2]);
              acc[g][3] = fmaf(pz, vv[3], acc[g][3]);
            }
          }
          __syncwarp();
        }
      }
      if constexpr (WIN) {
        if (ent.src >= 0 && nv > 0) {
          // a fetched tile: its valid rows go to the page's window slot
          char *kw = static_cast<char *>(const_cast<void *>(a.k));
          char *vw = static_cast<char *>(const_cast<void *>(a.v));
          const size_t dst0 =
              ((size_t)(((long long)ent.phys * a.Hkv + kvh) * ps) + (size_t)(j % UPP) * TT) *
              (SL * 128);
          for (int i = lane; i < nv * SL * 8; i += 32) {
            const int row = i / (SL * 8), rem = i % (SL * 8);
            const uint8_t *src = st + (rem >> 3) * slab_bytes + swz(row, rem & 7);
            const size_t off = dst0 + (size_t)row * (SL * 128) + rem * 16;
            *reinterpret_cast<uint4 *>(kw + off) = *reinterpret_cast<const uint4 *>(src);
            *reinterpret_cast<uint4 *>(vw + off) = *reinterpret_cast<const uint4 *>(src + kv_off);
          }
          // the stage may next be filled by TMA: order this warp's view of
          // the cp.async data before those async-proxy writes
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    // a warp with no tile of segment B still hands in its segment A
    if (segB != INT_MAX && !in_b) finish_a();
  }

  // ======================= merge the consumer warps =======================
  __syncthreads();  // every stage is consumed (or abandoned): reuse the ring
  pdl_trigger();
  float *mw = reinterpret_cast<float *>(stages);  // [warps][GC] (at most 64)
  float *lw = mw + 64;                            // [warps][GC]
  float *ow = mw + 128;                           // [warps][GC][128], 16-byte aligned
  if (warp > 0) {
    if constexpr (MMA) {
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1)
          l_run[i] += __shfl_xor_sync(0xFFFFFFFFu, l_run[i], off);
      const int h0 = 2 * tig, h1 = h0 + 1;
      if (gid == 0) {
        if (h0 < GC) { mw[cw * GC + h0] = m_run[0]; lw[cw * GC + h0] = l_run[0]; }
        if (h1 < GC) { mw[cw * GC + h1] = m_run[1]; lw[cw * GC + h1] = l_run[1]; }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int d0 = 16 * mt + gid, d1 = d0 + 8;
        if (h0 < GC) {
          ow[(cw * GC + h0) * kHeadDim + d0] = acc[mt][0];
          ow[(cw * GC + h0) * kHeadDim + d1] = acc[mt][2];
        }
        if (h1 < GC) {
          ow[(cw * GC + h1) * kHeadDim + d0] = acc[mt][1];
          ow[(cw * GC + h1) * kHeadDim + d1] = acc[mt][3];
        }
      }
    } else {
#pragma unroll
      for (int g = 0; g < GC; ++g) {
        float l = l_run[g];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, off);
        if (lane == 0) { mw[cw * GC + g] = m_run[g]; lw[cw * GC + g] = l; }
        float4 o4 = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
        *reinterpret_cast<float4 *>(ow + (cw * GC + g) * kHeadDim + 4 * lane) = o4;
      }
    }
  }
  __syncthreads();
  // a thread per 4 consecutive channels of one head: 16-byte loads of the
  // warps' partials and one 16-byte store (the stores of a CTA's last
  // partials queue behind the other CTAs' loads at the end of the call)
  const long long rows = (long long)a.B * a.Hq;
  for (int i = threadIdx.x; i < GC * (kHeadDim / 4); i += blockDim.x) {
    const int g = i / (kHeadDim / 4), d4 = i % (kHeadDim / 4);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < a.nw; ++w) M = fmaxf(M, mw[w * GC + g]);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < a.nw; ++w) {
        const float m = mw[w * GC + g];
        const float f = m == -INFINITY ? 0.f : ex2(m - M);
        const float4 x = *reinterpret_cast<const float4 *>(ow + (w * GC + g) * kHeadDim + 4 * d4);
        o.x = fmaf(f, x.x, o.x);
        o.y = fmaf(f, x.y, o.y);
        o.z = fmaf(f, x.z, o.z);
        o.w = fmaf(f, x.w, o.w);
        l = fmaf(f, lw[w * GC + g], l);
      }
    }
    const long long r = (long long)b * a.Hq + head0 + g;
    if (a.num_splits == 1) {
      float4 y;
      y.x = l > 0.f ? o.x / l : 0.f;
      y.y = l > 0.f ? o.y / l : 0.f;
      y.z = l > 0.f ? o.z / l : 0.f;
      y.w = l > 0.f ? o.w / l : 0.f;
      *reinterpret_cast<float4 *>(a.out + r * kHeadDim + 4 * d4) = y;
    } else {
      *reinterpret_cast<float4 *>(a.part_o + ((long long)split * rows + r) * kHeadDim + 4 * d4) =
          o;
      if (d4 == 0) {
        a.part_ml[((long long)split * rows + r) * 2] = M;
        a.part_ml[((long long)split * rows + r) * 2 + 1] = l;
      }
    }
  }
}

template <class T, int GC, bool MMA, bool WIN = false>
cudaError_t launch_attn_t(const AttnArgs &a, const CUtensorMap *tk, const CUtensorMap *tv,
                          dim3 grid, size_t smem, cudaStream_t st) {
  auto kern = attn_kernel<T, GC, MMA, WIN>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  return launch_pdl(kern, grid, dim3(32 * (1 + a.nw)), smem, st, a, *tk, *tv);
}

template <class T, int GC, bool MMA, bool WIN = false>
int attn_occupancy_t(int threads, size_t smem) {
  auto kern = attn_kernel<T, GC, MMA, WIN>;
  int dev = 0;
  cudaGetDevice(&dev);
  static int attr_done[64] = {0};
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    attr_done[dev] = 1;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace kvs
