// kv_select_fused.cu -- page score, top-K selection and the GQA group's union
// of selected pages in one launch: a thread-block cluster per (sequence, kv
// head), one CTA per query head of the group.
//
// What it computes (KVDrive: A Holistic Multi-Tier KV Cache Management System
// for Long-Context LLM Inference, section 2.2 and section 2.3 steps (1)-(2)):
// for every query head h of the group, the page score
//   s[p] = sum_c max(q_c mn_c, q_c mx_c)
// of each page p against its channel-wise key minimum and maximum (an upper
// bound on q.k over the page), then the K pages with the largest score (ties
// to the lower page, ascending), then, for the attention that follows, the
// union of the group's selections with a head mask per page.  The results are
// those of kv_page_score + kv_topk_select + the union the sparse attention
// builds: the scores come from the same tensor-core contraction (bit for bit),
// the selection from the same radix select.
//
// Design on GB300:
//  * Cluster of G CTAs (G = 4 or 8 query heads per kv head).  CTA c scores a
//    contiguous 1/G of the pages for all G heads (its share of the index is
//    read once, not G times) and stores each head's key into the shared
//    memory of the CTA that owns that head (distributed shared memory), so no
//    score reaches global memory.
//  * After a cluster barrier every CTA runs the radix select of its own head
//    over keys already on chip, writes its selection, and ORs its head's bit
//    into the page map (a byte of head bits per page) of the CTA that owns
//    the page's 1/G of the pages (red.shared::cluster, no reply awaited).
//  * After a second barrier each CTA holds the complete map of its pages:
//    it counts their union pages, the CTAs' counts are exchanged through
//    distributed shared memory, and after a third barrier each writes its
//    part of the list in page order.  An entry holds the physical page (from
//    the block-table entries CTA c loaded for its scoring) and the page's
//    valid tokens | head mask << 8, so the attention needs no block-table
//    lookup.  (Reading the other CTAs' bitmaps remotely instead cost a round
//    trip; OR-ing into every CTA's map, to skip the count exchange, cost G
//    remote atomics per selected page: 13.7 -> 19.9 us on 8-head groups.)
#include <algorithm>

#include "kv_internal.cuh"
#include "kv_launch.h"
#include "kv_radix.cuh"

namespace kvs {
namespace {

__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void red_or_cluster(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.or.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mma_bound(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, __nv_bfloat16) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bound(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, __half) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// the halves of a packed 16-bit pair whose sign is set (neg) or clear
__device__ __forceinline__ uint32_t sign_half(uint32_t w, bool neg) {
  const uint32_t s = (w >> 15) & 0x00010001u;
  const uint32_t m = (neg ? s : (s ^ 0x00010001u)) * 0xFFFFu;
  return w & m;
}

// Shared memory after the radix state: keys[maxP4] | map[PC bytes: head
// bits of this CTA's pages] | bt_s[PC] | cnt[16]
struct SelLayout {
  int off_map, off_bt, off_cnt, bytes;
};
__host__ __device__ inline SelLayout sel_layout(int maxP, int PC) {
  SelLayout l;
  const int maxP4 = (maxP + 3) & ~3;
  l.off_map = maxP4 * 4;
  l.off_bt = l.off_map + PC;  // PC is a multiple of 32
  l.off_cnt = l.off_bt + PC * 4;
  l.bytes = l.off_cnt + 16 * 4;
  return l;
}

// SCORE: the cluster scores the pages itself (keys stored remotely into each
// head's CTA); otherwise each CTA reads its row of scores (a.scores, written
// by the page-score kernel just before) into its keys.
template <class T, int G, int THREADS, bool SCORE>
__global__ void __launch_bounds__(THREADS, THREADS <= 128 ? 4 : 1)
    select_fused_kernel(const SelectArgs a) {
  constexpr int WARPS = THREADS / 32;
  extern __shared__ __align__(16) uint8_t sel_smem[];
  __shared__ RadixSmem<THREADS> rs;
  const SelLayout L = sel_layout(a.maxP, a.PC);
  uint32_t *keys = reinterpret_cast<uint32_t *>(sel_smem);
  uint32_t *map = reinterpret_cast<uint32_t *>(sel_smem + L.off_map);  // 4 pages a word
  int32_t *bt_s = reinterpret_cast<int32_t *>(sel_smem + L.off_bt);
  uint32_t *cnt = reinterpret_cast<uint32_t *>(sel_smem + L.off_cnt);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int c = blockIdx.x;  // rank in the cluster == head within the group
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int head0 = kvh * G;
  const int maxP = a.maxP, PC = a.PC, ps = a.ps;
  const int lo = c * PC;  // this CTA's pages for the score and the union
  const long long row = (long long)b * a.Hq + head0 + c;
  int32_t *orow = a.indices + row * a.K;
  const long long gbase = (long long)b * a.Hkv + kvh;

  // every CTA of the cluster must have started before its shared memory is
  // written remotely: arrive now, wait just before the first remote store
  if constexpr (SCORE) cluster_arrive_relaxed();
  if (!a.early_inputs) pdl_wait();
  // the group's [q- | q+] coefficients, as the page-score kernel takes them:
  // lane (gid, tig) holds chunks tig + 4 i of head gid's row
  uint4 cf[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    cf[i] = make_uint4(0u, 0u, 0u, 0u);
    if (SCORE && gid < G) {
      const int ch = tig + 4 * i;
      const uint4 w = reinterpret_cast<const uint4 *>(
          static_cast<const T *>(a.q) + ((long long)b * a.Hq + head0 + gid) * kHeadDim)[ch & 15];
      const bool neg = ch < 16;
      cf[i] = make_uint4(sign_half(w.x, neg), sign_half(w.y, neg), sign_half(w.z, neg),
                         sign_half(w.w, neg));
    }
  }
  for (int i = tid; i < PC; i += THREADS)
    bt_s[i] = lo + i < maxP ? a.block_table[(long long)b * maxP + lo + i] : -1;
  if (a.early_inputs) pdl_wait();
  const int len = a.context_lens[b];
  const bool bad_len = len < 1 || len > maxP * ps;
  const int P = bad_len ? 0 : (len + ps - 1) / ps;
  if (bad_len && c == 0 && tid == 0) flag_error(a.status, KV_ERR_BOUNDS);
  const int nmw = PC / 4;  // words of this CTA's page map
  for (int i = tid; i < nmw; i += THREADS) map[i] = 0u;
  for (int i = tid; i < 256; i += THREADS) rs.hist[0][i] = 0;
  __syncthreads();
  // (without the scoring below, this barrier alone orders every CTA's zeroed
  // map before the other CTAs' ORs into it)
  if constexpr (!SCORE) cluster_arrive();

  // ---- scores of this CTA's pages for every head of the group -------------
  if constexpr (!SCORE) {
    // this CTA's own row of scores
    const float *srow = a.scores + row * maxP;
    for (int p = tid; p < P; p += THREADS) keys[p] = score_key(srow[p]);
    __syncthreads();
  } else {
  cluster_wait();
  const T *tab = static_cast<const T *>(a.table);
  const uint32_t keys_addr = smem_u32(keys);
  for (int t = warp; t * 16 < PC; t += WARPS) {
    const int p0 = lo + 16 * t;
    if (p0 >= maxP) break;
    const int pa = p0 + gid, pb = pa + 8;
    long long ph_a = -1, ph_b = -1;
    if (pa < P) {
      const long long x = bt_s[pa - lo];
      if (x >= 0 && x < a.nphys) ph_a = x;
      else flag_error(a.status, KV_ERR_BOUNDS);
    }
    if (pb < P) {
      const long long x = bt_s[pb - lo];
      if (x >= 0 && x < a.nphys) ph_b = x;
      else flag_error(a.status, KV_ERR_BOUNDS);
    }
    const uint4 *rowa = reinterpret_cast<const uint4 *>(
        tab + ((ph_a < 0 ? 0 : ph_a) * a.Hkv + kvh) * (2 * kHeadDim));
    const uint4 *rowb = reinterpret_cast<const uint4 *>(
        tab + ((ph_b < 0 ? 0 : ph_b) * a.Hkv + kvh) * (2 * kHeadDim));
    uint4 ra[8], rb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ra[i] = ph_a >= 0 ? rowa[tig + 4 * i] : make_uint4(0u, 0u, 0u, 0u);
      rb[i] = ph_b >= 0 ? rowb[tig + 4 * i] : make_uint4(0u, 0u, 0u, 0u);
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t a0[4] = {ra[i].x, rb[i].x, ra[i].y, rb[i].y};
      mma_bound(acc, a0, cf[i].x, cf[i].y, T());
      const uint32_t a1[4] = {ra[i].z, rb[i].z, ra[i].w, rb[i].w};
      mma_bound(acc, a1, cf[i].z, cf[i].w, T());
    }
    // acc[0..1]: page pa, heads 2 tig and 2 tig + 1; acc[2..3]: page pb
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int h = 2 * tig + (e & 1);
      const int p = e < 2 ? pa : pb;
      const bool ok = e < 2 ? ph_a >= 0 : ph_b >= 0;
      if (h < G && p < maxP)
        st_cluster(map_rank(keys_addr + 4u * p, h), score_key(ok ? acc[e] : -INFINITY));
    }
  }
  cluster_arrive();
  cluster_wait();
  }

  // ---- top-K of this CTA's head over the keys on chip ---------------------
  const uint32_t map_addr = smem_u32(map);
  const uint32_t my_bit = 1u << c;
  const int keff = min(a.K, P);
  if (keff == P) {  // every page: the map is every head's on every valid page
    if constexpr (!SCORE) cluster_wait();
    for (int i = tid; i < a.K; i += THREADS) orow[i] = i < P ? i : -1;
    const uint32_t all = (1u << G) - 1u;
    for (int i = tid; i < nmw; i += THREADS) {
      const int n = min(4, P - (lo + 4 * i));
      map[i] = n <= 0 ? 0u : (all * 0x01010101u) & (n == 4 ? 0xFFFFFFFFu : (1u << (8 * n)) - 1u);
    }
  } else {
    const int f_sink = a.sink_tokens > 0 ? min(P, (a.sink_tokens + ps - 1) / ps) : 0;
    const int f_local = a.local_tokens > 0 ? max(0, len - a.local_tokens) / ps : P;
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    for (int p = tid; p < P; p += THREADS) {
      uint32_t k = keys[p];
      if (p < f_sink || p >= f_local) keys[p] = k = kForcedKey;
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
    block_minmax<THREADS>(rs, kmin, kmax);
    uint32_t prefix, pmask;
    int krem;
    auto key_at = [&](int p) -> uint32_t { return keys[p]; };
    radix_threshold<THREADS>(rs, key_at, P, keff, kmin, kmax, prefix, pmask, krem);
    if constexpr (!SCORE) cluster_wait();
    radix_emit<THREADS>(rs, key_at, keys, P, prefix, pmask, krem, [&](int pos, int p) {
      if (pos < a.K) orow[pos] = p;
      const int owner = p / PC;  // the CTA whose pages p is in
      red_or_cluster(map_rank(map_addr + ((uint32_t)(p - owner * PC) & ~3u), owner),
                     my_bit << (8 * (p & 3)));
    });
    for (int i = keff + tid; i < a.K; i += THREADS) orow[i] = -1;
  }
  cluster_arrive();
  cluster_wait();

  // ---- the group's union over this CTA's pages ------------------------------
  // Each thread counts the union pages of a run of consecutive map words; a
  // block scan places the runs; the CTAs' totals are exchanged; the list is
  // written in page order at the CTA's offset.
  const int per = (nmw + THREADS - 1) / THREADS;  // map words per thread
  const int w0 = min(nmw, tid * per), w1 = min(nmw, w0 + per);
  auto page_bits = [&](int w) -> uint32_t {  // a valid page's head bits, 4 a word
    uint32_t m = map[w];
    const int n = P - (lo + 4 * w);
    if (n < 4) m &= n <= 0 ? 0u : (1u << (8 * n)) - 1u;
    return m;
  };
  uint32_t n = 0;
  for (int w = w0; w < w1; ++w) {
    uint32_t t = page_bits(w);
    t |= t >> 4;
    t |= t >> 2;
    t |= t >> 1;
    n += __popc(t & 0x01010101u);
  }
  uint32_t ni = n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, ni, off);
    if (lane >= off) ni += x;
  }
  if (lane == 31) rs.wmin[warp] = ni;
  __syncthreads();
  const uint32_t ws = lane < WARPS ? rs.wmin[lane] : 0u;
  uint32_t pos = __reduce_add_sync(0xFFFFFFFFu, lane < warp ? ws : 0u) + ni - n;
  const uint32_t mine = __reduce_add_sync(0xFFFFFFFFu, ws);  // this CTA's union pages
  if (tid < G) st_cluster(map_rank(smem_u32(&cnt[c]), tid), mine);
  cluster_arrive();
  cluster_wait();
  // no remote shared-memory access past this point
  uint32_t base = 0, total = 0;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    base += g < c ? cnt[g] : 0u;
    total += cnt[g];
  }
  pdl_trigger();
  pos += base;
  for (int w = w0; w < w1; ++w) {
    const uint32_t m4 = page_bits(w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t m = (m4 >> (8 * e)) & 0xFFu;
      if (m == 0u) continue;
      if (pos < (uint32_t)a.umax) {
        const int i = 4 * w + e;  // page lo + i
        const long long x = bt_s[i];
        const bool okp = x >= 0 && x < a.nphys;
        a.upages[gbase * a.umax + pos] = okp ? (int32_t)x : -1;
        a.umasks[gbase * a.umax + pos] = (uint32_t)min(ps, len - (lo + i) * ps) | (m << 8);
      }
      ++pos;
    }
  }
  if (c == 0 && tid == 0) a.ucount[gbase] = (int32_t)min(total, (uint32_t)a.umax);
}

template <class T, int G, int THREADS, bool SCORE>
cudaError_t launch_sel_t(const SelectArgs &a, int B, size_t smem, cudaStream_t st) {
  auto kern = select_fused_kernel<T, G, THREADS, SCORE>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G, a.Hkv, B);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = KVS_PDL ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <class T, int G>
cudaError_t launch_sel_g(const SelectArgs &a, int B, int threads, size_t smem, cudaStream_t st) {
  if (a.scores != nullptr) {  // selection and union over the score kernel's rows
    switch (threads) {
      case 256: return launch_sel_t<T, G, 256, false>(a, B, smem, st);
      default: return launch_sel_t<T, G, 1024, false>(a, B, smem, st);
    }
  }
  switch (threads) {
    case 128: return launch_sel_t<T, G, 128, true>(a, B, smem, st);
    case 256: return launch_sel_t<T, G, 256, true>(a, B, smem, st);
    default: return launch_sel_t<T, G, 512, true>(a, B, smem, st);
  }
}

}  // namespace

int select_fused_pages_per_cta(int G, int maxP) {
  const int per = (maxP + G - 1) / G;
  return (per + 31) / 32 * 32;
}

int select_fused_threads(int PC) {
  // two 16-page tiles per warp, 4 to 16 warps
  const int warps = std::min(16, std::max(4, PC / 32));
  return warps <= 4 ? 128 : warps <= 8 ? 256 : 512;
}

size_t select_fused_smem(int G, int maxP) {
  return (size_t)sel_layout(maxP, select_fused_pages_per_cta(G, maxP)).bytes;
}

cudaError_t launch_select_fused(int dtype, const SelectArgs &a, int B, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  // the select over scores in memory: as the top-K kernel, wide CTAs for
  // long rows
  const int threads =
      a.scores != nullptr ? (a.maxP >= 4096 ? 1024 : 256) : select_fused_threads(a.PC);
  const size_t smem = select_fused_smem(G, a.maxP);
  if (dtype == KV_F16)
    return G == 8 ? launch_sel_g<__half, 8>(a, B, threads, smem, st)
                  : launch_sel_g<__half, 4>(a, B, threads, smem, st);
  return G == 8 ? launch_sel_g<__nv_bfloat16, 8>(a, B, threads, smem, st)
                : launch_sel_g<__nv_bfloat16, 4>(a, B, threads, smem, st);
}

}  // namespace kvs
