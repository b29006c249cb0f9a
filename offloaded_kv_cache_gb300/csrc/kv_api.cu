// kv_api.cu -- the extern "C" boundary: argument checks, launch planning and
// launches for the paged decode-attention path.  Declarations and contracts
// are in include/kvsparse.h.
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kv_internal.cuh"
#include "kv_launch.h"

namespace {

using namespace kvs;

// device status word (one per device, zero-initialised at module load)
__device__ int g_kv_status;

constexpr int kMaxDevices = 64;
std::atomic<int *> g_status_ptr[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];

// testing hooks (kv_debug_config, kv_debug_split_mode)
std::atomic<int> g_debug_skip_page{-1};
std::atomic<int> g_split_mode{-1};
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

int *status_ptr(int dev) {
  int *p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void *addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_kv_status) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  g_status_ptr[dev].store(static_cast<int *>(addr), std::memory_order_release);
  return static_cast<int *>(addr);
}

int sm_count(int dev) {
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 152;
  }
  g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool al16(const void *p) { return p && ((uintptr_t)p & 15u) == 0; }
bool al4(const void *p) { return p && ((uintptr_t)p & 3u) == 0; }
int elem_bytes(int dtype) { return dtype == KV_F32 ? 4 : 2; }

int check_shape(const kv_shape *s) {
  if (!s) return KV_ERR_INVALID_ARG;
  if (s->batch < 1 || s->num_q_heads < 1 || s->num_kv_heads < 1 ||
      s->num_q_heads % s->num_kv_heads != 0 || s->max_pages_per_seq < 1 ||
      s->num_phys_pages < 1)
    return KV_ERR_INVALID_ARG;
  if (s->kv_loc != KV_LOC_HBM && s->kv_loc != KV_LOC_HOST_PINNED) return KV_ERR_INVALID_ARG;
  if (s->dtype != KV_F32 && s->dtype != KV_F16 && s->dtype != KV_BF16) return KV_ERR_UNSUPPORTED;
  if (s->head_dim != kHeadDim) return KV_ERR_UNSUPPORTED;
  // pages are whole 16-token tiles; the attention keeps a page's valid-token
  // count in 8 bits
  if (s->page_size != 16 && s->page_size != 32 && s->page_size != 64 && s->page_size != 128)
    return KV_ERR_UNSUPPORTED;
  // index arithmetic limits: tokens per row and K/V rows fit in int32
  if ((long long)s->max_pages_per_seq * s->page_size > INT_MAX) return KV_ERR_UNSUPPORTED;
  if (s->num_phys_pages * (long long)s->num_kv_heads * s->page_size > INT_MAX)
    return KV_ERR_UNSUPPORTED;
  if ((long long)s->batch * s->num_q_heads > INT_MAX) return KV_ERR_UNSUPPORTED;
  return KV_OK;
}

// Device-visible address of a K or V cache, checked against kv_loc.
int resolve_kv(const kv_shape *s, const void *p, const void **dev_ptr) {
  if (!al16(p)) return KV_ERR_INVALID_ARG;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  if (s->kv_loc == KV_LOC_HBM) {
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
      return KV_ERR_LOCATION;
    *dev_ptr = p;
  } else {
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return KV_ERR_LOCATION;
    *dev_ptr = at.devicePointer;
  }
  return KV_OK;
}

// ---------------------------------------------------------------------------
// attention launch plan: head chunking, split count, pipeline depth, workspace
// ---------------------------------------------------------------------------
struct Plan {
  int gc = 1, nchunk = 1, groups = 1;
  bool mma = false;
  bool win = false;  // the page-window instantiation (16-byte page-list entries)
  int S = 1, umax = 0, nstages = 4, nw = 4, header = 8192;
  size_t smem = 0;
  size_t off_part_o = 0, off_part_ml = 0, off_upages = 0, off_umasks = 0, off_ucount = 0;
  // the attention over kv_select_pages' lists may cut all groups' lists into
  // equal chunks (AttnArgs::spread) when the shapes allow it (spread_ok; its
  // workspace is then reserved)
  bool spread_ok = false;
  size_t off_spa_o = 0, off_spa_ml = 0, off_gmeta = 0;
  size_t total = 0;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// CTA shapes the planner chooses between (consumer warps, stages):
//  * wide: small CTAs, many resident per SM, for many short (b, head) units
//    that fit one wave without splitting;
//  * deep: four consumer warps double-buffered over an 8-stage ring (4 for
//    fp32), split along the context when there are few long units.
#ifndef KVS_WIDE_NW
#define KVS_WIDE_NW 3
#endif
#ifndef KVS_WIDE_NS
#define KVS_WIDE_NS 3
#endif
#ifndef KVS_DEEP_NW
#define KVS_DEEP_NW 4
#endif
#ifndef KVS_DEEP_RING_BYTES
#define KVS_DEEP_RING_BYTES (64 * 1024)
#endif
#ifndef KVS_SPLIT_OVERHEAD_TILES
#define KVS_SPLIT_OVERHEAD_TILES 4  // fixed cost of a CTA, in tiles, for the split choice
#endif
// The attention over kv_select_pages' lists takes equal chunks of all groups'
// lists when the longest CTA of the per-group split would stream more K/V
// than an equal chunk for longer than this: the prefix sums' round trip
// before the first load and the combine's lookup of where the partials are
// (measured together at about 2.5 us on GB300)
#ifndef KVS_SPREAD_FIXED_NS
#define KVS_SPREAD_FIXED_NS 2500
#endif
// Making that choice at all costs the kernels about 1.5 us (the groups'
// lengths and a block reduction before the first load, the combine's lookup;
// Llama-3.1-8B 32k call 36.4 -> 37.8 us when the split per group is kept), so
// the plan only lets the kernel choose when a CTA's share of a group's list
// can take this long to stream with all CTAs sharing the link (70B-class
// layer: about 300 us; Llama-3.1-8B 32k: about 38 us)
#ifndef KVS_SPREAD_MIN_CTA_NS
#define KVS_SPREAD_MIN_CTA_NS 100000
#endif
constexpr int kSpreadMaxGroups = 4096;

int header_bytes(const Plan &pl, int elem, long long list_pages) {
  const long long b = attn_fixed_header(elem, pl.gc, pl.mma) +
                      (long long)attn_entry_bytes(pl.win) *
                          std::min<long long>(list_pages, kMaxListPages);
  return (int)((b + 1023) / 1024 * 1024);
}

// occupancy answers, cached per (device, kernel, threads, shared memory):
// the calculator costs microseconds of host time per query
struct OccEntry {
  int dev, dtype, gc, mma, win, threads;
  size_t smem;
  int n;
};
std::mutex g_occ_mutex;
OccEntry g_occ[64];
int g_occ_n = 0;     // entries in use (at most 64)
int g_occ_next = 0;  // the slot the next answer goes to (a ring over the 64)

int cached_occupancy(int dtype, int gc, bool mma, bool win, int threads, size_t smem) {
  const int dev = current_device();
  {
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    for (int i = 0; i < g_occ_n; ++i) {
      const OccEntry &e = g_occ[i];
      if (e.dev == dev && e.dtype == dtype && e.gc == gc && e.mma == (int)mma &&
          e.win == (int)win && e.threads == threads && e.smem == smem)
        return e.n;
    }
  }
  const int n = win   ? attn_occupancy_win(dtype, gc, mma, threads, smem)
                : mma ? attn_occupancy_mma(dtype, gc, threads, smem)
                      : attn_occupancy_core(dtype, gc, threads, smem);
  if (n > 0) {
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    g_occ[g_occ_next] = OccEntry{dev, dtype, gc, (int)mma, (int)win, threads, smem, n};
    g_occ_next = (g_occ_next + 1) % 64;
    if (g_occ_n < 64) ++g_occ_n;
  }
  return n;
}

// resident CTAs per SM: the occupancy calculator on the real kernel when a
// device is present, else an estimate from shared memory and threads
int resident_ctas(const Plan &pl, int dtype, bool have_device) {
  const int threads = 32 * (1 + pl.nw);
  int n = 0;
  if (have_device) n = cached_occupancy(dtype, pl.gc, pl.mma, pl.win, threads, pl.smem);
  if (n <= 0) {
    n = (int)((228 * 1024) / (pl.smem + 1024));
    n = std::min(n, 2048 / threads);
  }
  return std::max(n, 1);
}

Plan make_plan(const kv_shape *s, int k, int sms, bool have_device, bool win) {
  Plan pl;
  pl.win = win;
  const int G = s->num_q_heads / s->num_kv_heads;
  if (s->dtype == KV_F32) {
    pl.gc = (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
  } else if (G % 8 == 0) {
    pl.gc = 8;
    pl.mma = true;
  } else if (G % 4 == 0) {
    pl.gc = 4;
    pl.mma = true;
  } else {
    pl.gc = (G % 2 == 0) ? 2 : 1;
  }
  pl.nchunk = G / pl.gc;
  pl.groups = s->num_kv_heads * pl.nchunk;
  const int stage = 2 * kTileTokens * kHeadDim * elem_bytes(s->dtype);  // one K+V tile
  const long long maxP = s->max_pages_per_seq;
  const long long work = k > 0 ? std::min<long long>((long long)pl.gc * k, maxP) : maxP;
  const long long units = (long long)s->batch * pl.groups;
  const long long upp = s->page_size / kTileTokens;

  // wide: one CTA per unit, all resident at once
  Plan wide = pl;
  wide.nw = KVS_WIDE_NW;
  wide.nstages = KVS_WIDE_NS;
  wide.S = 1;
  wide.header = header_bytes(wide, elem_bytes(s->dtype), work);
  wide.smem = 1024 + wide.header + (size_t)wide.nstages * stage;
  // wide when the units alone keep enough K/V bytes in flight on every SM
  // (about 96 KB) without splitting them
#ifndef KVS_WIDE_INFLIGHT
#define KVS_WIDE_INFLIGHT (96 * 1024)
#endif
  (void)have_device;
  const bool use_wide = work <= kMaxListPages &&
                        units * wide.nstages * stage >= (long long)sms * KVS_WIDE_INFLIGHT;

  if (use_wide) {
    pl = wide;
  } else {
    pl.nw = KVS_DEEP_NW;
    int ns = (KVS_DEEP_RING_BYTES / stage) / pl.nw * pl.nw;
    ns = std::max(ns, 2 * pl.nw);
    ns = std::min(ns, kMaxStages / pl.nw * pl.nw);
    pl.nstages = ns;
    pl.header = header_bytes(pl, elem_bytes(s->dtype), kMaxListPages);
    pl.smem = 1024 + pl.header + (size_t)ns * stage;
    const long long slots = (long long)sms * resident_ctas(pl, s->dtype, have_device);
    // split count minimising (waves x tiles per CTA) plus a fixed cost per
    // CTA; a split keeps at least one page and at most kMaxListPages
    const int smin = (int)std::max<long long>(1, (work + kMaxListPages - 1) / kMaxListPages);
    const int smax = (int)std::min<long long>(1024, std::max<long long>(smin, work * upp / 4));
    long long best = LLONG_MAX;
    int bestS = smin;
    for (int S = smin; S <= smax && S <= work; ++S) {
      const long long waves = (units * S + slots - 1) / slots;
      const long long cost = waves * (((work + S - 1) / S) * upp + KVS_SPLIT_OVERHEAD_TILES);
      if (cost < best) {
        best = cost;
        bestS = S;
      }
    }
#ifdef KVS_FORCE_SPLITS
    bestS = (int)std::min<long long>(std::max(KVS_FORCE_SPLITS, smin), std::max<long long>(work, 1));
#endif
    pl.S = bestS;
    // a smaller page list leaves more shared memory
    pl.header = header_bytes(pl, elem_bytes(s->dtype), (work + pl.S - 1) / pl.S);
    pl.smem = 1024 + pl.header + (size_t)ns * stage;
  }
  pl.umax = k > 0 ? (int)work : 0;
  {
    const long long ng = (long long)s->batch * pl.groups;
    const long long ring = (long long)pl.nstages * stage;
    pl.spread_ok = k > 0 && !win && pl.mma && pl.nchunk == 1 && pl.S > 1 &&
                   ng <= kSpreadMaxGroups && ng * pl.umax < (1LL << 30) &&
                   ((ng + 1 + 31) / 32 * 32 + 96) * 4 <= ring;
  }
  size_t off = 0;
  const size_t rows = (size_t)s->batch * s->num_q_heads;
  if (pl.S > 1) {
    pl.off_part_o = off;
    off = align256(off + (size_t)pl.S * rows * kHeadDim * 4);
    pl.off_part_ml = off;
    off = align256(off + (size_t)pl.S * rows * 2 * 4);
  }
  if (k > 0) {
    const size_t ng = (size_t)s->batch * pl.groups;
    pl.off_upages = off;
    off = align256(off + ng * pl.umax * 4);
    pl.off_umasks = off;
    off = align256(off + ng * pl.umax * 4);
    pl.off_ucount = off;
    off = align256(off + ng * 4);
    if (pl.spread_ok) {
      pl.off_spa_o = off;
      off = align256(off + ng * pl.nw * pl.gc * kHeadDim * 4);
      pl.off_spa_ml = off;
      off = align256(off + ng * pl.nw * pl.gc * 2 * 4);
      pl.off_gmeta = off;
      off = align256(off + ng * 16);
    }
  }
  pl.total = off;
  return pl;
}

// Plans depend only on (device, shape, k): cache them, since the split search
// and the occupancy query cost host time on every call.
struct PlanEntry {
  int dev, k, win;
  kv_shape shape;
  Plan plan;
};
std::mutex g_plan_mutex;
PlanEntry g_plans[32];
int g_plan_n = 0;

bool same_shape(const kv_shape &x, const kv_shape &y) {
  return x.batch == y.batch && x.num_q_heads == y.num_q_heads &&
         x.num_kv_heads == y.num_kv_heads && x.head_dim == y.head_dim &&
         x.page_size == y.page_size && x.max_pages_per_seq == y.max_pages_per_seq &&
         x.num_phys_pages == y.num_phys_pages && x.dtype == y.dtype && x.kv_loc == y.kv_loc;
}

Plan cached_plan(const kv_shape *s, int k, bool win = false) {
  const int dev = current_device();
  {
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    for (int i = 0; i < std::min(g_plan_n, 32); ++i)
      if (g_plans[i].dev == dev && g_plans[i].k == k && g_plans[i].win == (int)win &&
          same_shape(g_plans[i].shape, *s))
        return g_plans[i].plan;
  }
  const Plan pl = make_plan(s, k, dev >= 0 ? sm_count(dev) : 152, dev >= 0, win);
  if (dev >= 0) {
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    g_plans[g_plan_n % 32] = PlanEntry{dev, k, (int)win, *s, pl};
    ++g_plan_n;
  }
  return pl;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// 3-D view [slab][rows = N * Hkv * ps][128 bytes]: a 128-element row is
// `elem` slabs of 128 bytes (strides: a row, 128 bytes), so one box of every
// slab x kTileTokens rows is one K (or V) tile of the kernel's ring, in its
// [slab][row] layout with the 128-byte swizzle.  (Two boxes per tile instead
// of one per slab: the 70B-class sparse call 176.7 -> 174.7 us.)
int make_kv_map(const kv_shape *s, const void *base, CUtensorMap *map) {
  auto fn = encode_fn();
  if (!fn) return KV_ERR_CUDA;
  const CUtensorMapDataType dt = s->dtype == KV_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : s->dtype == KV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int eb = elem_bytes(s->dtype);
  const int slabs = eb;  // 128-byte slabs per 128-element row
  cuuint64_t dims[3] = {(cuuint64_t)(128 / eb),
                        (cuuint64_t)(s->num_phys_pages * s->num_kv_heads * s->page_size),
                        (cuuint64_t)slabs};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * eb, 128};
  cuuint32_t box[3] = {(cuuint32_t)(128 / eb), (cuuint32_t)kTileTokens, (cuuint32_t)slabs};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KV_OK : KV_ERR_CUDA;
}

// The page window's part of an attention call: its state, this step's page
// scores, and the shape the attention sees (K/V = the window arrays).
struct WindowCall {
  const kv_window *win;
  const float *scores;
  kv_shape wshape;  // num_phys_pages = B * C, kv_loc = HBM
};

// Window shape and workspace: the attention plan of the window shape, then
// the fetch bits [B][Hkv][ceil(maxP / 32)] (pages this step reads from the
// source cache).
kv_shape window_shape(const kv_shape *s, int C) {
  kv_shape w = *s;
  w.num_phys_pages = (int64_t)s->batch * C;
  w.kv_loc = KV_LOC_HBM;
  return w;
}
int fetch_words(const kv_shape *s) { return (int)((s->max_pages_per_seq + 31) / 32); }
size_t window_bits_bytes(const kv_shape *s) {
  return align256((size_t)s->batch * s->num_kv_heads * fetch_words(s) * 4);
}

// Encoded tensor maps depend only on (device, base address, rows, dtype);
// encoding two per call cost measurable host time, so keep the last few.
struct MapEntry {
  int dev, dtype;
  const void *base;
  long long rows;
  CUtensorMap map;
};
std::mutex g_map_mutex;
MapEntry g_maps[16];
int g_map_n = 0;

int kv_map_cached(const kv_shape *s, const void *base, CUtensorMap *map) {
  const int dev = current_device();
  const long long rows = s->num_phys_pages * (long long)s->num_kv_heads * s->page_size;
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (int i = 0; i < std::min(g_map_n, 16); ++i) {
      const MapEntry &e = g_maps[i];
      if (e.dev == dev && e.base == base && e.rows == rows && e.dtype == s->dtype) {
        *map = e.map;
        return KV_OK;
      }
    }
  }
  const int rc = make_kv_map(s, base, map);
  if (rc == KV_OK && dev >= 0) {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    MapEntry &e = g_maps[g_map_n % 16];
    e.dev = dev;
    e.dtype = s->dtype;
    e.base = base;
    e.rows = rows;
    e.map = *map;
    ++g_map_n;
  }
  return rc;
}

// The fused selection (page score + top-K + union in one cluster launch)
// covers 16-bit data with 4 or 8 query heads per kv head, whose attention
// runs one head chunk per group.
bool fused_select_ok(const kv_shape *s) {
  const int G = s->num_q_heads / s->num_kv_heads;
  return (s->dtype == KV_F16 || s->dtype == KV_BF16) && (G == 4 || G == 8) &&
         select_fused_smem(G, s->max_pages_per_seq) <= 200 * 1024;
}

// Attention over union lists a selection call left in the workspace
// (kv_select_pages), instead of building them from `indices`.
struct ListsReady {
  bool resolved;  // entries hold physical pages (the fused selection)
  int early_inputs;
};

int attn_common(const kv_shape *s, const void *q, const void *k_cache, const void *v_cache,
                const int32_t *bt, const int32_t *ctx, const int32_t *indices, int32_t k,
                float scale, float *out, void *ws, size_t ws_bytes, void *stream,
                const WindowCall *wc = nullptr, const ListsReady *ready = nullptr) {
  int rc = check_shape(s);
  if (rc) return rc;
  if (!al16(q) || !al16(out) || !al4(bt) || !al4(ctx)) return KV_ERR_INVALID_ARG;
  if (ready && (k < 1 || wc)) return KV_ERR_INVALID_ARG;
  if (indices && (!al4(indices) || k < 1)) return KV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return KV_ERR_INVALID_ARG;
  const bool sparse_call = indices != nullptr || ready != nullptr;
  if (sparse_call && (long long)(s->max_pages_per_seq + 3) / 4 * 4 > 200 * 1024)
    return KV_ERR_UNSUPPORTED;
  // a row's pages are spread over at most 1024 splits of at most
  // kMaxListPages pages each
  if ((long long)s->max_pages_per_seq > 1024LL * kMaxListPages) return KV_ERR_UNSUPPORTED;
  const int dev = current_device();
  if (dev < 0) return KV_ERR_CUDA;
  const void *kd = nullptr, *vd = nullptr;
  if ((rc = resolve_kv(s, k_cache, &kd)) != KV_OK) return rc;
  if ((rc = resolve_kv(s, v_cache, &vd)) != KV_OK) return rc;
  const kv_shape *as = wc ? &wc->wshape : s;  // the shape the attention reads
  const Plan pl = cached_plan(as, sparse_call ? k : 0, wc != nullptr);
  const int C = wc ? wc->win->cache_pages : 0;
  const size_t need_ws = pl.total + (wc ? window_bits_bytes(s) : 0);
  if (need_ws > 0 && (ws == nullptr || ws_bytes < need_ws || !al16(ws))) return KV_ERR_WORKSPACE;
  int *status = status_ptr(dev);
  if (!status) return KV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char *w = static_cast<char *>(ws);
  uint32_t *fbits = nullptr;
  const void *src_k = kd, *src_v = vd;
  if (wc) {
    // the attention below reads the window, and this step's fetched pages
    // from the cache
    fbits = reinterpret_cast<uint32_t *>(w + pl.total);
    kd = wc->win->cache_k;
    vd = wc->win->cache_v;
  }

  AttnArgs a{};
  a.q = q;
  a.k = kd;
  a.v = vd;
  a.block_table = bt;
  a.context_lens = ctx;
  a.out = out;
  a.status = status;
  a.nphys = as->num_phys_pages;
  if (wc) {
    a.page_slot = wc->win->page_slot;
    a.cache_C = C;
    a.fetch_bits = fbits;
    a.fetch_words = fetch_words(s);
    a.src_k = src_k;
    a.src_v = src_v;
    a.src_nphys = s->num_phys_pages;
  }
  a.B = s->batch;
  a.Hq = s->num_q_heads;
  a.Hkv = s->num_kv_heads;
  a.G = s->num_q_heads / s->num_kv_heads;
  a.ps = s->page_size;
  a.maxP = s->max_pages_per_seq;
  a.nchunk = pl.nchunk;
  a.num_splits = pl.S;
  a.nstages = pl.nstages;
  a.nw = pl.nw;
  a.header_bytes = pl.header;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.debug_skip_page = g_debug_skip_page.load();
  // the sparse and window calls launch their union (or window update) kernel
  // first, which writes neither q nor the block table; a dense call's
  // attention kernel is the first of the call
  a.early_inputs = ready ? ready->early_inputs : indices ? 1 : 0;
  a.union_resolved = ready && ready->resolved ? 1 : 0;
  const int split_mode = g_split_mode.load();
  a.spread = 0;
  if (a.union_resolved && pl.spread_ok && split_mode != 0) {
    // a CTA's share of the link when all CTAs stream (nominal HBM 7 TB/s,
    // host link 200 GB/s), in bytes per ns
    const double link = as->kv_loc == KV_LOC_HBM ? 7.0e3 : 2.0e2;
    const double ctas = (double)pl.S * s->batch * pl.groups;
    const double share_bytes = (double)((pl.umax + pl.S - 1) / pl.S) * 2.0 * as->page_size *
                               kHeadDim * elem_bytes(as->dtype);
    if (split_mode == 1) a.spread = 2;
    else if (split_mode == 2 || share_bytes / (link / ctas) >= KVS_SPREAD_MIN_CTA_NS) a.spread = 1;
    // K/V bytes a CTA streams in KVS_SPREAD_FIXED_NS
    a.spread_min_gain = (int)std::min(1.0e9, link / ctas * KVS_SPREAD_FIXED_NS);
  }
  if (a.spread) {
    a.ngroups = s->batch * pl.groups;
    a.spa_o = reinterpret_cast<float *>(w + pl.off_spa_o);
    a.spa_ml = reinterpret_cast<float *>(w + pl.off_spa_ml);
    a.gmeta = reinterpret_cast<int32_t *>(w + pl.off_gmeta);
  }
  if (pl.S > 1) {
    a.part_o = reinterpret_cast<float *>(w + pl.off_part_o);
    a.part_ml = reinterpret_cast<float *>(w + pl.off_part_ml);
  }
  if (sparse_call) {
    a.union_pages = reinterpret_cast<int32_t *>(w + pl.off_upages);
    a.union_masks = reinterpret_cast<uint32_t *>(w + pl.off_umasks);
    a.union_count = reinterpret_cast<int32_t *>(w + pl.off_ucount);
    a.umax = pl.umax;
  }
  if (indices) {
    cudaError_t e;
    if (wc) {
      // the window step: update the state and mark this step's fetches, and,
      // in the same launch beside it, build the union lists
      const kv_window *win = wc->win;
      e = launch_window_step(indices, wc->scores, ctx, s->batch, s->num_q_heads, s->num_kv_heads,
                             s->page_size, s->max_pages_per_seq, k, C, win->slot_page,
                             win->page_slot, fbits, win->stats, pl.gc, pl.umax,
                             const_cast<int32_t *>(a.union_pages),
                             const_cast<uint32_t *>(a.union_masks),
                             const_cast<int32_t *>(a.union_count), status, st);
    } else {
      e = launch_union(indices, ctx, s->batch, s->num_q_heads, s->num_kv_heads, pl.gc,
                       s->page_size, s->max_pages_per_seq, k, pl.umax,
                       const_cast<int32_t *>(a.union_pages), const_cast<uint32_t *>(a.union_masks),
                       const_cast<int32_t *>(a.union_count), status, st);
    }
    if (e != cudaSuccess) return KV_ERR_CUDA;
  }
  CUtensorMap tk, tv;
  memset(&tk, 0, sizeof tk);
  memset(&tv, 0, sizeof tv);
  a.use_tma = as->kv_loc == KV_LOC_HBM ? 1 : 0;
  if (a.use_tma) {
    if ((rc = kv_map_cached(as, kd, &tk)) != KV_OK) return rc;
    if ((rc = kv_map_cached(as, vd, &tv)) != KV_OK) return rc;
  }
  dim3 grid(pl.S, pl.groups, s->batch);
  cudaError_t e = wc       ? launch_attn_win(s->dtype, pl.gc, pl.mma, a, &tk, &tv, grid, pl.smem, st)
                  : pl.mma ? launch_attn_mma(s->dtype, pl.gc, a, &tk, &tv, grid, pl.smem, st)
                           : launch_attn_core(s->dtype, pl.gc, a, &tk, &tv, grid, pl.smem, st);
  if (e != cudaSuccess) return KV_ERR_CUDA;
  if (pl.S > 1) {
    e = a.spread ? launch_combine_lists(a.part_o, a.part_ml, a.spa_o, a.spa_ml, a.gmeta, out,
                                        pl.S, s->batch, s->num_q_heads, s->num_kv_heads, pl.nw,
                                        status, st)
                 : launch_combine(a.part_o, a.part_ml, out, pl.S, s->batch, s->num_q_heads, st);
    if (e != cudaSuccess) return KV_ERR_CUDA;
  }
  return KV_OK;
}

}  // namespace

extern "C" {

int kv_page_minmax_build(const kv_shape *shape, const void *k_cache, const int32_t *block_table,
                         const int32_t *context_lens, void *minmax, void *stream) {
  KV_API_RANGE();
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!al16(minmax) || !al4(block_table) || !al4(context_lens)) return KV_ERR_INVALID_ARG;
  const int dev = current_device();
  if (dev < 0) return KV_ERR_CUDA;
  const void *kd = nullptr;
  if ((rc = resolve_kv(shape, k_cache, &kd)) != KV_OK) return rc;
  int *status = status_ptr(dev);
  if (!status) return KV_ERR_CUDA;
  cudaError_t e = launch_minmax_build(shape->dtype, kd, block_table, context_lens, minmax,
                                      shape->batch, shape->num_kv_heads, shape->page_size,
                                      shape->max_pages_per_seq, shape->num_phys_pages, status,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

int kv_append_token(const kv_shape *shape, const void *k_new, const void *v_new, void *k_cache,
                    void *v_cache, const int32_t *block_table, const int32_t *context_lens,
                    int32_t *context_lens_out, void *minmax, void *stream) {
  KV_API_RANGE();
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!al16(k_new) || !al16(v_new) || !al4(block_table) || !al4(context_lens) ||
      (minmax && !al16(minmax)) || (context_lens_out && !al4(context_lens_out)))
    return KV_ERR_INVALID_ARG;
  const int dev = current_device();
  if (dev < 0) return KV_ERR_CUDA;
  const void *kd = nullptr, *vd = nullptr;
  if ((rc = resolve_kv(shape, k_cache, &kd)) != KV_OK) return rc;
  if ((rc = resolve_kv(shape, v_cache, &vd)) != KV_OK) return rc;
  int *status = status_ptr(dev);
  if (!status) return KV_ERR_CUDA;
  cudaError_t e = launch_append(shape->dtype, k_new, v_new, const_cast<void *>(kd),
                                const_cast<void *>(vd), block_table, context_lens,
                                context_lens_out, minmax, shape->batch, shape->num_kv_heads,
                                shape->page_size, shape->max_pages_per_seq,
                                shape->num_phys_pages, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

// early_inputs: the kernel before this one in the stream is the library's
// own (see launch_page_score)
static int page_score_common(const kv_shape *shape, const void *q, const void *minmax,
                             const int32_t *block_table, const int32_t *context_lens,
                             float *scores, int early_inputs, void *stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!al16(q) || !al16(minmax) || !al16(scores) || !al4(block_table) || !al4(context_lens))
    return KV_ERR_INVALID_ARG;
  const int dev = current_device();
  if (dev < 0) return KV_ERR_CUDA;
  int *status = status_ptr(dev);
  if (!status) return KV_ERR_CUDA;
  cudaError_t e = launch_page_score(shape->dtype, false, q, minmax, block_table, context_lens,
                                    scores, shape->batch, shape->num_q_heads,
                                    shape->num_kv_heads, shape->page_size,
                                    shape->max_pages_per_seq, shape->num_phys_pages,
                                    early_inputs, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

int kv_page_score(const kv_shape *shape, const void *q, const void *minmax,
                  const int32_t *block_table, const int32_t *context_lens, float *scores,
                  void *stream) {
  KV_API_RANGE();
  return page_score_common(shape, q, minmax, block_table, context_lens, scores, 0, stream);
}

static int mean_build_common(const kv_shape *shape, const void *k_cache, const int32_t *block_table,
                      const int32_t *context_lens, void *mean, bool last_only, void *stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!al16(mean) || !al4(block_table) || !al4(context_lens)) return KV_ERR_INVALID_ARG;
  const int dev = current_device();
  if (dev < 0) return KV_ERR_CUDA;
  const void *kd = nullptr;
  if ((rc = resolve_kv(shape, k_cache, &kd)) != KV_OK) return rc;
  int *status = status_ptr(dev);
  if (!status) return KV_ERR_CUDA;
  cudaError_t e = launch_mean_build(shape->dtype, kd, block_table, context_lens, mean,
                                    shape->batch, shape->num_kv_heads, shape->page_size,
                                    shape->max_pages_per_seq, shape->num_phys_pages, last_only,
                                    status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

int kv_page_mean_build(const kv_shape *shape, const void *k_cache, const int32_t *block_table,
                       const int32_t *context_lens, void *mean, void *stream) {
  KV_API_RANGE();
  return mean_build_common(shape, k_cache, block_table, context_lens, mean, false, stream);
}

int kv_page_mean_refresh(const kv_shape *shape, const void *k_cache, const int32_t *block_table,
                         const int32_t *context_lens, void *mean, void *stream) {
  KV_API_RANGE();
  return mean_build_common(shape, k_cache, block_table, context_lens, mean, true, stream);
}

int kv_page_score_mean(const kv_shape *shape, const void *q, const void *mean,
                       const int32_t *block_table, const int32_t *context_lens, float *scores,
                       void *stream) {
  KV_API_RANGE();
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!al16(q) || !al16(mean) || !al16(scores) || !al4(block_table) || !al4(context_lens))
    return KV_ERR_INVALID_ARG;
  const int dev = current_device();
  if (dev < 0) return KV_ERR_CUDA;
  int *status = status_ptr(dev);
  if (!status) return KV_ERR_CUDA;
  cudaError_t e = launch_page_score(shape->dtype, true, q, mean, block_table, context_lens,
                                    scores, shape->batch, shape->num_q_heads,
                                    shape->num_kv_heads, shape->page_size,
                                    shape->max_pages_per_seq, shape->num_phys_pages, 0, status,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

size_t kv_topk_workspace_bytes(const kv_shape *shape, int32_t k) {
  (void)shape;
  (void)k;
  return 0;
}

int kv_topk_select_forced(const kv_shape *shape, const float *scores,
                          const int32_t *context_lens, int32_t k, int32_t sink_tokens,
                          int32_t local_tokens, int32_t *indices, void *workspace,
                          size_t workspace_bytes, void *stream) {
  KV_API_RANGE();
  (void)workspace;
  (void)workspace_bytes;
  int rc = check_shape(shape);
  if (rc) return rc;
  if (k < 1 || sink_tokens < 0 || local_tokens < 0 || !al16(scores) || !al4(indices) ||
      !al4(context_lens))
    return KV_ERR_INVALID_ARG;
  const int dev = current_device();
  if (dev < 0) return KV_ERR_CUDA;
  int *status = status_ptr(dev);
  if (!status) return KV_ERR_CUDA;
  cudaError_t e = launch_topk(scores, context_lens, shape->batch, shape->num_q_heads,
                              shape->page_size, shape->max_pages_per_seq, k, sink_tokens,
                              local_tokens, indices, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

int kv_topk_select(const kv_shape *shape, const float *scores, const int32_t *context_lens,
                   int32_t k, int32_t *indices, void *workspace, size_t workspace_bytes,
                   void *stream) {
  KV_API_RANGE();
  return kv_topk_select_forced(shape, scores, context_lens, k, 0, 0, indices, workspace,
                               workspace_bytes, stream);
}

size_t kv_attn_workspace_bytes(const kv_shape *shape, int32_t k) {
  if (check_shape(shape) != KV_OK || k < 0) return 0;
  return cached_plan(shape, k).total;
}

int32_t kv_attn_num_splits(const kv_shape *shape, int32_t k) {
  if (check_shape(shape) != KV_OK || k < 0) return 0;
  return cached_plan(shape, k).S;
}

// The cluster scores the pages itself while each CTA's share is short (one
// launch for the whole selection); with longer rows its few CTAs read the
// index too slowly, so the page-score kernel's wide grid scores them first
// (128k-token rows: 22.6 us fused against 13.3 us for score + top-K).
#ifndef KVS_SELECT_SCORE_MAX_PAGES
#define KVS_SELECT_SCORE_MAX_PAGES 512
#endif
bool select_scores_in_cluster(const kv_shape *s) {
  const int G = s->num_q_heads / s->num_kv_heads;
  return select_fused_pages_per_cta(G, s->max_pages_per_seq) <= KVS_SELECT_SCORE_MAX_PAGES;
}

static size_t select_ws_bytes(const kv_shape *shape, int32_t k) {
  size_t n = cached_plan(shape, k).total;
  if (!fused_select_ok(shape) || !select_scores_in_cluster(shape))  // scores kept there
    n += align256((size_t)shape->batch * shape->num_q_heads * shape->max_pages_per_seq * 4);
  return n;
}

size_t kv_select_workspace_bytes(const kv_shape *shape, int32_t k) {
  if (check_shape(shape) != KV_OK || k < 1) return 0;
  return select_ws_bytes(shape, k);
}

// early_inputs: as for the score kernel (the previous kernel in the stream is
// the library's own)
static int select_common(const kv_shape *shape, const void *q, const void *minmax,
                         const int32_t *block_table, const int32_t *context_lens, int32_t k,
                         int32_t sink_tokens, int32_t local_tokens, int32_t *indices,
                         void *workspace, size_t workspace_bytes, int early_inputs,
                         void *stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  if (k < 1 || sink_tokens < 0 || local_tokens < 0 || !al16(q) || !al16(minmax) ||
      !al4(block_table) || !al4(context_lens) || !al4(indices))
    return KV_ERR_INVALID_ARG;
  if ((long long)(shape->max_pages_per_seq + 3) / 4 * 4 > 200 * 1024) return KV_ERR_UNSUPPORTED;
  const int dev = current_device();
  if (dev < 0) return KV_ERR_CUDA;
  const Plan pl = cached_plan(shape, k);
  const size_t need = select_ws_bytes(shape, k);
  if (workspace == nullptr || workspace_bytes < need || !al16(workspace)) return KV_ERR_WORKSPACE;
  int *status = status_ptr(dev);
  if (!status) return KV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char *w = static_cast<char *>(workspace);
  int32_t *upages = reinterpret_cast<int32_t *>(w + pl.off_upages);
  uint32_t *umasks = reinterpret_cast<uint32_t *>(w + pl.off_umasks);
  int32_t *ucount = reinterpret_cast<int32_t *>(w + pl.off_ucount);
  cudaError_t e;
  if (fused_select_ok(shape)) {
    SelectArgs a{};
    a.q = q;
    a.table = minmax;
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.indices = indices;
    a.upages = upages;
    a.umasks = umasks;
    a.ucount = ucount;
    a.status = status;
    a.nphys = shape->num_phys_pages;
    a.Hq = shape->num_q_heads;
    a.Hkv = shape->num_kv_heads;
    a.ps = shape->page_size;
    a.maxP = shape->max_pages_per_seq;
    a.K = k;
    a.umax = pl.umax;
    a.PC = select_fused_pages_per_cta(shape->num_q_heads / shape->num_kv_heads, a.maxP);
    a.sink_tokens = sink_tokens;
    a.local_tokens = local_tokens;
    a.early_inputs = early_inputs;
    e = cudaSuccess;
    if (!select_scores_in_cluster(shape)) {
      float *scores = reinterpret_cast<float *>(w + pl.total);
      e = launch_page_score(shape->dtype, false, q, minmax, block_table, context_lens, scores,
                            shape->batch, shape->num_q_heads, shape->num_kv_heads,
                            shape->page_size, shape->max_pages_per_seq, shape->num_phys_pages,
                            early_inputs, status, st);
      a.scores = scores;
      a.early_inputs = 1;  // after the score kernel, which writes neither q nor the table
    }
    if (e == cudaSuccess) e = launch_select_fused(shape->dtype, a, shape->batch, st);
  } else {
    float *scores = reinterpret_cast<float *>(w + pl.total);
    e = launch_page_score(shape->dtype, false, q, minmax, block_table, context_lens, scores,
                          shape->batch, shape->num_q_heads, shape->num_kv_heads,
                          shape->page_size, shape->max_pages_per_seq, shape->num_phys_pages,
                          early_inputs, status, st);
    if (e == cudaSuccess)
      e = launch_topk(scores, context_lens, shape->batch, shape->num_q_heads, shape->page_size,
                      shape->max_pages_per_seq, k, sink_tokens, local_tokens, indices, status,
                      st);
    if (e == cudaSuccess)
      e = launch_union(indices, context_lens, shape->batch, shape->num_q_heads,
                       shape->num_kv_heads, pl.gc, shape->page_size, shape->max_pages_per_seq,
                       k, pl.umax, upages, umasks, ucount, status, st);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  return KV_OK;
}

int kv_select_pages(const kv_shape *shape, const void *q, const void *minmax,
                    const int32_t *block_table, const int32_t *context_lens, int32_t k,
                    int32_t sink_tokens, int32_t local_tokens, int32_t *indices, void *workspace,
                    size_t workspace_bytes, void *stream) {
  KV_API_RANGE();
  return select_common(shape, q, minmax, block_table, context_lens, k, sink_tokens, local_tokens,
                       indices, workspace, workspace_bytes, 0, stream);
}

static int attn_selected_common(const kv_shape *shape, const void *q, const void *k_cache,
                                const void *v_cache, const int32_t *block_table,
                                const int32_t *context_lens, int32_t k, float scale, float *out,
                                void *workspace, size_t workspace_bytes, int early_inputs,
                                void *stream) {
  if (check_shape(shape) != KV_OK) return check_shape(shape);
  if (k < 1) return KV_ERR_INVALID_ARG;
  const ListsReady ready{fused_select_ok(shape), early_inputs};
  return attn_common(shape, q, k_cache, v_cache, block_table, context_lens, nullptr, k, scale,
                     out, workspace, workspace_bytes, stream, nullptr, &ready);
}

int kv_sparse_decode_attn_selected(const kv_shape *shape, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_table,
                                   const int32_t *context_lens, int32_t k, float scale,
                                   float *out, void *workspace, size_t workspace_bytes,
                                   void *stream) {
  KV_API_RANGE();
  return attn_selected_common(shape, q, k_cache, v_cache, block_table, context_lens, k, scale,
                              out, workspace, workspace_bytes, 0, stream);
}

int kv_sparse_decode_attn(const kv_shape *shape, const void *q, const void *k_cache,
                          const void *v_cache, const int32_t *block_table,
                          const int32_t *context_lens, const int32_t *indices, int32_t k,
                          float scale, float *out, void *workspace, size_t workspace_bytes,
                          void *stream) {
  KV_API_RANGE();
  if (!indices) return KV_ERR_INVALID_ARG;
  return attn_common(shape, q, k_cache, v_cache, block_table, context_lens, indices, k, scale, out,
                     workspace, workspace_bytes, stream);
}

int kv_dense_decode_attn(const kv_shape *shape, const void *q, const void *k_cache,
                         const void *v_cache, const int32_t *block_table,
                         const int32_t *context_lens, float scale, float *out, void *workspace,
                         size_t workspace_bytes, void *stream) {
  KV_API_RANGE();
  return attn_common(shape, q, k_cache, v_cache, block_table, context_lens, nullptr, 0, scale,
                     out, workspace, workspace_bytes, stream);
}

// Device-visible address of host memory the device has mapped (pinned), or
// nullptr when it is not mapped.
static void *mapped_host(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

int kv_decode_step(const kv_shape *shape, const kv_step_io *io, void *stream) {
  KV_API_RANGE();
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!io || !io->q_host || !io->context_lens_host || !io->out_host || io->k < 0)
    return KV_ERR_INVALID_ARG;
  if (io->k > 0 && (!io->minmax || !io->indices)) return KV_ERR_INVALID_ARG;
  if (io->k > 0 && !io->scores && io->workspace_bytes < select_ws_bytes(shape, io->k))
    return KV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)shape->batch * shape->num_q_heads;
  // Host buffers the device has mapped are read (q, lengths) and written
  // (out) across the host link, as the pages read K/V; others are copied
  // through the device buffers.  For a sparse step, mapped q and lengths are
  // first staged into the device buffers by one kernel whose host reads
  // overlap the previous kernel, so the score, top-K, union and attention
  // kernels each read device memory instead of paying a host round trip
  // (Llama-3.1-8B 32k step 61.3 -> 59.5 us).  That staging kernel never
  // releases its dependents early, so the score kernel after it may load q
  // and the block table before its own PDL wait.  A dense step is one
  // attention kernel: it reads q and the lengths in place.
  const void *q = mapped_host(io->q_host);
  const int32_t *ctx = static_cast<const int32_t *>(mapped_host(io->context_lens_host));
  float *out = static_cast<float *>(mapped_host(io->out_host));
  const size_t q_bytes = rows * kHeadDim * elem_bytes(shape->dtype);
  int staged = 0;
  if (io->k > 0 && q && ctx && io->q && io->context_lens && al16(q) && al16(io->q) &&
      al4(io->context_lens)) {
    if (launch_stage_inputs(q, io->q, q_bytes, ctx, io->context_lens, shape->batch, st) !=
        cudaSuccess) {
      cudaGetLastError();
      return KV_ERR_CUDA;
    }
    q = io->q;
    ctx = io->context_lens;
    staged = 1;
  }
  if (!q) {
    if (!al16(io->q)) return KV_ERR_INVALID_ARG;
    if (cudaMemcpyAsync(io->q, io->q_host, q_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) {
      cudaGetLastError();
      return KV_ERR_CUDA;
    }
    q = io->q;
  }
  if (!ctx) {
    if (!al4(io->context_lens)) return KV_ERR_INVALID_ARG;
    if (cudaMemcpyAsync(io->context_lens, io->context_lens_host, (size_t)shape->batch * 4,
                        cudaMemcpyHostToDevice, st) != cudaSuccess) {
      cudaGetLastError();
      return KV_ERR_CUDA;
    }
    ctx = io->context_lens;
  }
  const bool copy_out = out == nullptr;
  if (copy_out) {
    if (!al16(io->out)) return KV_ERR_INVALID_ARG;
    out = io->out;
  }
  if (io->k > 0 && io->workspace_bytes >= select_ws_bytes(shape, io->k)) {
    // selection and the group unions in one launch where the shape allows,
    // then the attention over those lists; the selection kernel writes
    // neither q nor the block table, so the attention may load them early
    if ((rc = select_common(shape, q, io->minmax, io->block_table, ctx, io->k, 0, 0,
                            io->indices, io->workspace, io->workspace_bytes, staged, stream)) !=
        KV_OK)
      return rc;
    rc = attn_selected_common(shape, q, io->k_cache, io->v_cache, io->block_table, ctx, io->k,
                              io->scale, out, io->workspace, io->workspace_bytes, 1, stream);
  } else if (io->k > 0) {
    if ((rc = page_score_common(shape, q, io->minmax, io->block_table, ctx, io->scores, staged,
                                stream)) != KV_OK)
      return rc;
    if ((rc = kv_topk_select(shape, io->scores, ctx, io->k, io->indices, nullptr, 0, stream)) !=
        KV_OK)
      return rc;
    rc = kv_sparse_decode_attn(shape, q, io->k_cache, io->v_cache, io->block_table, ctx,
                               io->indices, io->k, io->scale, out, io->workspace,
                               io->workspace_bytes, stream);
  } else {
    rc = kv_dense_decode_attn(shape, q, io->k_cache, io->v_cache, io->block_table, ctx,
                              io->scale, out, io->workspace, io->workspace_bytes, stream);
  }
  if (rc != KV_OK) return rc;
  if (copy_out && cudaMemcpyAsync(io->out_host, io->out, rows * kHeadDim * 4,
                                  cudaMemcpyDeviceToHost, st) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  return KV_OK;
}

size_t kv_window_workspace_bytes(const kv_shape *shape, int32_t k, int32_t cache_pages) {
  if (check_shape(shape) != KV_OK || k < 1 || cache_pages < 1) return 0;
  const kv_shape w = window_shape(shape, cache_pages);
  return cached_plan(&w, k, true).total + window_bits_bytes(shape);
}

static int check_window(const kv_shape *s, const kv_window *win, int32_t k) {
  if (!win || win->cache_pages < 1) return KV_ERR_INVALID_ARG;
  const long long C = win->cache_pages;
  const long long G = s->num_q_heads / s->num_kv_heads;
  if (C < std::min<long long>(G * k, s->max_pages_per_seq)) return KV_ERR_INVALID_ARG;
  if (window_update_smem(s->max_pages_per_seq, (int)C) > 200 * 1024) return KV_ERR_UNSUPPORTED;
  if ((long long)s->batch * C * s->num_kv_heads * s->page_size > INT_MAX) return KV_ERR_UNSUPPORTED;
  if (!al16(win->cache_k) || !al16(win->cache_v) || !al4(win->slot_page) ||
      !al4(win->page_slot) || (win->stats && !al4(win->stats)))
    return KV_ERR_INVALID_ARG;
  return KV_OK;
}

int kv_window_reset(const kv_shape *shape, const kv_window *win, void *stream) {
  KV_API_RANGE();
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!win || win->cache_pages < 1 || !al4(win->slot_page) || !al4(win->page_slot))
    return KV_ERR_INVALID_ARG;
  const long long groups = (long long)shape->batch * shape->num_kv_heads;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_fill(win->slot_page, groups * win->cache_pages, -1, st) != cudaSuccess ||
      launch_fill(win->page_slot, groups * shape->max_pages_per_seq, -1, st) != cudaSuccess)
    return KV_ERR_CUDA;
  return KV_OK;
}

int kv_sparse_decode_attn_window(const kv_shape *shape, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_table,
                                 const int32_t *context_lens, const int32_t *indices, int32_t k,
                                 const float *scores, float scale, float *out,
                                 const kv_window *win, void *workspace, size_t workspace_bytes,
                                 void *stream) {
  KV_API_RANGE();
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!indices || k < 1 || !al16(scores)) return KV_ERR_INVALID_ARG;
  if ((rc = check_window(shape, win, k)) != KV_OK) return rc;
  cudaPointerAttributes at;
  for (const void *p : {win->cache_k, win->cache_v}) {
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();
      return KV_ERR_CUDA;
    }
    if (at.type != cudaMemoryTypeDevice) return KV_ERR_LOCATION;
  }
  WindowCall wc{win, scores, window_shape(shape, win->cache_pages)};
  return attn_common(shape, q, k_cache, v_cache, block_table, context_lens, indices, k, scale, out,
                     workspace, workspace_bytes, stream, &wc);
}

int kv_device_status(void *stream) {
  const int dev = current_device();
  if (dev < 0) return KV_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  int *p = status_ptr(dev);
  if (!p) return KV_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return KV_ERR_CUDA;
    }
  }
  return v;
}

const char *kv_status_string(int status) {
  switch (status) {
    case KV_OK: return "KV_OK";
    case KV_ERR_INVALID_ARG: return "KV_ERR_INVALID_ARG";
    case KV_ERR_UNSUPPORTED: return "KV_ERR_UNSUPPORTED";
    case KV_ERR_LOCATION: return "KV_ERR_LOCATION";
    case KV_ERR_WORKSPACE: return "KV_ERR_WORKSPACE";
    case KV_ERR_CUDA: return "KV_ERR_CUDA";
    case KV_ERR_DEVICE_TIMEOUT: return "KV_ERR_DEVICE_TIMEOUT";
    case KV_ERR_BOUNDS: return "KV_ERR_BOUNDS";
    default: return "KV_ERR_UNKNOWN";
  }
}

int kv_debug_split_mode(int32_t mode) {
  if (mode < -1 || mode > 2) return KV_ERR_INVALID_ARG;
  g_split_mode.store(mode);
  return KV_OK;
}

int kv_debug_config(int32_t skip_page, uint64_t wait_limit_ns) {
  if (wait_limit_ns == 0 || wait_limit_ns > 60000000000ull) return KV_ERR_INVALID_ARG;
  g_debug_skip_page.store(skip_page < 0 ? -1 : skip_page);
  g_wait_limit_ns.store(wait_limit_ns);
  return KV_OK;
}

}  // extern "C"
