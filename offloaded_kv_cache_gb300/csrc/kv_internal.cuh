// kv_internal.cuh -- device helpers and launcher declarations shared by the
// kvsparse translation units (sm_103a only).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "kvsparse.h"

namespace kvs {

constexpr int kHeadDim = 128;
// tokens per K/V tile: one pipeline stage, one TMA box height
constexpr int kTileTokens = 16;

// ---------------------------------------------------------------------------
// device status word: the first error a kernel records wins
// ---------------------------------------------------------------------------
__device__ __forceinline__ void flag_error(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
template <class T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kBytes = 4;
  __device__ __forceinline__ static float to_f32(float x) { return x; }
};
template <> struct Elem<__half> {
  static constexpr int kBytes = 2;
  __device__ __forceinline__ static float to_f32(__half x) { return __half2float(x); }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  __device__ __forceinline__ static float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
};

// two packed 16-bit elements -> two floats
__device__ __forceinline__ float2 unpack2(uint32_t w, __half) {
  return __half22float2(*reinterpret_cast<__half2 *>(&w));
}
__device__ __forceinline__ float2 unpack2(uint32_t w, __nv_bfloat16) {
  // bf16 is the upper half of an fp32: widening is a shift / mask
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// ---------------------------------------------------------------------------
// IEEE totalOrder keys (non-NaN): unsigned order of the key == totalOrder of
// the value, so -0.0 < +0.0 and min/max are exact and order independent
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t key16x2(uint32_t x) {
  uint32_t s = (x >> 15) & 0x00010001u;  // sign bit of each half
  return x ^ (0x80008000u | (s * 0x7FFFu));
}
__device__ __forceinline__ uint32_t unkey16x2(uint32_t k) {
  uint32_t s = ((~k) >> 15) & 0x00010001u;  // halves that were negative
  return k ^ (0x80008000u | (s * 0x7FFFu));
}
__device__ __forceinline__ uint32_t key32(uint32_t x) {
  return x ^ (uint32_t)(((int32_t)x >> 31) | (int32_t)0x80000000);
}
__device__ __forceinline__ uint32_t unkey32(uint32_t k) {
  return k ^ (uint32_t)(((int32_t)~k >> 31) | (int32_t)0x80000000);
}

// ---------------------------------------------------------------------------
// fast exp2 (PTX ex2.approx: relative error ~2^-22; ex2(-inf) = +0)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch.  Every kernel of the path waits for its
// predecessor in the stream to finish (and its writes to be visible) before
// it reads anything a kernel of the library may have written (pdl_wait), and
// lets the next kernel be scheduled once its own main loop is done
// (pdl_trigger), so the next kernel's launch and prologue overlap this
// kernel's tail.  Inputs no kernel of the library writes (q, the block table)
// are read before the wait only by a kernel whose predecessor in the stream
// is known to be one of the library's own (a later kernel of the same call):
// the first kernel of a call may follow a kernel of another library that
// releases its dependents before it writes them, so it reads every input
// after its wait.  No data dependence changes: a kernel that never reaches
// pdl_trigger releases its dependent when it exits.
// Kernel parameters are not declared __restrict__: the compiler may treat a
// load through a const __restrict__ pointer as invariant and schedule it
// above the wait, which returned stale split partials in the combine.
//   KVS_PDL 0: plain stream order; 1: trigger at entry; 2: trigger late.
// ---------------------------------------------------------------------------
#ifndef KVS_PDL
#define KVS_PDL 2
#endif
__device__ __forceinline__ void pdl_wait() {
#if KVS_PDL == 1
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
#if KVS_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
__device__ __forceinline__ void pdl_trigger() {
#if KVS_PDL == 2
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = KVS_PDL ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier (CTA scope) with bounded waits
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Global loads issued where they stand: volatile asm keeps their order
// among themselves and against barriers, so a load meant to be in flight
// beside others (speculatively, its result used only on one branch) is not
// sunk by the compiler into that branch, behind a decision that needs its
// own round trip.  The result is waited for at its first use, as usual.
__device__ __forceinline__ int32_t ld_issue(const int32_t *p) {
  int32_t v;
  asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_issue(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float ld_issue(const float *p) {
  float v;
  asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int4 ld_issue(const int4 *p) {
  int4 v;
  asm volatile("ld.global.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase of `parity` to complete; gives up after limit_ns of
// wall time and returns false (the caller records KV_ERR_DEVICE_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// async copies into shared memory
// ---------------------------------------------------------------------------
// TMA tiled load of a 3-D box (x = element column within a 128-byte slab,
// y = row, z = slab) completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// 16-byte asynchronous global->shared copy (L2 only).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once all prior cp.async of this thread have landed; the
// barrier's expected count already includes this arrival.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// Wait until every cp.async of this thread has landed.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------------------
// 128-byte swizzle: inside each 1024-byte block of eight 128-byte rows, the
// 16-byte chunk c of row r sits at chunk c ^ (r & 7).  This is the layout TMA
// writes with CU_TENSOR_MAP_SWIZZLE_128B into a 1024-byte aligned box; the
// cp.async producer writes the same layout by hand.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------------------
// launch parameter blocks (host fills, kernels read)
// ---------------------------------------------------------------------------
struct AttnArgs {
  const void *q;
  const void *k;  // device-visible K cache
  const void *v;  // device-visible V cache
  const int32_t *block_table;
  const int32_t *context_lens;
  const int32_t *union_pages;   // sparse: [B][groups][umax], else null
  const uint32_t *union_masks;  // sparse: [B][groups][umax]
  const int32_t *union_count;   // sparse: [B][groups]
  const int32_t *page_slot;     // window: [B][Hkv][maxP] slot of a page, else null
  int cache_C;                  // window: slots per (b, kv head); K/V are the window
  const uint32_t *fetch_bits;   // window: [B][Hkv][fetch_words] pages read from the source
  int fetch_words;              // window: ceil(maxP / 32)
  const void *src_k;            // window: device-visible source K cache (host or HBM)
  const void *src_v;            // window: device-visible source V cache
  long long src_nphys;          // window: physical pages of the source cache
  float *out;                   // [B][Hq][d]      (num_splits == 1)
  float *part_o;                // [S][B][Hq][d]   (num_splits > 1)
  float *part_ml;               // [S][B][Hq][2]   (log2-domain max, sum)
  int *status;
  long long nphys;
  int B, Hq, Hkv, G, ps, maxP;
  int nchunk;      // head chunks per kv head (G / heads-per-CTA)
  int num_splits;  // CTAs per (b, head chunk)
  int umax;        // union capacity per group (sparse)
  int nstages;     // pipeline depth, a multiple of nw
  int nw;          // consumer warps (blockDim.x == 32 * (1 + nw))
  int header_bytes;  // shared-memory bytes before the stage ring (multiple of 1024)
  int use_tma;     // 1: TMA producer, 0: cp.async producer
  float scale_log2;
  unsigned long long wait_limit_ns;
  int debug_skip_page;  // >= 0: the producer never fills that page (timeout test)
  // 1: the kernel before this one in the stream is one of this library's that
  // writes neither q nor the block table, so they may load before the PDL
  // wait; 0 (the first kernel of a call): they load after it, since a kernel
  // of another library may release its dependents before it writes them
  int early_inputs;
  // sparse: 1 when the union lists hold resolved entries (physical page;
  // valid tokens | head mask << 8), as the fused selection writes them
  int union_resolved;
  // Resolved lists, one head chunk per group, num_splits > 1: 1 lets the
  // kernel cut the concatenation of every group's list into equal chunks, one
  // per CTA, when every group is at least a chunk long (so a CTA covers the
  // tail of one group and the head of the next at most) and the longest CTA of
  // the split per group would hold spread_min_gain bytes more; 2 whenever
  // every group is a chunk long (testing); otherwise (and with 0) each group's
  // list is split over its own num_splits CTAs.  Either way the CTAs record in
  // gmeta[g] where the combine finds group g's partials.
  int spread;
  int spread_min_gain;
  int ngroups;      // B * Hkv
  float *spa_o;     // [ngroups][nw][GC][d]: per consumer warp, a group's tail
  float *spa_ml;    // [ngroups][nw][GC][2]   segment in a CTA that goes on to the next group
  int32_t *gmeta;   // [ngroups][4]: see kSpreadMeta*
};

// gmeta[g] = {mode, first CTA, last CTA, tail}: mode kSplitPerGroup (group g's
// partials are splits 0..S-1 of g), or kSplitSpread (the merged partials of
// CTAs first..last, except that with tail = 1 the last CTA's part of g is its
// first of two segments and sits in spa_o/spa_ml[g] as nw warp partials).
constexpr int kSplitPerGroup = 0;
constexpr int kSplitSpread = 1;

// Arguments of the fused selection kernel (page score + top-K + union).
struct SelectArgs {
  const void *q;               // [B][Hq][d]
  const void *table;           // min/max index [N_phys][Hkv][2][d]
  const int32_t *block_table;  // [B][maxP]
  const int32_t *context_lens; // [B]
  const float *scores;         // [B][Hq][maxP] page scores already computed, or null:
                               // the kernel scores the pages itself
  int32_t *indices;            // [B][Hq][K]
  int32_t *upages;             // [B][Hkv][umax]: physical page (-1: bad entry)
  uint32_t *umasks;            // [B][Hkv][umax]: valid tokens | head mask << 8
  int32_t *ucount;             // [B][Hkv]
  int *status;
  long long nphys;
  int Hq, Hkv, ps, maxP, K, umax;
  int PC;                      // pages each CTA scores (a multiple of 32)
  int sink_tokens, local_tokens;
  int early_inputs;            // as AttnArgs::early_inputs
};

// Attention CTA shape: one producer warp plus 1..kMaxConsumerWarps consumer
// warps (chosen per launch); a CTA owns at most kMaxListPages pages.
constexpr int kMaxConsumerWarps = 4;
constexpr int kAttnMaxThreads = 32 * (1 + kMaxConsumerWarps);
constexpr int kMaxListPages = 512;

// Bytes of an attention CTA's shared memory before its page list: mbarriers,
// then (CUDA-core path) q in fp32 and the per-warp weight buffers.  The page
// list follows; the stage ring starts at the next 1024-byte boundary.
__host__ __device__ inline int attn_fixed_header(int elem_bytes, int gc, bool mma) {
  const int SL = elem_bytes, QSTR = 128 / elem_bytes + 4, TP = 32 / SL;
  int off = 256;
  if (!mma) off += gc * SL * QSTR * 4 + 4 * gc * TP * 4;  // q_s + pbuf (<= 4 warps)
  return (off + 255) & ~255;
}
constexpr int kMaxStages = 16;
// Bytes of one page-list entry: (page, tokens | head mask), plus the source
// page to fetch in the window instantiations.
__host__ __device__ constexpr int attn_entry_bytes(bool win) { return win ? 16 : 8; }

}  // namespace kvs
