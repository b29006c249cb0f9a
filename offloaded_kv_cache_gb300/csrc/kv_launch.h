// kv_launch.h -- host-side launcher declarations of the kvsparse kernels
// (each returns a cudaError_t).  Kept apart from kv_internal.cuh, which holds
// only what the kernels are compiled from.
#pragma once

#include <nvtx3/nvToolsExt.h>

#include "kv_internal.cuh"

namespace kvs {

// An NVTX range over one call of the C ABI, named after the call, so that a
// profiler's timeline shows which call each kernel launch belongs to.  With no
// profiler attached a range costs a few nanoseconds.
struct ApiRange {
  explicit ApiRange(const char *name) { nvtxRangePushA(name); }
  ~ApiRange() { nvtxRangePop(); }
  ApiRange(const ApiRange &) = delete;
  ApiRange &operator=(const ApiRange &) = delete;
};
#define KV_API_RANGE() ::kvs::ApiRange kv_api_range_(__func__)

cudaError_t launch_minmax_build(int dtype, const void *k, const int32_t *bt, const int32_t *ctx,
                                void *minmax, int B, int Hkv, int ps, int maxP, long long nphys,
                                int *status, cudaStream_t st);
cudaError_t launch_append(int dtype, const void *k_new, const void *v_new, void *k_cache,
                          void *v_cache, const int32_t *bt, const int32_t *ctx,
                          int32_t *ctx_out, void *minmax, int B, int Hkv, int ps, int maxP,
                          long long nphys, int *status, cudaStream_t st);
size_t window_update_smem(int maxP, int C);
// the window update and, beside it in the same launch, the union lists
cudaError_t launch_window_step(const int32_t *indices, const float *scores, const int32_t *ctx,
                               int B, int Hq, int Hkv, int ps, int maxP, int K, int C,
                               int32_t *slot_page, int32_t *page_slot, uint32_t *fetch_bits,
                               int32_t *stats, int gc, int umax, int32_t *upages,
                               uint32_t *umasks, int32_t *ucount, int *status, cudaStream_t st);
cudaError_t launch_fill(int32_t *p, long long n, int32_t v, cudaStream_t st);
// one decode step's q and context lengths, mapped host -> device buffers
cudaError_t launch_stage_inputs(const void *q_src, void *q_dst, size_t q_bytes,
                                const int32_t *ctx_src, int32_t *ctx_dst, int B,
                                cudaStream_t st);
// early_inputs: the previous kernel in the stream is one of the library's,
// so q and the block table may load before the PDL wait
cudaError_t launch_page_score(int dtype, bool mean, const void *q, const void *table,
                              const int32_t *bt, const int32_t *ctx, float *scores, int B, int Hq,
                              int Hkv, int ps, int maxP, long long nphys, int early_inputs,
                              int *status, cudaStream_t st);
cudaError_t launch_mean_build(int dtype, const void *k, const int32_t *bt, const int32_t *ctx,
                              void *mean, int B, int Hkv, int ps, int maxP, long long nphys,
                              bool last_only, int *status, cudaStream_t st);
cudaError_t launch_topk(const float *scores, const int32_t *ctx, int B, int Hq, int ps, int maxP,
                        int k, int sink_tokens, int local_tokens, int32_t *indices, int *status,
                        cudaStream_t st);
cudaError_t launch_union(const int32_t *indices, const int32_t *ctx, int B, int Hq, int Hkv,
                         int gc, int ps, int maxP, int k, int umax, int32_t *upages,
                         uint32_t *umasks, int32_t *ucount, int *status, cudaStream_t st);
cudaError_t launch_attn_core(int dtype, int gc, const AttnArgs &a, const CUtensorMap *tk,
                             const CUtensorMap *tv, dim3 grid, size_t smem, cudaStream_t st);
cudaError_t launch_attn_mma(int dtype, int gc, const AttnArgs &a, const CUtensorMap *tk,
                            const CUtensorMap *tv, dim3 grid, size_t smem, cudaStream_t st);
// the window instantiations: attention that also fetches the step's misses
cudaError_t launch_attn_win(int dtype, int gc, bool mma, const AttnArgs &a, const CUtensorMap *tk,
                            const CUtensorMap *tv, dim3 grid, size_t smem, cudaStream_t st);
// resident attention CTAs per SM for a launch shape (0 when unknown)
int attn_occupancy_core(int dtype, int gc, int threads, size_t smem);
int attn_occupancy_mma(int dtype, int gc, int threads, size_t smem);
int attn_occupancy_win(int dtype, int gc, bool mma, int threads, size_t smem);
// the fused selection: page score + top-K + group union in one cluster launch
// (16-bit data, G = 4 or 8 query heads per kv head)
int select_fused_pages_per_cta(int G, int maxP);
size_t select_fused_smem(int G, int maxP);
cudaError_t launch_select_fused(int dtype, const SelectArgs &a, int B, cudaStream_t st);
cudaError_t launch_combine(const float *part_o, const float *part_ml, float *out, int S, int B,
                           int Hq, cudaStream_t st);
// the combine after an attention over kv_select_pages' lists (AttnArgs::spread)
cudaError_t launch_combine_lists(const float *part_o, const float *part_ml, const float *spa_o,
                                 const float *spa_ml, const int32_t *gmeta, float *out, int S,
                                 int B, int Hq, int Hkv, int nw, int *status, cudaStream_t st);

}  // namespace kvs
