// kv_attn_core.cu -- CUDA-core instantiations of the paged decode attention
// kernel: fp32 data, and 16-bit data whose GQA group is too small (1 or 2
// query heads per CTA) for a tokens x heads tile to be a real contraction.
#include "kv_attn.cuh"
#include "kv_launch.h"

namespace kvs {

cudaError_t launch_attn_core(int dtype, int gc, const AttnArgs &a, const CUtensorMap *tk,
                             const CUtensorMap *tv, dim3 grid, size_t smem, cudaStream_t st) {
  if (dtype == KV_F32) {
    if (gc == 4) return launch_attn_t<float, 4, false>(a, tk, tv, grid, smem, st);
    if (gc == 2) return launch_attn_t<float, 2, false>(a, tk, tv, grid, smem, st);
    return launch_attn_t<float, 1, false>(a, tk, tv, grid, smem, st);
  }
  if (dtype == KV_F16) {
    if (gc == 2) return launch_attn_t<__half, 2, false>(a, tk, tv, grid, smem, st);
    return launch_attn_t<__half, 1, false>(a, tk, tv, grid, smem, st);
  }
  if (gc == 2) return launch_attn_t<__nv_bfloat16, 2, false>(a, tk, tv, grid, smem, st);
  return launch_attn_t<__nv_bfloat16, 1, false>(a, tk, tv, grid, smem, st);
}

int attn_occupancy_core(int dtype, int gc, int threads, size_t smem) {
  if (dtype == KV_F32) {
    if (gc == 4) return attn_occupancy_t<float, 4, false>(threads, smem);
    if (gc == 2) return attn_occupancy_t<float, 2, false>(threads, smem);
    return attn_occupancy_t<float, 1, false>(threads, smem);
  }
  if (dtype == KV_F16) {
    if (gc == 2) return attn_occupancy_t<__half, 2, false>(threads, smem);
    return attn_occupancy_t<__half, 1, false>(threads, smem);
  }
  if (gc == 2) return attn_occupancy_t<__nv_bfloat16, 2, false>(threads, smem);
  return attn_occupancy_t<__nv_bfloat16, 1, false>(threads, smem);
}

}  // namespace kvs
