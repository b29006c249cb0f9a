// kv_attn_mma.cu -- tensor-core instantiations of the paged decode attention
// kernel: 16-bit data with 4 or 8 query heads per CTA, where q . K^T over a
// 16-token tile and V^T . P^T are dense tokens x heads contractions.
#include "kv_attn.cuh"
#include "kv_launch.h"

namespace kvs {

cudaError_t launch_attn_mma(int dtype, int gc, const AttnArgs &a, const CUtensorMap *tk,
                            const CUtensorMap *tv, dim3 grid, size_t smem, cudaStream_t st) {
  if (dtype == KV_F16) {
    if (gc == 8) return launch_attn_t<__half, 8, true>(a, tk, tv, grid, smem, st);
    return launch_attn_t<__half, 4, true>(a, tk, tv, grid, smem, st);
  }
  if (gc == 8) return launch_attn_t<__nv_bfloat16, 8, true>(a, tk, tv, grid, smem, st);
  return launch_attn_t<__nv_bfloat16, 4, true>(a, tk, tv, grid, smem, st);
}

int attn_occupancy_mma(int dtype, int gc, int threads, size_t smem) {
  if (dtype == KV_F16) {
    if (gc == 8) return attn_occupancy_t<__half, 8, true>(threads, smem);
    return attn_occupancy_t<__half, 4, true>(threads, smem);
  }
  if (gc == 8) return attn_occupancy_t<__nv_bfloat16, 8, true>(threads, smem);
  return attn_occupancy_t<__nv_bfloat16, 4, true>(threads, smem);
}

}  // namespace kvs
