// kv_attn_win.cu -- the page-window instantiations of the paged decode
// attention kernel: K/V come from the GPU-resident window, except the pages
// this step fetches, which the kernel reads from the source cache and stores
// into their window slots as it goes.  Same head chunking as the plain
// instantiations: tensor cores for 16-bit data with 4 or 8 heads per CTA,
// CUDA cores otherwise.
#include "kv_attn.cuh"
#include "kv_launch.h"

namespace kvs {

cudaError_t launch_attn_win(int dtype, int gc, bool mma, const AttnArgs &a, const CUtensorMap *tk,
                            const CUtensorMap *tv, dim3 grid, size_t smem, cudaStream_t st) {
  if (dtype == KV_F32) {
    if (gc == 4) return launch_attn_t<float, 4, false, true>(a, tk, tv, grid, smem, st);
    if (gc == 2) return launch_attn_t<float, 2, false, true>(a, tk, tv, grid, smem, st);
    return launch_attn_t<float, 1, false, true>(a, tk, tv, grid, smem, st);
  }
  if (dtype == KV_F16) {
    if (mma) {
      if (gc == 8) return launch_attn_t<__half, 8, true, true>(a, tk, tv, grid, smem, st);
      return launch_attn_t<__half, 4, true, true>(a, tk, tv, grid, smem, st);
    }
    if (gc == 2) return launch_attn_t<__half, 2, false, true>(a, tk, tv, grid, smem, st);
    return launch_attn_t<__half, 1, false, true>(a, tk, tv, grid, smem, st);
  }
  if (mma) {
    if (gc == 8) return launch_attn_t<__nv_bfloat16, 8, true, true>(a, tk, tv, grid, smem, st);
    return launch_attn_t<__nv_bfloat16, 4, true, true>(a, tk, tv, grid, smem, st);
  }
  if (gc == 2) return launch_attn_t<__nv_bfloat16, 2, false, true>(a, tk, tv, grid, smem, st);
  return launch_attn_t<__nv_bfloat16, 1, false, true>(a, tk, tv, grid, smem, st);
}

int attn_occupancy_win(int dtype, int gc, bool mma, int threads, size_t smem) {
  if (dtype == KV_F32) {
    if (gc == 4) return attn_occupancy_t<float, 4, false, true>(threads, smem);
    if (gc == 2) return attn_occupancy_t<float, 2, false, true>(threads, smem);
    return attn_occupancy_t<float, 1, false, true>(threads, smem);
  }
  if (dtype == KV_F16) {
    if (mma) {
      if (gc == 8) return attn_occupancy_t<__half, 8, true, true>(threads, smem);
      return attn_occupancy_t<__half, 4, true, true>(threads, smem);
    }
    if (gc == 2) return attn_occupancy_t<__half, 2, false, true>(threads, smem);
    return attn_occupancy_t<__half, 1, false, true>(threads, smem);
  }
  if (mma) {
    if (gc == 8) return attn_occupancy_t<__nv_bfloat16, 8, true, true>(threads, smem);
    return attn_occupancy_t<__nv_bfloat16, 4, true, true>(threads, smem);
  }
  if (gc == 2) return attn_occupancy_t<__nv_bfloat16, 2, false, true>(threads, smem);
  return attn_occupancy_t<__nv_bfloat16, 1, false, true>(threads, smem);
}

}  // namespace kvs
