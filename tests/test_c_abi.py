"""The boundary is plain C: a C99 program includes the header, links the
library and calls the entry points that need no GPU (status strings, argument
checks, workspace sizes); on a GPU, a C99 program runs the whole path through
the header alone and gets the same bits as the Python binding."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "offloaded_kv_cache_gb300")


def build_dir(name):
    """A scratch directory in the package's (git-ignored) build tree."""
    d = os.path.join(LIBDIR, "_build", name)
    os.makedirs(d, exist_ok=True)
    return d


def compile_c(src_text, name, cflags=(), ldflags=(), std=("-std=c99", "-pedantic")):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    d = build_dir(name)
    src = os.path.join(d, name + ".c")
    with open(src, "w") as fh:
        fh.write(src_text)
    exe = os.path.join(d, name)
    subprocess.run([gcc, "-pipe", *std, "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), *cflags, src, "-o", exe,
                    "-L", LIBDIR, "-lkvsparse", "-Wl,-rpath," + LIBDIR, *ldflags], check=True)
    return exe, d

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "kvsparse.h"

int main(void) {
  kv_shape s;
  memset(&s, 0, sizeof s);
  s.batch = 2; s.num_q_heads = 8; s.num_kv_heads = 2; s.head_dim = 128; s.page_size = 16;
  s.max_pages_per_seq = 4; s.num_phys_pages = 8; s.dtype = KV_BF16; s.kv_loc = KV_LOC_HBM;
  int fails = 0;
  if (strcmp(kv_status_string(KV_ERR_BOUNDS), "KV_ERR_BOUNDS") != 0) ++fails;
  /* null outputs are refused before any device work */
  if (kv_page_minmax_build(&s, (void *)0x10000, (void *)0x10000, (void *)0x10000, NULL, NULL)
      != KV_ERR_INVALID_ARG) ++fails;
  if (kv_topk_select(&s, (const float *)0x10000, (const int32_t *)0x10000, 0,
                     (int32_t *)0x10000, NULL, 0, NULL) != KV_ERR_INVALID_ARG) ++fails;
  s.head_dim = 64;
  if (kv_dense_decode_attn(&s, NULL, NULL, NULL, NULL, NULL, 0.1f, NULL, NULL, 0, NULL)
      != KV_ERR_UNSUPPORTED) ++fails;
  if (kv_attn_workspace_bytes(&s, 0) != 0) ++fails;
  kv_window w;
  memset(&w, 0, sizeof w);
  if (kv_window_reset(&s, &w, NULL) == KV_OK) ++fails;
  kv_step_io io;
  memset(&io, 0, sizeof io);
  s.head_dim = 128;
  if (kv_decode_step(&s, &io, NULL) != KV_ERR_INVALID_ARG) ++fails;
  printf("%d %zu %zu %zu\n", fails, sizeof(kv_shape), sizeof(kv_window), sizeof(kv_step_io));
  return fails;
}
"""


def test_header_is_c99_and_the_library_links(kvlib):
    exe, _ = compile_c(C_PROGRAM, "abi")
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    fails, n_shape, n_window, n_io = (int(x) for x in out.stdout.split())
    assert fails == 0
    assert n_shape == 40 and n_window == 48 and n_io == 120


# The whole path from C: inputs from files, device buffers from the CUDA
# runtime, every step through kvsparse.h, outputs to files.
C_PATH_PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "kvsparse.h"

static void *load(const char *dir, const char *name, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  void *h = malloc(bytes);
  if (!f || !h || fread(h, 1, bytes, f) != bytes) { fprintf(stderr, "read %s\n", path); exit(2); }
  fclose(f);
  void *d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess ||
      cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) exit(3);
  free(h);
  return d;
}

static void save(const char *dir, const char *name, const void *d, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  void *h = malloc(bytes);
  if (!h || cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) exit(4);
  FILE *f = fopen(path, "wb");
  if (!f || fwrite(h, 1, bytes, f) != bytes) exit(5);
  fclose(f);
  free(h);
}

static void *dalloc(size_t bytes) {
  void *d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) exit(6);
  return d;
}

#define CHECK(call) do { int rc_ = (call); if (rc_ != KV_OK) { \
  fprintf(stderr, "%s: %s\n", #call, kv_status_string(rc_)); return 1; } } while (0)

int main(int argc, char **argv) {
  if (argc != 2) return 9;
  const char *dir = argv[1];
  int B, Hq, Hkv, ps, maxP, k;
  long long nphys;
  float scale;
  char p[1024];
  snprintf(p, sizeof p, "%s/shape.txt", dir);
  FILE *f = fopen(p, "r");
  if (!f || fscanf(f, "%d %d %d %d %d %lld %d %f", &B, &Hq, &Hkv, &ps, &maxP, &nphys, &k,
                   &scale) != 8) return 8;
  fclose(f);
  kv_shape s;
  memset(&s, 0, sizeof s);
  s.batch = B; s.num_q_heads = Hq; s.num_kv_heads = Hkv; s.head_dim = 128; s.page_size = ps;
  s.max_pages_per_seq = maxP; s.num_phys_pages = nphys; s.dtype = KV_BF16; s.kv_loc = KV_LOC_HBM;
  const size_t kv_bytes = (size_t)nphys * Hkv * ps * 128 * 2;
  void *q = load(dir, "q.bin", (size_t)B * Hq * 128 * 2);
  void *kc = load(dir, "k.bin", kv_bytes);
  void *vc = load(dir, "v.bin", kv_bytes);
  int32_t *bt = (int32_t *)load(dir, "bt.bin", (size_t)B * maxP * 4);
  int32_t *ctx = (int32_t *)load(dir, "ctx.bin", (size_t)B * 4);
  void *mm = dalloc((size_t)nphys * Hkv * 2 * 128 * 2);
  float *scores = (float *)dalloc((size_t)B * Hq * maxP * 4);
  int32_t *idx = (int32_t *)dalloc((size_t)B * Hq * k * 4);
  float *out = (float *)dalloc((size_t)B * Hq * 128 * 4);
  const size_t ws_t = kv_topk_workspace_bytes(&s, k);
  const size_t ws_s = kv_attn_workspace_bytes(&s, k);
  const size_t ws_d = kv_attn_workspace_bytes(&s, 0);
  size_t ws_max = ws_t > ws_s ? ws_t : ws_s;
  if (ws_d > ws_max) ws_max = ws_d;
  void *ws = dalloc(ws_max);
  CHECK(kv_page_minmax_build(&s, kc, bt, ctx, mm, NULL));
  CHECK(kv_page_score(&s, q, mm, bt, ctx, scores, NULL));
  CHECK(kv_topk_select(&s, scores, ctx, k, idx, ws, ws_max, NULL));
  CHECK(kv_sparse_decode_attn(&s, q, kc, vc, bt, ctx, idx, k, scale, out, ws, ws_max, NULL));
  CHECK(kv_device_status(NULL));
  save(dir, "minmax.out", mm, (size_t)nphys * Hkv * 2 * 128 * 2);
  save(dir, "scores.out", scores, (size_t)B * Hq * maxP * 4);
  save(dir, "indices.out", idx, (size_t)B * Hq * k * 4);
  save(dir, "sparse.out", out, (size_t)B * Hq * 128 * 4);
  CHECK(kv_dense_decode_attn(&s, q, kc, vc, bt, ctx, scale, out, ws, ws_max, NULL));
  CHECK(kv_device_status(NULL));
  save(dir, "dense.out", out, (size_t)B * Hq * 128 * 4);
  /* the one-call selection and the attention over its lists */
  const size_t ws_sel = kv_select_workspace_bytes(&s, k);
  void *ws2 = dalloc(ws_sel);
  int32_t *idx2 = (int32_t *)dalloc((size_t)B * Hq * k * 4);
  CHECK(kv_select_pages(&s, q, mm, bt, ctx, k, 0, 0, idx2, ws2, ws_sel, NULL));
  CHECK(kv_sparse_decode_attn_selected(&s, q, kc, vc, bt, ctx, k, scale, out, ws2, ws_sel,
                                       NULL));
  CHECK(kv_device_status(NULL));
  save(dir, "indices_sel.out", idx2, (size_t)B * Hq * k * 4);
  save(dir, "selected.out", out, (size_t)B * Hq * 128 * 4);
  printf("ok\n");
  return 0;
}
"""


@pytest.mark.gpu
def test_c_program_runs_the_path_and_matches_the_binding(kvlib):
    import torch

    import oracle
    from offloaded_kv_cache_gb300 import workloads as W
    from offloaded_kv_cache_gb300.pipeline import DecodeLayer, torch_to_bits
    from parity_util import ATOL

    cuda = "/usr/local/cuda"
    # the CUDA runtime's own headers need C11 (anonymous unions); kvsparse.h
    # alone is checked as strict C99 above
    exe, d = compile_c(C_PATH_PROGRAM, "path", cflags=("-I", os.path.join(cuda, "include")),
                       ldflags=("-L", os.path.join(cuda, "lib64"), "-lcudart",
                                "-Wl,-rpath," + os.path.join(cuda, "lib64")),
                       std=("-std=c11",))
    spec = W.tiny_spec(dtype="bf16", batch=3, hq=8, hkv=2, context=16 * 40 + 3, ps=16, topk=6,
                       index=140)
    wl = W.generate(spec, context_lens=[16 * 40 + 3, 16 * 11, 5])
    k = 6
    with open(os.path.join(d, "shape.txt"), "w") as fh:
        fh.write(f"{spec.batch} {spec.num_q_heads} {spec.num_kv_heads} {spec.page_size} "
                 f"{spec.max_pages} {spec.num_phys_pages} {k} {float(wl.scale)!r}\n")
    for name, arr in (("q", wl.q), ("k", wl.k_cache), ("v", wl.v_cache), ("bt", wl.block_table),
                      ("ctx", wl.context_lens.astype(np.int32))):
        np.ascontiguousarray(arr).tofile(os.path.join(d, name + ".bin"))
    out = subprocess.run([exe, d], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr

    # the same calls through the Python binding: the same bits
    layer = DecodeLayer(wl, topk=k)
    layer.build_index()
    layer.score()
    layer.select()
    layer.sparse_attn()
    torch.cuda.synchronize()
    sparse_py = layer.out.cpu().numpy().copy()
    layer.dense_step()
    torch.cuda.synchronize()
    dense_py = layer.out.cpu().numpy().copy()

    def rd(name, dtype):
        return np.fromfile(os.path.join(d, name), dtype=dtype)

    assert np.array_equal(rd("minmax.out", np.uint16), layer.minmax_bits().reshape(-1))
    assert np.array_equal(rd("scores.out", np.float32), layer.scores.cpu().numpy().reshape(-1))
    assert np.array_equal(rd("indices.out", np.int32), layer.indices.cpu().numpy().reshape(-1))
    assert np.array_equal(rd("sparse.out", np.float32), sparse_py.reshape(-1))
    assert np.array_equal(rd("dense.out", np.float32), dense_py.reshape(-1))
    # the one-call selection chose the same pages, and the attention over its
    # lists (each group's list over its own splits on this shape) gives the
    # same bits as the sparse call
    assert np.array_equal(rd("indices_sel.out", np.int32), layer.indices.cpu().numpy().reshape(-1))
    assert np.array_equal(rd("selected.out", np.float32), sparse_py.reshape(-1))
    # and the dense output against the oracle
    ref = oracle.attention("bf16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                           wl.context_lens, wl.scale)
    assert np.abs(rd("dense.out", np.float32).reshape(ref.shape) - ref).max() <= ATOL["bf16"]
