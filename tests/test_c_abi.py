"""The boundary is plain C: a C99 program includes the header, links the
library and calls the entry points that need no GPU (status strings, argument
checks, workspace sizes)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

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


def test_header_is_c99_and_the_library_links(kvlib, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.join(ROOT, "offloaded_kv_cache_gb300")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lkvsparse", "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    fails, n_shape, n_window, n_io = (int(x) for x in out.stdout.split())
    assert fails == 0
    assert n_shape == 40 and n_window == 48 and n_io == 120
