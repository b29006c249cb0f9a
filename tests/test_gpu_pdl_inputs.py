"""Inputs written by a kernel of another library that releases its dependents
early.

Every kernel of the library is launched with programmatic dependent launch.
A kernel of another library in the same stream may call
`griddepcontrol.launch_dependents` before it writes its outputs, expecting its
dependents to read them only after `griddepcontrol.wait`.  Here such a kernel
releases its dependents at entry and rewrites q (or the block table) about
30 us later; the call right after it must compute with the rewritten inputs.
The helper kernel is test code, compiled here with nvcc; its one wait is
bounded in time and in iterations.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer, storage_to_torch
from parity_util import ATOL, check_scores, score_tolerance

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

LATE_WRITER = r"""
#include <cuda_runtime.h>
#include <stdint.h>

// Releases its dependents at entry, waits delay_ns (bounded by an iteration
// count too), then copies src to dst.
__global__ void late_writer(uint4 *dst, const uint4 *src, size_t n16,
                            unsigned long long delay_ns) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int i = 0; i < 100000; ++i) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 >= delay_ns) break;
    __nanosleep(200);
  }
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

extern "C" int late_write(void *dst, const void *src, size_t bytes,
                          unsigned long long delay_ns, void *stream) {
  if (bytes % 16 || ((uintptr_t)dst & 15) || ((uintptr_t)src & 15)) return 1;
  late_writer<<<4, 128, 0, (cudaStream_t)stream>>>((uint4 *)dst, (const uint4 *)src,
                                                   bytes / 16, delay_ns);
  return (int)cudaGetLastError();
}
"""


@pytest.fixture(scope="module")
def late_write(kvlib):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    d = os.path.join(ROOT, "offloaded_kv_cache_gb300", "_build", "late_writer")
    os.makedirs(d, exist_ok=True)
    src = os.path.join(d, "late_writer.cu")
    with open(src, "w") as fh:
        fh.write(LATE_WRITER)
    so = os.path.join(d, "liblatewriter.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", "-o", so, src], check=True)
    lib = ctypes.CDLL(so)
    lib.late_write.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                               ctypes.c_ulonglong, ctypes.c_void_p]
    lib.late_write.restype = ctypes.c_int

    def call(dst: torch.Tensor, src: torch.Tensor, delay_ns=30_000):
        st = torch.cuda.current_stream()
        rc = lib.late_write(dst.data_ptr(), src.data_ptr(), dst.numel() * dst.element_size(),
                            delay_ns, st.cuda_stream)
        assert rc == 0
    return call


def _rewritten_q(wl, seed):
    """A second query of the workload's shape (the one the late writer stores)."""
    spec = wl.spec
    q2 = W._normal_storage(np.random.SeedSequence(seed), spec.batch * spec.num_q_heads * 128,
                           spec.value_scale, spec.dtype).reshape(wl.q.shape)
    return q2


@pytest.mark.parametrize("dtype,hq,hkv", [("f16", 4, 4), ("f32", 2, 1), ("bf16", 8, 2)])
def test_dense_reads_q_written_after_an_early_release(late_write, dtype, hq, hkv):
    # f16/f32 MHA run the CUDA-core attention, bf16 G=4 the tensor-core one
    spec = W.tiny_spec(dtype=dtype, batch=2, hq=hq, hkv=hkv, context=200, ps=16, topk=0,
                       index=4100 + hq)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=0)
    q2 = _rewritten_q(wl, 77)
    q2_dev = storage_to_torch(q2, dtype).cuda()
    for _ in range(3):
        layer.q.copy_(storage_to_torch(wl.q, dtype).cuda())
        late_write(layer.q, q2_dev)
        layer.dense_step()
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        ref = oracle.attention(dtype, q2, wl.k_cache, wl.v_cache, wl.block_table,
                               wl.context_lens, wl.scale)
        err = np.abs(layer.out.cpu().numpy() - ref).max()
        assert err <= ATOL[dtype], f"max-abs {err}: the kernel read q before it was written"


def test_dense_reads_block_table_written_after_an_early_release(late_write):
    # 16 pages a row: the table is a whole number of 16-byte chunks
    spec = W.tiny_spec(dtype="f16", batch=2, hq=4, hkv=4, context=250, ps=16, topk=0,
                       index=4200)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=0)
    # the rewritten table: each row's pages in reverse physical order
    bt2 = wl.block_table[:, ::-1].copy()
    bt2_dev = torch.from_numpy(bt2).cuda()
    for _ in range(3):
        layer.block_table.copy_(torch.from_numpy(wl.block_table).cuda())
        late_write(layer.block_table, bt2_dev)
        layer.dense_step()
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        ref = oracle.attention("f16", wl.q, wl.k_cache, wl.v_cache, bt2, wl.context_lens,
                               wl.scale)
        err = np.abs(layer.out.cpu().numpy() - ref).max()
        assert err <= ATOL["f16"], f"max-abs {err}: the kernel read the old block table"


@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 8, 2), ("f16", 4, 4)])
def test_page_score_reads_q_written_after_an_early_release(late_write, dtype, hq, hkv):
    # bf16 G=4: the tensor-core score kernel; f16 MHA: the CUDA-core one
    spec = W.tiny_spec(dtype=dtype, batch=2, hq=hq, hkv=hkv, context=600, ps=16, topk=4,
                       index=4300 + hq)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=4)
    layer.build_index()
    q2 = _rewritten_q(wl, 78)
    q2_dev = storage_to_torch(q2, dtype).cuda()
    mn, mx = oracle.minmax_build(dtype, wl.k_cache, wl.block_table, wl.context_lens)
    ref = oracle.scores(dtype, q2, mn, mx, wl.block_table, wl.context_lens, spec.page_size)
    tol = score_tolerance(dtype, q2, mn, mx, wl.block_table, wl.context_lens, spec.page_size)
    for _ in range(3):
        layer.q.copy_(storage_to_torch(wl.q, dtype).cuda())
        late_write(layer.q, q2_dev)
        layer.score()
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        check_scores(layer.scores.cpu().numpy(), ref, tol, wl.context_lens, spec.page_size)
