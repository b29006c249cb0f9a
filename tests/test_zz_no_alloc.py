"""kv_dense_decode_attn_noalloc: dense decode attention without a workspace.

For callers that cannot allocate device memory (a plugin handed only its
inputs and outputs, a loop where cudaMalloc would synchronise the device), the
split-K partials live in a fixed scratch array inside the library.  This test
calls it through the C ABI and checks it against kv_dense_decode_attn with a
caller-allocated workspace, on two calls in a row, within the same tolerance
as the other attention tests, and both against the fp64 oracle; it also
checks the size limit.  It sits in a file of its own that runs last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer

pytestmark = pytest.mark.gpu

ATOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}
SCRATCH_BYTES = 1 << 20


def _noalloc_fn(lib):
    fn = lib.kv_dense_decode_attn_noalloc
    P = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(kv.kv_shape), P, P, P, P, P, ctypes.c_float, P, P]
    return fn


def _call(fn, layer, out, stream):
    return fn(ctypes.byref(layer.shape), layer.q.data_ptr(), layer.k_cache.data_ptr(),
              layer.v_cache.data_ptr(), layer.block_table.data_ptr(),
              layer.context_lens.data_ptr(), float(layer.scale), out.data_ptr(),
              stream.cuda_stream)


@pytest.mark.parametrize("dtype,hq,hkv,ctx", [("bf16", 8, 2, [16 * 300 + 5, 16 * 77]),
                                              ("f16", 4, 4, [16 * 120 + 3, 9]),
                                              ("f32", 2, 1, [16 * 250, 16 * 31 + 1])])
def test_noalloc_matches_workspace_call_twice(kvlib, dtype, hq, hkv, ctx):
    kv.kv_debug_config(-1, 2_000_000_000)
    kv.kv_device_status()
    fn = _noalloc_fn(kvlib)
    spec = W.tiny_spec(dtype=dtype, batch=len(ctx), hq=hq, hkv=hkv, context=max(ctx), ps=16,
                       topk=0, index=3000 + hq)
    wl = W.generate(spec, context_lens=ctx)
    layer = DecodeLayer(wl, topk=0)
    assert kv.kv_attn_num_splits(layer.shape, 0) > 1       # the scratch is really used
    assert 0 < layer.ws_dense_bytes <= SCRATCH_BYTES
    stream = torch.cuda.current_stream()
    layer.dense_step(stream)
    ref = layer.out.clone()
    exact = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                             wl.context_lens, wl.scale)
    assert np.abs(ref.cpu().numpy() - exact).max() <= ATOL[dtype]
    for _ in range(2):
        out = torch.full_like(layer.out, float("nan"))
        assert _call(fn, layer, out, stream) == kv.KV_OK
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        err = (out - ref).abs().max().item()
        assert err <= ATOL[dtype], err
        assert np.abs(out.cpu().numpy() - exact).max() <= ATOL[dtype]


def test_noalloc_refuses_shapes_beyond_its_scratch(kvlib):
    fn = _noalloc_fn(kvlib)
    shape = kv.make_shape(8, 64, 8, 128, 64, 1024, 8 * 1024, "bf16")
    need = kv.kv_attn_workspace_bytes(shape, 0)
    assert need > SCRATCH_BYTES
    fake = 0x10000
    rc = fn(ctypes.byref(shape), fake, fake, fake, fake, fake, 0.1, fake, None)
    assert rc == kv.KV_ERR_WORKSPACE
