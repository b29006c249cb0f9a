"""kv_decode_step (one decode step on host buffers) against the separate calls
and the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer, storage_to_torch
from parity_util import ATOL

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(kvlib):
    kv.kv_debug_config(-1, 2_000_000_000)
    kv.kv_device_status()
    yield


@pytest.mark.parametrize("dtype,sparse,kv_loc,pinned", [
    ("bf16", True, "hbm", True), ("f16", False, "hbm", True), ("bf16", True, "host", True),
    ("f32", False, "host", True),
    ("bf16", True, "hbm", False), ("f16", False, "hbm", False),   # pageable: copied
])
def test_host_step_equals_separate_calls_and_oracle(dtype, sparse, kv_loc, pinned):
    spec = W.tiny_spec(dtype=dtype, batch=3, hq=8, hkv=2, context=16 * 20 + 5, ps=16, topk=4,
                       index=130)
    wl = W.generate(spec, context_lens=[16 * 20 + 5, 16 * 7, 9])
    layer = DecodeLayer(wl, kv_loc=kv_loc, topk=4)
    layer.build_index()
    # a new step's query and lengths arrive in host memory
    q2 = W.drifting_queries(spec, wl.q, 1, 0.5)[0]
    ctx2 = np.array([16 * 20 + 5, 16 * 7 - 1, 9], dtype=np.int32)
    q_host = storage_to_torch(q2, dtype).clone()
    ctx_host = torch.from_numpy(ctx2).clone()
    out_host = torch.full(layer.out.shape, np.nan, dtype=torch.float32)
    if pinned:      # mapped: staged by one kernel into the device buffers, out in place
        q_host, ctx_host, out_host = q_host.pin_memory(), ctx_host.pin_memory(), out_host.pin_memory()
    layer.host_step(layer.host_io(q_host, ctx_host, out_host, sparse))
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    got = out_host.numpy().copy()
    # copied, or staged (a sparse step on mapped buffers): the device buffers
    # hold this step's inputs; a dense step on mapped buffers reads them in place
    if sparse or not pinned:
        assert torch.equal(layer.q.cpu(), q_host)
        assert torch.equal(layer.context_lens.cpu(), ctx_host)
    # the separate calls on the same inputs give the same bits
    layer.q.copy_(q_host)
    layer.context_lens.copy_(ctx_host)
    if sparse:
        layer.sparse_step()
    else:
        layer.dense_step()
    torch.cuda.synchronize()
    assert np.array_equal(layer.out.cpu().numpy(), got)
    # and the oracle agrees (sparse: on the oracle's own selection)
    if sparse:
        mn, mx = oracle.minmax_build(dtype, wl.k_cache, wl.block_table, wl.context_lens)
        s = oracle.scores(dtype, q2, mn, mx, wl.block_table, ctx2, 16)
        idx = oracle.topk(s, ctx2, 16, 4)
        layer.sparse_attn(indices=torch.from_numpy(idx).cuda())
        torch.cuda.synchronize()
        ref = oracle.attention(dtype, q2, wl.k_cache, wl.v_cache, wl.block_table, ctx2, wl.scale,
                               indices=idx)
        assert np.abs(layer.out.cpu().numpy() - ref).max() <= ATOL[dtype]
    else:
        ref = oracle.attention(dtype, q2, wl.k_cache, wl.v_cache, wl.block_table, ctx2, wl.scale)
        assert np.abs(got - ref).max() <= ATOL[dtype]


@pytest.mark.parametrize("sparse", [True, False])
def test_host_step_in_place_without_device_buffers(sparse):
    # mapped q and lengths with no device copies given: the kernels read them
    # in place across the host link; the same bits as the staged step
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=8, hkv=2, context=16 * 9 + 3, ps=16, topk=3,
                       index=132)
    wl = W.generate(spec, context_lens=[16 * 9 + 3, 16 * 4])
    layer = DecodeLayer(wl, topk=3)
    layer.build_index()
    q2 = W.drifting_queries(spec, wl.q, 1, 0.5)[0]
    q_host = storage_to_torch(q2, "bf16").clone().pin_memory()
    ctx_host = torch.from_numpy(wl.context_lens.astype(np.int32)).clone().pin_memory()
    outs = []
    for staged in (True, False):
        out_host = torch.full(layer.out.shape, np.nan, dtype=torch.float32).pin_memory()
        io = layer.host_io(q_host, ctx_host, out_host, sparse)
        if not staged:
            io.q = None
            io.context_lens = None
        layer.host_step(io)
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        outs.append(out_host.numpy().copy())
    assert not np.isnan(outs[1]).any()
    assert np.array_equal(outs[0], outs[1])


def test_host_step_rejects_missing_sparse_buffers():
    spec = W.tiny_spec(dtype="bf16", batch=1, hq=4, hkv=1, context=64, ps=16, index=131)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=2)
    q_host = layer.q.cpu().pin_memory()
    ctx_host = layer.context_lens.cpu().pin_memory()
    out_host = torch.empty(layer.out.shape, dtype=torch.float32).pin_memory()
    io = layer.host_io(q_host, ctx_host, out_host, True)
    io.minmax = None
    assert kv.kv_decode_step(layer.shape, io, check=False) == kv.KV_ERR_INVALID_ARG
    # without a scores buffer the step needs the selection's workspace
    io = layer.host_io(q_host, ctx_host, out_host, True)
    io.scores = None
    io.workspace_bytes = kv.kv_attn_workspace_bytes(layer.shape, 2)
    if io.workspace_bytes < kv.kv_select_workspace_bytes(layer.shape, 2):
        assert kv.kv_decode_step(layer.shape, io, check=False) == kv.KV_ERR_INVALID_ARG
    io.workspace_bytes = kv.kv_select_workspace_bytes(layer.shape, 2)
    assert kv.kv_decode_step(layer.shape, io, check=False) == kv.KV_OK
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK


@pytest.mark.parametrize("kv_loc", ["hbm", "host"])
def test_host_step_equal_chunks(kv_loc):
    # the step's attention with all groups' lists cut into equal chunks
    # (kv_debug_split_mode 1) against the per-group split (mode 0)
    ctx = [16 * 60 + 5, 16 * 44, 16 * 52 + 9]
    spec = W.tiny_spec(dtype="bf16", batch=3, hq=16, hkv=2, context=max(ctx), ps=16, topk=8,
                       index=131)
    wl = W.generate(spec, context_lens=ctx)
    layer = DecodeLayer(wl, kv_loc=kv_loc, topk=8)
    layer.build_index()
    q_host = layer.q.cpu().pin_memory()
    ctx_host = layer.context_lens.cpu().pin_memory()
    outs = {}
    try:
        for mode in (0, 1):
            kv.kv_debug_split_mode(mode)
            out_host = torch.full(layer.out.shape, np.nan, dtype=torch.float32).pin_memory()
            layer.host_step(layer.host_io(q_host, ctx_host, out_host, True))
            torch.cuda.synchronize()
            assert kv.kv_device_status() == kv.KV_OK
            outs[mode] = out_host.numpy().copy()
    finally:
        kv.kv_debug_split_mode(-1)
    assert np.isfinite(outs[1]).all()
    np.testing.assert_allclose(outs[1], outs[0], rtol=0, atol=1e-5)
