"""Full-size parity on the five workloads, in the launch configuration the
benchmark times, on outputs sampled per (sequence, head).

For each workload the GPU runs the whole path (index build, page scores,
top-K, sparse attention, dense attention, and the one-call selection with the
attention over its lists) over every row; the fp64 oracle then recomputes,
for the first and last sequence, their index entries (bit-exact), score rows
(fp32-accumulation bound), selections (boundary exemption) and, for every
query head of those sequences (every head chunk of every kv-head group), the
sparse attention over the oracle's own selection and the dense attention
(max-abs 2e-3 for 16-bit inputs, 1e-5 for fp32); the one-call path's output
is compared on the heads whose selection equals the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer

from parity_util import (ATOL, check_topk_with_exemption, f64_to_bits, referenced_pages,
                         score_tolerance)

pytestmark = pytest.mark.gpu


def sample_rows(spec):
    bs = sorted({0, spec.batch - 1})
    return bs, list(range(spec.num_q_heads))


@pytest.fixture(autouse=True)
def _lib(kvlib):
    kv.kv_debug_config(-1, 2_000_000_000)
    kv.kv_device_status()
    yield


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_full_workload_sampled(name):
    spec = W.WORKLOADS[name]
    dtype = spec.dtype
    k = max(1, spec.topk)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=k)
    layer.build_index()
    layer.score()
    layer.select()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    gpu_mm = layer.minmax_bits()
    gpu_scores = layer.scores.cpu().numpy()
    gpu_idx = layer.indices.cpu().numpy()

    bs, hs = sample_rows(spec)
    oracle_idx = {}
    for b in bs:
        sl = slice(b, b + 1)
        mn, mx = oracle.minmax_build(dtype, wl.k_cache, wl.block_table[sl], wl.context_lens[sl])
        pages = referenced_pages(wl, [b])
        assert np.array_equal(gpu_mm[pages, :, 0], f64_to_bits(mn[pages], dtype))
        assert np.array_equal(gpu_mm[pages, :, 1], f64_to_bits(mx[pages], dtype))
        s = oracle.scores(dtype, wl.q[sl], mn, mx, wl.block_table[sl], wl.context_lens[sl],
                          spec.page_size)
        tol = score_tolerance(dtype, wl.q[sl], mn, mx, wl.block_table[sl], wl.context_lens[sl],
                              spec.page_size)
        P = -(-int(wl.context_lens[b]) // spec.page_size)
        g = gpu_scores[b:b + 1, :, :P].astype(np.float64)
        assert (np.abs(g - s[:, :, :P]) <= tol[:, :, :P]).all()
        idx = oracle.topk(s, wl.context_lens[sl], spec.page_size, k)
        check_topk_with_exemption(gpu_idx[b:b + 1], idx, s, wl.context_lens[sl],
                                  spec.page_size, k)
        oracle_idx[b] = idx[0]

    # sparse attention over the oracle's selection for the sampled sequences
    sel = gpu_idx.copy()
    for b, idx in oracle_idx.items():
        sel[b] = idx
    layer.sparse_attn(indices=torch.from_numpy(sel).cuda())
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    sparse = layer.out.cpu().numpy()
    layer.dense_step()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    dense = layer.out.cpu().numpy()
    rows = [b * spec.num_q_heads + h for b in bs for h in hs]
    ref_s = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                             wl.context_lens, wl.scale, indices=sel, rows=rows)
    ref_d = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                             wl.context_lens, wl.scale, rows=rows)
    for b in bs:
        for h in hs:
            es = np.abs(sparse[b, h] - ref_s[b, h]).max()
            ed = np.abs(dense[b, h] - ref_d[b, h]).max()
            assert es <= ATOL[dtype], (name, b, h, "sparse", es)
            assert ed <= ATOL[dtype], (name, b, h, "dense", ed)

    # the one-call selection and the attention over its lists: its selection
    # is the separate calls' (bit for bit); its output on the sampled heads
    # whose selection is the oracle's
    if spec.topk:
        layer.select_fused()
        layer.sparse_attn_selected()
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        assert np.array_equal(layer.indices.cpu().numpy(), gpu_idx)
        fused = layer.out.cpu().numpy()
        same = 0
        for b in bs:
            for h in hs:
                if np.array_equal(gpu_idx[b, h], oracle_idx[b][h]):
                    same += 1
                    ef = np.abs(fused[b, h] - ref_s[b, h]).max()
                    assert ef <= ATOL[dtype], (name, b, h, "one-call", ef)
        assert same >= 0.9 * len(bs) * len(hs)
