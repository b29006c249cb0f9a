"""GPU parity of kv_append_token against the fp64 oracle.

Bars: the K/V caches and the min/max table after an append are bit-exact
against the oracle's append (a byte copy, then the page's min/max recomputed
by its definition); the lengths advance by one; the path that follows (score,
top-K, sparse and dense attention) keeps the usual bars on the grown cache.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer, storage_to_torch, torch_to_bits
from parity_util import check_minmax, f64_to_bits
from test_gpu_parity import run_pipeline_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(kvlib):
    kv.kv_debug_config(-1, 2_000_000_000)
    kv.kv_device_status()
    yield


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint8)


def _gpu_append(layer, spec, step, advance=True):
    kn, vn = W.new_tokens(spec, step)
    layer.append(storage_to_torch(kn, spec.dtype).cuda(), storage_to_torch(vn, spec.dtype).cuda(),
                 advance=advance)
    return kn, vn


def _oracle_append(wl, kn, vn, mn=None, mx=None):
    k2, v2, mn2, mx2 = oracle.append_token(wl.spec.dtype, kn, vn, wl.k_cache, wl.v_cache,
                                           wl.block_table, wl.context_lens, mn, mx)
    lens = wl.context_lens.copy()
    ok = (lens >= 0) & (lens < wl.spec.max_pages * wl.spec.page_size)
    lens[ok] += 1
    return dataclasses.replace(wl, k_cache=k2, v_cache=v2, context_lens=lens), mn2, mx2


def _check_caches(layer, wl):
    assert np.array_equal(_bits(torch_to_bits(layer.k_cache)), _bits(wl.k_cache))
    assert np.array_equal(_bits(torch_to_bits(layer.v_cache)), _bits(wl.v_cache))
    assert np.array_equal(layer.context_lens.cpu().numpy(), wl.context_lens)


@pytest.mark.parametrize("dtype,ps,kv_loc", [
    ("bf16", 16, "hbm"), ("f16", 16, "hbm"), ("f32", 16, "hbm"),
    ("bf16", 64, "hbm"), ("f16", 64, "host"), ("bf16", 16, "host"),
    ("bf16", 32, "hbm"), ("f16", 128, "host"),
])
def test_one_append_matches_oracle(dtype, ps, kv_loc):
    # rows that open a new page (len % ps == 0), fill a page's last slot, and
    # land mid-page
    spec = W.tiny_spec(dtype=dtype, batch=4, hq=8, hkv=2, context=4 * ps, ps=ps, index=60)
    lens = [2 * ps, 3 * ps - 1, ps + 5, 1]
    wl = W.generate(spec, context_lens=lens)
    layer = DecodeLayer(wl, kv_loc=kv_loc, topk=2)
    layer.build_index()
    kn, vn = _gpu_append(layer, spec, 0)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    wl2, _, _ = _oracle_append(wl, kn, vn)
    _check_caches(layer, wl2)
    check_minmax(layer, wl2)


@pytest.mark.parametrize("dtype,ps,kv_loc", [("bf16", 16, "hbm"), ("f32", 64, "hbm"),
                                             ("bf16", 16, "host")])
def test_many_appends_then_the_decode_path(dtype, ps, kv_loc):
    # 40 decode steps of appends from ragged lengths (several pages opened and
    # filled), the table kept only by the incremental updates; then the whole
    # path on the grown cache against the oracle
    spec = W.tiny_spec(dtype=dtype, batch=3, hq=8, hkv=2, context=5 * ps, ps=ps, index=61)
    lens = [ps, 2 * ps + 3, 1]
    wl = W.generate(spec, context_lens=lens)
    layer = DecodeLayer(wl, kv_loc=kv_loc, topk=3)
    layer.build_index()
    steps = 40 if ps == 16 else 70
    for s in range(steps):
        kn, vn = _gpu_append(layer, spec, s)
        wl, _, _ = _oracle_append(wl, kn, vn)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    _check_caches(layer, wl)
    check_minmax(layer, wl)
    run_pipeline_and_check(wl, 3, kv_loc=kv_loc)


def test_append_without_advancing_keeps_the_lengths():
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=4, hkv=2, context=64, ps=16, index=62)
    wl = W.generate(spec, context_lens=[17, 40])
    layer = DecodeLayer(wl, topk=2)
    layer.build_index()
    kn, vn = _gpu_append(layer, spec, 1, advance=False)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    wl2, _, _ = _oracle_append(wl, kn, vn)
    assert np.array_equal(layer.context_lens.cpu().numpy(), wl.context_lens)
    assert np.array_equal(_bits(torch_to_bits(layer.k_cache)), _bits(wl2.k_cache))
    check_minmax(layer, wl2)


def test_append_without_index_leaves_the_table():
    spec = W.tiny_spec(dtype="f16", batch=2, hq=4, hkv=2, context=64, ps=16, index=64)
    wl = W.generate(spec, context_lens=[16, 29])
    layer = DecodeLayer(wl, topk=2)
    layer.build_index()
    before = layer.minmax_bits()
    kn, vn = W.new_tokens(spec, 2)
    layer.append(storage_to_torch(kn, "f16").cuda(), storage_to_torch(vn, "f16").cuda(),
                 update_index=False)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    wl2, _, _ = _oracle_append(wl, kn, vn)
    _check_caches(layer, wl2)
    assert np.array_equal(layer.minmax_bits(), before)


def test_out_of_range_row_is_flagged_and_skipped():
    spec = W.tiny_spec(dtype="f16", batch=3, hq=4, hkv=2, context=48, ps=16, index=63)
    wl = W.generate(spec, context_lens=[48, 20, 33])     # row 0 is full
    layer = DecodeLayer(wl, topk=2)
    layer.build_index()
    kn, vn = _gpu_append(layer, spec, 0)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_ERR_BOUNDS
    assert kv.kv_device_status() == kv.KV_OK               # the status word was cleared
    wl2, _, _ = _oracle_append(wl, kn, vn)
    assert wl2.context_lens[0] == 48
    _check_caches(layer, wl2)
    check_minmax(layer, wl2)


def test_append_at_full_size_llama_32k():
    # the 32k-token Llama-3.1-8B layer with one free slot per row, one row
    # opening a new page; caches and the touched index entries checked exactly
    spec = W.WORKLOADS["llama3.1-8b-b4-ctx32k"]
    T = spec.context
    lens = [T - 1, T - 16, T - 17, T - 1]
    wl = W.generate(spec, context_lens=lens)
    layer = DecodeLayer(wl, topk=spec.topk)
    layer.build_index()
    mm_before = layer.minmax_bits()
    kn, vn = _gpu_append(layer, spec, 0)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ps = spec.page_size
    mm = layer.minmax_bits()
    kc = torch_to_bits(layer.k_cache)
    vc = torch_to_bits(layer.v_cache)
    touched = set()
    for b, L in enumerate(lens):
        phys = int(wl.block_table[b, L // ps])
        touched.add(phys)
        t = L % ps
        assert np.array_equal(kc[phys, :, t], kn[b].view(kc.dtype))
        assert np.array_equal(vc[phys, :, t], vn[b].view(vc.dtype))
        page = wl.k_cache[phys].copy()
        page[:, t] = kn[b]
        for h in range(spec.num_kv_heads):
            mn, mx = oracle.page_minmax(spec.dtype, page[h], t + 1)
            assert np.array_equal(mm[phys, h, 0], f64_to_bits(mn, spec.dtype))
            assert np.array_equal(mm[phys, h, 1], f64_to_bits(mx, spec.dtype))
    others = np.array(sorted(set(range(spec.num_phys_pages)) - touched))
    assert np.array_equal(mm[others], mm_before[others])
    assert np.array_equal(layer.context_lens.cpu().numpy(), np.array(lens) + 1)
