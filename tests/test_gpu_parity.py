"""GPU parity: every step of the path through the C ABI against the fp64 oracle.

Bars (element by element):
  * minmax tables: bit-exact (elements of K, totalOrder with -0.0 < +0.0);
  * page scores: |gpu - oracle| <= 1e-5 * sum_c |max(q_c mn_c, q_c mx_c)|
    (fp32 accumulation of 128 exact products);
  * top-K on identical fp32 scores: exact; top-K of the pipeline against the
    oracle's fp64 scores: the two sets differ only by equal numbers of
    boundary pages, |s - tau| < 1e-6 |tau| + 1e-30 with tau the oracle's
    K-th score;
  * attention outputs: max-abs error 2e-3 for f16/bf16 inputs, 1e-5 for fp32.
The oracle never sees a value produced by the GPU: sparse attention is run on
the oracle's own selection.
"""
import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer
from parity_util import (ATOL, check_minmax, check_scores, check_topk_with_exemption,
                         score_tolerance)

pytestmark = pytest.mark.gpu


def run_pipeline_and_check(wl, k, kv_loc=None, check_dense=True):
    spec = wl.spec
    dtype = spec.dtype
    layer = DecodeLayer(wl, kv_loc=kv_loc, topk=k)
    layer.build_index()
    layer.score()
    layer.select()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    mn, mx = check_minmax(layer, wl)
    ref_s = oracle.scores(dtype, wl.q, mn, mx, wl.block_table, wl.context_lens, spec.page_size)
    tol = score_tolerance(dtype, wl.q, mn, mx, wl.block_table, wl.context_lens, spec.page_size)
    check_scores(layer.scores.cpu().numpy(), ref_s, tol, wl.context_lens, spec.page_size)
    ref_idx = oracle.topk(ref_s, wl.context_lens, spec.page_size, k)
    check_topk_with_exemption(layer.indices.cpu().numpy(), ref_idx, ref_s, wl.context_lens,
                              spec.page_size, k)
    # sparse attention on the oracle's own selection
    layer.sparse_attn(indices=torch.from_numpy(ref_idx).cuda())
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ref_o = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                             wl.context_lens, wl.scale, indices=ref_idx)
    err = np.abs(layer.out.cpu().numpy() - ref_o).max()
    assert err <= ATOL[dtype], f"sparse max-abs {err}"
    if check_dense:
        layer.dense_step()
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        ref_d = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                                 wl.context_lens, wl.scale)
        err = np.abs(layer.out.cpu().numpy() - ref_d).max()
        assert err <= ATOL[dtype], f"dense max-abs {err}"
    return layer


@pytest.fixture(autouse=True)
def _lib(kvlib):
    kv.kv_debug_config(-1, 2_000_000_000)
    yield


# ---------------------------------------------------------------- small, many shapes

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 2), (6, 2), (8, 2), (16, 2), (24, 2), (32, 2)])
@pytest.mark.parametrize("ps", [16, 64])
def test_pipeline_small(dtype, hq, hkv, ps):
    # several pages per row, a ragged last page, rows of different lengths
    ctx = [5 * ps + 7, 2 * ps, 1] if ps == 16 else [3 * ps + 33, ps + 1, 17]
    spec = W.tiny_spec(dtype=dtype, batch=3, hq=hq, hkv=hkv, context=max(ctx), ps=ps, topk=3,
                       index=1000 + hq * 7 + hkv + ps)
    wl = W.generate(spec, context_lens=ctx)
    run_pipeline_and_check(wl, 3)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_pipeline_long_rows_many_splits(dtype):
    spec = W.tiny_spec(dtype=dtype, batch=2, hq=8, hkv=2, context=16 * 300 + 5, ps=16, topk=40,
                       index=2000)
    wl = W.generate(spec, context_lens=[16 * 300 + 5, 16 * 171 + 9])
    run_pipeline_and_check(wl, 40)


@pytest.mark.parametrize("k", [1, 2, 7, 64])
def test_topk_sizes_including_k_beyond_pages(k):
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=4, hkv=1, context=16 * 6, ps=16, topk=k,
                       index=2100 + k)
    wl = W.generate(spec, context_lens=[16 * 6, 16 * 2 + 3])
    run_pipeline_and_check(wl, k)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_large_logits_peaked_softmax(dtype):
    # q, K, V ~ N(0, 16^2): scaled logits of a few hundred, so the softmax is
    # dominated by a handful of tokens and every tile's and split's running
    # maximum moves by large amounts (rescale factors far below 2^-100)
    ctx = [16 * 300 + 5, 16 * 137 + 11]
    spec = W.tiny_spec(dtype=dtype, batch=2, hq=8, hkv=2, context=max(ctx), ps=16, topk=40,
                       scale=16.0, index=2900)
    wl = W.generate(spec, context_lens=ctx)
    run_pipeline_and_check(wl, 40)


def test_single_token_context_returns_its_value():
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=8, hkv=1, context=1, ps=16, topk=2, index=2200)
    wl = W.generate(spec)
    layer = run_pipeline_and_check(wl, 2)
    out = layer.out.cpu().numpy()
    for b in range(2):
        v = W.storage_to_f64(wl.v_cache[wl.block_table[b, 0], 0, 0], "bf16")
        assert np.abs(out[b] - v[None, :]).max() <= 1e-6


def test_identical_keys_give_mean_of_values():
    spec = W.tiny_spec(dtype="f16", batch=1, hq=8, hkv=2, context=16 * 9 + 3, ps=16, topk=4,
                       index=2300)
    wl = W.generate(spec)
    wl.k_cache[:] = wl.k_cache[0, 0, 0]
    run_pipeline_and_check(wl, 4)


def test_signed_zeros_in_keys_minmax_bits():
    spec = W.tiny_spec(dtype="bf16", batch=1, hq=2, hkv=1, context=48, ps=16, topk=1, index=2400)
    wl = W.generate(spec)
    phys = wl.block_table[0]
    k = wl.k_cache
    k[phys[0], 0, :, 0:4] = np.uint16(0x8000)      # all -0
    k[phys[0], 0, 3, 1] = np.uint16(0x0000)        # one +0 among -0
    k[phys[1], 0, :, 5] = np.uint16(0x0000)        # all +0
    k[phys[1], 0, 7, 5] = np.uint16(0x8000)        # one -0 among +0
    layer = DecodeLayer(wl, topk=1)
    layer.build_index()
    torch.cuda.synchronize()
    check_minmax(layer, wl)
    bits = layer.minmax_bits()
    assert bits[phys[0], 0, 0, 1] == 0x8000 and bits[phys[0], 0, 1, 1] == 0x0000
    assert bits[phys[1], 0, 0, 5] == 0x8000 and bits[phys[1], 0, 1, 5] == 0x0000


# ---------------------------------------------------------------- top-K on given scores

@pytest.mark.parametrize("P,K", [(7, 3), (256, 32), (1000, 999), (2048, 256), (8192, 512),
                                 (20000, 700), (33, 33), (5, 9)])
def test_topk_exact_on_identical_scores(P, K):
    rng = np.random.default_rng(P * 31 + K)
    B, Hq = 2, 3
    s = np.round(rng.standard_normal((B, Hq, P)), 1).astype(np.float32)  # heavy ties
    s[0, 0] = 0.0
    s[0, 1, ::2] = -0.0                                                 # +-0 rank equal
    s[1, 2, :] = rng.integers(0, 3, P).astype(np.float32)
    ctx = np.array([P * 16, max(1, (P // 2) * 16 - 5)], dtype=np.int32)
    shape = kv.make_shape(B, Hq, 1, 128, 16, P, B * P, "f32")
    scores = torch.from_numpy(s).cuda()
    ctx_d = torch.from_numpy(ctx).cuda()
    idx = torch.empty((B, Hq, K), dtype=torch.int32, device="cuda")
    kv.kv_topk_select(shape, scores, ctx_d, K, idx)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ref = oracle.topk(s.astype(np.float64), ctx, 16, K)
    assert np.array_equal(idx.cpu().numpy(), ref)


# ---------------------------------------------------------------- host-resident KV

@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 8, 2), ("f16", 2, 2), ("f32", 4, 4)])
def test_host_pinned_kv(dtype, hq, hkv):
    spec = W.tiny_spec(dtype=dtype, batch=2, hq=hq, hkv=hkv, context=16 * 40 + 3, ps=16,
                       topk=6, index=2500)
    wl = W.generate(spec, context_lens=[16 * 40 + 3, 16 * 9])
    layer = run_pipeline_and_check(wl, 6, kv_loc="host")
    assert not layer.k_cache.is_cuda and layer.k_cache.is_pinned()


def test_location_mismatch_is_rejected():
    spec = W.tiny_spec(dtype="bf16", batch=1, hq=2, hkv=1, context=32, ps=16, topk=1, index=2600)
    wl = W.generate(spec)
    dev = DecodeLayer(wl, kv_loc="hbm", topk=1)
    host = DecodeLayer(wl, kv_loc="host", topk=1)
    rc = kv.kv_dense_decode_attn(host.shape, dev.q, dev.k_cache, dev.v_cache, dev.block_table,
                                 dev.context_lens, 0.1, dev.out, dev.workspace,
                                 dev.workspace.numel(), check=False)
    assert rc == kv.KV_ERR_LOCATION
    rc = kv.kv_page_minmax_build(dev.shape, host.k_cache, dev.block_table, dev.context_lens,
                                 dev.minmax, check=False)
    assert rc == kv.KV_ERR_LOCATION
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    big = DecodeLayer(W.generate(W.tiny_spec(dtype="bf16", batch=1, hq=8, hkv=1, context=16 * 400,
                                             ps=16, topk=8, index=2601)), topk=8)
    if big.ws_dense_bytes > 16:
        rc = kv.kv_dense_decode_attn(big.shape, big.q, big.k_cache, big.v_cache, big.block_table,
                                     big.context_lens, 0.1, big.out, small, 16, check=False)
        assert rc == kv.KV_ERR_WORKSPACE


# ---------------------------------------------------------------- failure detection

def test_bounded_wait_times_out_and_context_survives():
    spec = W.tiny_spec(dtype="bf16", batch=1, hq=8, hkv=1, context=16 * 64, ps=16, topk=4,
                       index=2700)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=4)
    kv.kv_debug_config(0, 50_000_000)       # tile 0 of every CTA is never filled; 50 ms limit
    try:
        layer.dense_step()
        assert kv.kv_device_status() == kv.KV_ERR_DEVICE_TIMEOUT
    finally:
        kv.kv_debug_config(-1, 2_000_000_000)
    assert kv.kv_device_status() == kv.KV_OK  # cleared by the read
    layer.dense_step()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ref = oracle.attention("bf16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                           wl.context_lens, wl.scale)
    assert np.abs(layer.out.cpu().numpy() - ref).max() <= ATOL["bf16"]


def test_out_of_range_device_data_is_flagged_not_read():
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=4, hkv=1, context=16 * 5, ps=16, topk=2,
                       index=2800)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=2)
    bt = layer.block_table.clone()
    bt[0, 2] = spec.num_phys_pages + 1000          # physical page past the cache
    layer.block_table = bt
    layer.build_index()
    layer.dense_step()
    assert kv.kv_device_status() == kv.KV_ERR_BOUNDS
    bad_idx = torch.full_like(layer.indices, 1)
    bad_idx[1, 0, 0] = 99                          # selected page past the row's pages
    layer.block_table = torch.from_numpy(wl.block_table).cuda()
    layer.sparse_attn(indices=bad_idx)
    assert kv.kv_device_status() == kv.KV_ERR_BOUNDS
    ctx = layer.context_lens.clone()
    ctx[1] = 10_000                                # longer than the block table
    layer.context_lens = ctx
    layer.score()
    layer.select()
    assert kv.kv_device_status() == kv.KV_ERR_BOUNDS
    assert kv.kv_device_status() == kv.KV_OK


@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 8, 2), ("f16", 4, 1), ("f32", 2, 1)])
def test_block_table_entries_past_the_context_are_ignored(dtype, hq, hkv):
    # entries past each row's pages hold other rows' pages, pages past the
    # cache and negative values: none is used, none is an error
    spec = W.tiny_spec(dtype=dtype, batch=3, hq=hq, hkv=hkv, context=16 * 20, ps=16, topk=4,
                       index=2900 + hq)
    wl = W.generate(spec, context_lens=[16 * 20, 16 * 3 + 5, 1])
    rng = np.random.default_rng(2901)
    for b in range(spec.batch):
        P = -(-int(wl.context_lens[b]) // spec.page_size)
        n = spec.max_pages - P
        junk = rng.choice([0, 1, 2], size=n)
        wl.block_table[b, P:] = np.where(
            junk == 0, rng.integers(0, spec.num_phys_pages, size=n),
            np.where(junk == 1, spec.num_phys_pages + rng.integers(0, 1 << 20, size=n),
                     -rng.integers(1, 1 << 20, size=n))).astype(np.int32)
    run_pipeline_and_check(wl, 4)
    assert kv.kv_device_status() == kv.KV_OK


# ---------------------------------------------------------------- wide block table

@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 8, 2), ("f16", 4, 4)])
def test_sparse_attention_with_a_70000_page_block_table(dtype, hq, hkv):
    # Short contexts in a block table 70000 pages wide: the union's page map
    # and the top-K rows span the whole width, only the first pages are used.
    spec = W.tiny_spec(dtype=dtype, batch=2, hq=hq, hkv=hkv, context=16 * 40 + 3, ps=16,
                       index=140 + hq)
    wl = W.generate(spec, context_lens=[16 * 40 + 3, 16 * 13])
    wide = 70000
    bt = np.full((spec.batch, wide), -1, dtype=np.int32)
    bt[:, :spec.max_pages] = wl.block_table
    K = 5
    mn, mx = oracle.minmax_build(dtype, wl.k_cache, wl.block_table, wl.context_lens)
    s = oracle.scores(dtype, wl.q, mn, mx, wl.block_table, wl.context_lens, 16)
    idx = oracle.topk(s, wl.context_lens, 16, K)
    shape = kv.make_shape(spec.batch, hq, hkv, 128, 16, wide, spec.num_phys_pages, dtype)
    layer = DecodeLayer(wl, topk=K)
    out = torch.empty_like(layer.out)
    nbytes = kv.kv_attn_workspace_bytes(shape, K)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    kv.kv_sparse_decode_attn(shape, layer.q, layer.k_cache, layer.v_cache,
                             torch.from_numpy(bt).cuda(), layer.context_lens,
                             torch.from_numpy(idx).cuda(), K, wl.scale, out, ws, ws.numel())
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ref = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, bt, wl.context_lens, wl.scale,
                           indices=idx)
    assert np.abs(out.cpu().numpy() - ref).max() <= ATOL[dtype]


# ---------------------------------------------------------------- page sizes 32 and 128

@pytest.mark.parametrize("dtype,ps,kv_loc,hq,hkv", [
    ("bf16", 32, "hbm", 8, 2), ("f16", 128, "hbm", 16, 2), ("f32", 32, "hbm", 2, 1),
    ("bf16", 128, "host", 8, 2), ("f16", 32, "host", 4, 4),
])
def test_pages_of_32_and_128_tokens(dtype, ps, kv_loc, hq, hkv):
    # page sizes the tiered-offload guidance recommends for 70B-class models;
    # pages are whole 16-token tiles, ragged last pages included
    spec = W.tiny_spec(dtype=dtype, batch=3, hq=hq, hkv=hkv, context=ps * 9 + 5, ps=ps,
                       topk=3, index=150 + ps)
    wl = W.generate(spec, context_lens=[ps * 9 + 5, ps * 4, 17])
    run_pipeline_and_check(wl, 3, kv_loc=kv_loc)
