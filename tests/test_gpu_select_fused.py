"""The one-call selection (kv_select_pages) and the attention over its lists
(kv_sparse_decode_attn_selected).

For 16-bit data with 4 or 8 query heads per kv head the selection is one
cluster launch that keeps the scores on chip; other shapes run the separate
kernels.  Bars:
  * indices: bit-exact against kv_page_score + kv_topk_select(_forced) on the
    GPU (the same contraction and the same select), and against the oracle's
    top-K up to the boundary exemption of the parity rules;
  * attention: bit-exact against kv_sparse_decode_attn on the same indices
    (the same pages, head masks and split ranges), and within max-abs 2e-3
    (16-bit) / 1e-5 (fp32) of the oracle's attention on the oracle's own
    selection for every row whose selection equals the oracle's;
  * bad context lengths: flagged as KV_ERR_BOUNDS, selection -1, no page read.
"""
import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer
from parity_util import ATOL, check_topk_with_exemption

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(kvlib):
    kv.kv_debug_config(-1, 2_000_000_000)
    yield


def fused_vs_separate(wl, k, sink=0, local=0, kv_loc=None):
    """Runs both paths on one layer; returns (layer, fused idx, separate idx,
    fused out, separate out)."""
    layer = DecodeLayer(wl, topk=k, kv_loc=kv_loc)
    layer.build_index()
    layer.score()
    layer.select(sink_tokens=sink, local_tokens=local)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    idx_sep = layer.indices.cpu().numpy().copy()
    layer.sparse_attn()
    torch.cuda.synchronize()
    out_sep = layer.out.cpu().numpy().copy()
    layer.indices.fill_(-7)
    layer.out.fill_(float("nan"))
    layer.select_fused(sink_tokens=sink, local_tokens=local)
    layer.sparse_attn_selected()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    return layer, layer.indices.cpu().numpy(), idx_sep, layer.out.cpu().numpy(), out_sep


def check_against_oracle(wl, k, idx, out):
    spec = wl.spec
    dtype = spec.dtype
    mn, mx = oracle.minmax_build(dtype, wl.k_cache, wl.block_table, wl.context_lens)
    ref_s = oracle.scores(dtype, wl.q, mn, mx, wl.block_table, wl.context_lens, spec.page_size)
    ref_idx = oracle.topk(ref_s, wl.context_lens, spec.page_size, k)
    check_topk_with_exemption(idx, ref_idx, ref_s, wl.context_lens, spec.page_size, k)
    same = np.all(idx == ref_idx, axis=-1)          # [B][Hq]
    rows = [b * spec.num_q_heads + h for b in range(spec.batch)
            for h in range(spec.num_q_heads) if same[b, h]]
    assert len(rows) >= 0.9 * spec.batch * spec.num_q_heads
    ref_o = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                             wl.context_lens, wl.scale, indices=ref_idx, rows=rows)
    flat_o = out.reshape(-1, spec.head_dim)[rows]
    flat_r = ref_o.reshape(-1, spec.head_dim)[rows]
    err = np.abs(flat_o - flat_r).max()
    assert err <= ATOL[dtype], f"max-abs {err}"


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (16, 2), (4, 1), (8, 1)])
@pytest.mark.parametrize("ps", [16, 64])
def test_fused_selection_small(dtype, hq, hkv, ps):
    # several pages per row, a ragged last page, rows of different lengths
    ctx = [37 * ps + 5, 9 * ps, 3] if ps == 16 else [21 * ps + 33, 4 * ps + 1, 17]
    spec = W.tiny_spec(dtype=dtype, batch=3, hq=hq, hkv=hkv, context=max(ctx), ps=ps, topk=5,
                       index=5000 + hq * 3 + hkv + ps)
    wl = W.generate(spec, context_lens=ctx)
    _, idx, idx_sep, out, out_sep = fused_vs_separate(wl, 5)
    assert np.array_equal(idx, idx_sep)
    assert np.array_equal(out, out_sep)
    check_against_oracle(wl, 5, idx, out)


@pytest.mark.parametrize("k", [1, 7, 40, 400])
def test_fused_selection_budgets(k):
    # k from one page to more than a row holds (all pages, -1 padding)
    ctx = [300 * 16 + 9, 120 * 16, 40 * 16 + 1, 1]
    spec = W.tiny_spec(dtype="bf16", batch=4, hq=16, hkv=4, context=max(ctx), ps=16, topk=k,
                       index=5100 + k)
    wl = W.generate(spec, context_lens=ctx)
    _, idx, idx_sep, out, out_sep = fused_vs_separate(wl, k)
    assert np.array_equal(idx, idx_sep)
    assert np.array_equal(out, out_sep)
    check_against_oracle(wl, k, idx, out)


@pytest.mark.parametrize("maxp_pages", [1, 31, 33, 97, 600])
def test_fused_selection_page_counts(maxp_pages):
    # page counts around the 32-page words each CTA's share is cut into
    ctx = [maxp_pages * 16, max(1, maxp_pages * 16 - 23)]
    spec = W.tiny_spec(dtype="f16", batch=2, hq=8, hkv=1, context=max(ctx), ps=16, topk=6,
                       index=5200 + maxp_pages)
    wl = W.generate(spec, context_lens=ctx)
    _, idx, idx_sep, out, out_sep = fused_vs_separate(wl, 6)
    assert np.array_equal(idx, idx_sep)
    assert np.array_equal(out, out_sep)


@pytest.mark.parametrize("sink,local", [(4, 64), (0, 200), (100, 0), (10_000, 0)])
def test_fused_selection_forced_pages(sink, local):
    ctx = [150 * 16 + 3, 60 * 16]
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=8, hkv=2, context=max(ctx), ps=16, topk=12,
                       index=5300 + sink + local)
    wl = W.generate(spec, context_lens=ctx)
    _, idx, idx_sep, out, out_sep = fused_vs_separate(wl, 12, sink=sink, local=local)
    assert np.array_equal(idx, idx_sep)
    assert np.array_equal(out, out_sep)


@pytest.mark.parametrize("dtype,hq,hkv", [("f32", 4, 1), ("bf16", 4, 2), ("f16", 4, 4),
                                          ("bf16", 32, 2)])
def test_separate_kernels_behind_the_same_calls(dtype, hq, hkv):
    # shapes the cluster launch does not cover run score + top-K + union
    ctx = [45 * 16 + 2, 17]
    spec = W.tiny_spec(dtype=dtype, batch=2, hq=hq, hkv=hkv, context=max(ctx), ps=16, topk=6,
                       index=5400 + hq + hkv)
    wl = W.generate(spec, context_lens=ctx)
    layer, idx, idx_sep, out, out_sep = fused_vs_separate(wl, 6)
    assert layer.ws_select_bytes >= kv.kv_attn_workspace_bytes(layer.shape, 6)
    assert np.array_equal(idx, idx_sep)
    assert np.array_equal(out, out_sep)
    check_against_oracle(wl, 6, idx, out)


def test_fused_selection_host_resident_kv():
    ctx = [80 * 16 + 7, 33 * 16]
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=8, hkv=2, context=max(ctx), ps=16, topk=9,
                       index=5500)
    wl = W.generate(spec, context_lens=ctx)
    _, idx, idx_sep, out, out_sep = fused_vs_separate(wl, 9, kv_loc="host")
    assert np.array_equal(idx, idx_sep)
    assert np.array_equal(out, out_sep)
    check_against_oracle(wl, 9, idx, out)


def test_fused_selection_bad_length_is_flagged():
    spec = W.tiny_spec(dtype="bf16", batch=3, hq=8, hkv=2, context=200, ps=16, topk=4,
                       index=5600)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=4)
    layer.build_index()
    torch.cuda.synchronize()
    bad = layer.context_lens.clone()
    bad[1] = 0
    layer.context_lens.copy_(bad)
    layer.select_fused()
    layer.sparse_attn_selected()
    assert kv.kv_device_status() == kv.KV_ERR_BOUNDS
    idx = layer.indices.cpu().numpy()
    assert (idx[1] == -1).all()
    out = layer.out.cpu().numpy()
    assert (out[1] == 0).all()
    # the other rows are still right
    layer.context_lens.copy_(torch.from_numpy(wl.context_lens).cuda())
    layer.score()
    layer.select()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    sep = layer.indices.cpu().numpy()
    assert np.array_equal(idx[[0, 2]], sep[[0, 2]])


def test_selection_workspace_too_small_is_refused():
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=8, hkv=2, context=300, ps=16, topk=4,
                       index=5700)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=4)
    need = kv.kv_select_workspace_bytes(layer.shape, 4)
    rc = kv.kv_select_pages(layer.shape, layer.q, layer.minmax, layer.block_table,
                            layer.context_lens, 4, 0, 0, layer.indices, layer.workspace,
                            need - 1, check=False)
    assert rc == kv.KV_ERR_WORKSPACE


# ---------------------------------------------------------------------------
# the attention over the lists: each group's list split over its own CTAs, or
# all groups' lists cut into equal chunks (kv_debug_split_mode)
# ---------------------------------------------------------------------------

def union_sizes(idx, ctx, spec):
    G = spec.group
    U = []
    for b in range(spec.batch):
        P = -(-int(ctx[b]) // spec.page_size)
        for h in range(spec.num_kv_heads):
            sel = idx[b, h * G:(h + 1) * G].reshape(-1)
            U.append(len(np.unique(sel[(sel >= 0) & (sel < P)])))
    return U


def expect_equal_chunks(layer, idx, ctx, spec, k, adaptive=False):
    """Whether the kernel cuts the lists into equal chunks: every group
    (sequence, kv head) holds at least ceil(T / N) union pages, T their sum,
    N = splits x groups, T >= N; and, when it chooses (adaptive), the
    per-group split's longest CTA holds at least the K/V a CTA streams in
    2.5 us at 7 TB/s / N more than an equal chunk."""
    S = kv.kv_attn_num_splits(layer.shape, k)
    U = union_sizes(idx, ctx, spec)
    T, N = sum(U), S * len(U)
    ok = S > 1 and T >= N and min(U) * N >= T
    if ok and adaptive:
        page_bytes = 2 * spec.page_size * spec.head_dim * spec.elem_bytes
        gain = (-(-max(U) // S) - (-(-T // N))) * page_bytes
        ok = gain >= int(7.0e3 / N * 2500)
    return ok


def attn_in_both_modes(wl, k, kv_loc=None):
    layer = DecodeLayer(wl, topk=k, kv_loc=kv_loc)
    layer.build_index()
    layer.select_fused()
    torch.cuda.synchronize()
    outs = {}
    try:
        for mode in (0, 1):
            kv.kv_debug_split_mode(mode)
            layer.out.fill_(float("nan"))
            layer.sparse_attn_selected()
            torch.cuda.synchronize()
            assert kv.kv_device_status() == kv.KV_OK
            outs[mode] = layer.out.cpu().numpy().copy()
    finally:
        kv.kv_debug_split_mode(-1)
    return layer, layer.indices.cpu().numpy(), outs


@pytest.mark.parametrize("dtype,hq,hkv,ps,batch,ctx,k", [
    ("bf16", 16, 2, 64, 3, [300 * 64 + 17, 120 * 64, 41 * 64 + 63], 24),
    ("f16", 8, 2, 16, 4, [900 * 16 + 3, 700 * 16, 650 * 16 + 9, 999 * 16], 40),
    ("bf16", 32, 4, 16, 2, [2000 * 16, 1500 * 16 + 5], 64),
    ("bf16", 8, 1, 64, 5, [90 * 64, 80 * 64 + 1, 200 * 64, 33 * 64, 150 * 64 + 40], 10),
    # one row far shorter than the others: its groups hold fewer pages than
    # a chunk, so the kernel keeps the split per group
    ("bf16", 8, 2, 16, 3, [1200 * 16, 1100 * 16, 5], 30),
])
def test_equal_chunks_match_per_group_split(dtype, hq, hkv, ps, batch, ctx, k):
    if hq // hkv not in (4, 8):
        pytest.skip("the one-call selection covers 4 or 8 heads per kv head")
    spec = W.tiny_spec(dtype=dtype, batch=batch, hq=hq, hkv=hkv, context=max(ctx), ps=ps, topk=k,
                       index=5800 + hq + hkv + ps + batch)
    wl = W.generate(spec, context_lens=ctx)
    layer, idx, outs = attn_in_both_modes(wl, k)
    assert np.isfinite(outs[1]).all()
    if expect_equal_chunks(layer, idx, wl.context_lens, spec, k):
        # the same softmax merged in another order
        np.testing.assert_allclose(outs[1], outs[0], rtol=0, atol=1e-5)
        assert not np.array_equal(outs[1], outs[0])
    else:
        # the list combine merges the per-group splits in combine_kernel's order
        assert np.array_equal(outs[1], outs[0])
    check_against_oracle(wl, k, idx, outs[1])


def test_equal_chunks_many_groups():
    # 24 sequences x 8 kv heads = 192 groups, more than a CTA's 160 threads:
    # each thread sums the lengths of two groups in the prefix scan
    rng = np.random.default_rng(77)
    ctx = [int(x) for x in rng.integers(60 * 16, 200 * 16, size=24)]
    spec = W.tiny_spec(dtype="bf16", batch=24, hq=32, hkv=8, context=max(ctx), ps=16, topk=16,
                       index=5990)
    wl = W.generate(spec, context_lens=ctx)
    layer, idx, outs = attn_in_both_modes(wl, 16)
    assert expect_equal_chunks(layer, idx, wl.context_lens, spec, 16)
    np.testing.assert_allclose(outs[1], outs[0], rtol=0, atol=1e-5)
    assert not np.array_equal(outs[1], outs[0])
    check_against_oracle(wl, 16, idx, outs[1])


def test_equal_chunks_cover_both_decisions():
    # the parametrization above reaches both branches
    seen = set()
    for ctx, k in [([1200 * 16, 1100 * 16, 5], 30), ([900 * 16, 700 * 16, 650 * 16], 40)]:
        spec = W.tiny_spec(dtype="bf16", batch=len(ctx), hq=8, hkv=2, context=max(ctx), ps=16,
                           topk=k, index=5900 + k)
        wl = W.generate(spec, context_lens=ctx)
        layer = DecodeLayer(wl, topk=k)
        layer.build_index()
        layer.select_fused()
        torch.cuda.synchronize()
        seen.add(expect_equal_chunks(layer, layer.indices.cpu().numpy(), wl.context_lens, spec, k))
    assert seen == {True, False}


def test_equal_chunks_host_resident_kv():
    ctx = [700 * 16 + 7, 500 * 16, 640 * 16]
    spec = W.tiny_spec(dtype="bf16", batch=3, hq=8, hkv=2, context=max(ctx), ps=16, topk=32,
                       index=5950)
    wl = W.generate(spec, context_lens=ctx)
    layer, idx, outs = attn_in_both_modes(wl, 32, kv_loc="host")
    assert expect_equal_chunks(layer, idx, wl.context_lens, spec, 32)
    np.testing.assert_allclose(outs[1], outs[0], rtol=0, atol=1e-5)
    check_against_oracle(wl, 32, idx, outs[1])


@pytest.mark.parametrize("hq,hkv,ps,k,ctx", [
    # rows of very different lengths: the long rows' groups hold far more
    # pages, so the kernel takes equal chunks
    (16, 2, 64, 64, [600 * 64, 75 * 64 + 3, 600 * 64 - 1, 80 * 64]),
    (8, 2, 16, 256, [2400 * 16, 100 * 16 + 3, 2400 * 16 - 1, 110 * 16]),
    # equal lengths: the groups differ by a few pages, so it keeps the split
    # per group (bit for bit the per-group result)
    (8, 2, 16, 256, [2400 * 16, 2400 * 16, 2400 * 16, 2400 * 16]),
])
def test_kernel_chooses_the_split(hq, hkv, ps, k, ctx):
    spec = W.tiny_spec(dtype="bf16", batch=len(ctx), hq=hq, hkv=hkv, context=max(ctx), ps=ps,
                       topk=k, index=6000 + hq + ps + ctx[1])
    wl = W.generate(spec, context_lens=ctx)
    layer = DecodeLayer(wl, topk=k)
    layer.build_index()
    layer.select_fused()
    torch.cuda.synchronize()
    outs = {}
    try:
        for mode in (0, 2):
            kv.kv_debug_split_mode(mode)
            layer.out.fill_(float("nan"))
            layer.sparse_attn_selected()
            torch.cuda.synchronize()
            assert kv.kv_device_status() == kv.KV_OK
            outs[mode] = layer.out.cpu().numpy().copy()
    finally:
        kv.kv_debug_split_mode(-1)
    idx = layer.indices.cpu().numpy()
    chunks = expect_equal_chunks(layer, idx, wl.context_lens, spec, k, adaptive=True)
    assert chunks == (ctx[0] != ctx[1])
    if chunks:
        np.testing.assert_allclose(outs[2], outs[0], rtol=0, atol=1e-5)
        assert not np.array_equal(outs[2], outs[0])
    else:
        assert np.array_equal(outs[2], outs[0])
    check_against_oracle(wl, k, idx, outs[2])


def test_equal_chunks_bad_length_keeps_the_per_group_split():
    # a row whose length is out of range has an empty list, so no group is a
    # chunk long: the kernel keeps the split per group, flags the length and
    # writes zeros for that row; the other rows are the per-group results
    ctx = [300 * 16 + 5, 250 * 16, 280 * 16 + 9]
    spec = W.tiny_spec(dtype="bf16", batch=3, hq=8, hkv=2, context=max(ctx), ps=16, topk=24,
                       index=6100)
    wl = W.generate(spec, context_lens=ctx)
    layer = DecodeLayer(wl, topk=24)
    layer.build_index()
    layer.select_fused()
    kv.kv_debug_split_mode(0)
    try:
        layer.sparse_attn_selected()
        torch.cuda.synchronize()
        good = layer.out.cpu().numpy().copy()
        assert kv.kv_device_status() == kv.KV_OK
        bad = layer.context_lens.clone()
        bad[1] = 0
        layer.context_lens.copy_(bad)
        kv.kv_debug_split_mode(1)
        layer.out.fill_(float("nan"))
        layer.sparse_attn_selected()
        torch.cuda.synchronize()
    finally:
        kv.kv_debug_split_mode(-1)
    assert kv.kv_device_status() == kv.KV_ERR_BOUNDS
    out = layer.out.cpu().numpy()
    assert (out[1] == 0).all()
    assert np.array_equal(out[[0, 2]], good[[0, 2]])


def test_equal_chunks_bounded_wait_times_out_and_context_survives():
    # a tile no producer fills (testing hook): the waits give up after 50 ms,
    # the call's kernels finish, the status says so, and the next call is right
    ctx = [400 * 16, 380 * 16 + 7]
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=8, hkv=2, context=max(ctx), ps=16, topk=32,
                       index=6200)
    wl = W.generate(spec, context_lens=ctx)
    layer, idx, outs = attn_in_both_modes(wl, 32)
    assert expect_equal_chunks(layer, idx, wl.context_lens, spec, 32)
    kv.kv_debug_split_mode(1)
    kv.kv_debug_config(3, 50_000_000)
    try:
        layer.sparse_attn_selected()
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_ERR_DEVICE_TIMEOUT
        kv.kv_debug_config(-1, 2_000_000_000)
        layer.out.fill_(float("nan"))
        layer.sparse_attn_selected()
        torch.cuda.synchronize()
    finally:
        kv.kv_debug_config(-1, 2_000_000_000)
        kv.kv_debug_split_mode(-1)
    assert kv.kv_device_status() == kv.KV_OK
    assert np.array_equal(layer.out.cpu().numpy(), outs[1])


def test_split_mode_hook_refuses_bad_modes():
    for m in (-2, 3, 7):
        assert kv.kv_debug_split_mode(m, check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_debug_split_mode(-1) == kv.KV_OK


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama3.1-8b-b4-ctx32k", "70b-gqa-b8-ctx64k-ps64",
                                  "llama3.1-8b-b1-ctx128k-host"])
def test_fused_selection_full_size(name):
    spec = W.WORKLOADS[name]
    wl = W.generate(spec)
    kv.kv_debug_split_mode(0)
    try:
        layer, idx, idx_sep, out, out_sep = fused_vs_separate(wl, spec.topk)
    finally:
        kv.kv_debug_split_mode(-1)
    assert np.array_equal(idx, idx_sep)
    assert np.array_equal(out, out_sep)
    # the plan's own choice, and equal chunks forced, against the per-group split
    for mode in (-1, 1):
        kv.kv_debug_split_mode(mode)
        try:
            layer.out.fill_(float("nan"))
            layer.sparse_attn_selected()
            torch.cuda.synchronize()
        finally:
            kv.kv_debug_split_mode(-1)
        assert kv.kv_device_status() == kv.KV_OK
        np.testing.assert_allclose(layer.out.cpu().numpy(), out_sep, rtol=0, atol=1e-5)
