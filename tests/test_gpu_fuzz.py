"""Seeded random shapes through the whole path against the fp64 oracle.

Each case draws a dtype, batch, kv heads, GQA group size (odd ones too, so
that head chunking takes every form), page size, ragged per-row lengths, a
page budget K (sometimes beyond the row's pages) and the K/V location, then
checks the min/max index, the scores, the top-K selection, sparse and dense
attention (as in test_gpu_parity), the one-call selection and the attention
over its lists (both splits of the attention work), and in half of the cases
also the forced-page selection and two page-window steps.  Same bars as the parity
tests; the oracle never sees a GPU value.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import storage_to_torch
from parity_util import ATOL
from test_gpu_parity import run_pipeline_and_check

pytestmark = pytest.mark.gpu

N_CASES = int(os.environ.get("KVS_FUZZ_CASES", "64"))  # more for a longer stress run


def draw_case(i):
    rng = np.random.default_rng(20261202 + 7919 * i)
    dtype = ["f32", "f16", "bf16"][rng.integers(3)]
    hkv = int(rng.integers(1, 4))
    g = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16]))
    ps = int(rng.choice([16, 32, 64, 128]))
    batch = int(rng.integers(1, 5))
    max_pages = int(rng.integers(1, 41))
    ctx = [int(rng.integers(1, max_pages * ps + 1)) for _ in range(batch)]
    ctx[int(rng.integers(batch))] = max_pages * ps  # one full row
    k = int(rng.integers(1, 2 * max_pages + 2))
    kv_loc = "host" if rng.random() < 0.25 else "hbm"
    extras = bool(rng.random() < 0.5)
    return dict(dtype=dtype, hkv=hkv, hq=hkv * g, ps=ps, batch=batch, ctx=ctx, k=k,
                kv_loc=kv_loc, extras=extras, index=3000 + i)


@pytest.fixture(autouse=True)
def _lib(kvlib):
    kv.kv_debug_config(-1, 2_000_000_000)
    yield


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_through_the_path(i):
    c = draw_case(i)
    spec = W.tiny_spec(dtype=c["dtype"], batch=c["batch"], hq=c["hq"], hkv=c["hkv"],
                       context=max(c["ctx"]), ps=c["ps"], topk=c["k"], index=c["index"])
    wl = W.generate(spec, context_lens=c["ctx"])
    layer = run_pipeline_and_check(wl, c["k"], kv_loc=c["kv_loc"])
    ps, k, dtype = c["ps"], c["k"], c["dtype"]
    mn, mx = oracle.minmax_build(dtype, wl.k_cache, wl.block_table, wl.context_lens)
    s = oracle.scores(dtype, wl.q, mn, mx, wl.block_table, wl.context_lens, ps)

    # the one-call selection gives the separate calls' selection; the
    # attention over its lists, with each group's list over its own splits
    # and with equal chunks of all groups' lists where the shape allows, gives
    # the oracle's attention on every row whose selection is the oracle's
    sel_sep = layer.indices.cpu().numpy().copy()
    layer.select_fused()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    assert np.array_equal(layer.indices.cpu().numpy(), sel_sep)
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
    np.testing.assert_allclose(outs[1], outs[0], rtol=0, atol=1e-5)
    ref_idx = oracle.topk(s, wl.context_lens, ps, k)
    same = np.all(sel_sep == ref_idx, axis=-1)
    rows = [b * spec.num_q_heads + h for b in range(spec.batch) for h in range(spec.num_q_heads)
            if same[b, h]]
    if rows:
        ref_o = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                                 wl.context_lens, wl.scale, indices=ref_idx, rows=rows)
        got = outs[1].reshape(-1, spec.head_dim)[rows]
        err = np.abs(got - ref_o.reshape(-1, spec.head_dim)[rows]).max()
        assert err <= ATOL[dtype], err
    if not c["extras"]:
        return

    # forced pages: the oracle's own fp32 scores fed to the GPU selection
    s32 = s.astype(np.float32)
    layer.scores.copy_(torch.from_numpy(s32).cuda())
    layer.select(sink_tokens=4, local_tokens=64)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ref = oracle.topk_forced(s32.astype(np.float64), wl.context_lens, ps, k, 4, 64)
    assert np.array_equal(layer.indices.cpu().numpy(), ref)

    # two window steps on the oracle's selections of two queries
    C = min(spec.group * k, spec.max_pages) + 3
    layer.enable_window(C)
    ow = oracle.Window(spec.batch, spec.num_kv_heads, spec.max_pages, C)
    q2 = W.drifting_queries(spec, wl.q, 1, 0.5)[0]
    for q in (wl.q, q2):
        sq = oracle.scores(dtype, q, mn, mx, wl.block_table, wl.context_lens, ps)
        idx = oracle.topk(sq, wl.context_lens, ps, k)
        layer.q.copy_(storage_to_torch(q, dtype).cuda())
        layer.window_attn(indices=torch.from_numpy(idx).cuda(),
                          scores=torch.from_numpy(sq.astype(np.float32)).cuda())
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        ow.step(idx, sq.astype(np.float32).astype(np.float64), wl.context_lens, ps)
        assert np.array_equal(layer.win_slot_page.cpu().numpy(), ow.slot_page)
        ref_o = oracle.attention(dtype, q, wl.k_cache, wl.v_cache, wl.block_table,
                                 wl.context_lens, wl.scale, indices=idx)
        err = np.abs(layer.out.cpu().numpy() - ref_o).max()
        assert err <= ATOL[dtype], err
