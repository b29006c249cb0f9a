"""GPU parity of the page window (kv_sparse_decode_attn_window) against the
fp64 oracle.

Bars: on identical selections and fp32 scores the window state after every
step (slot -> page and page -> slot maps, per-group stats) is bit-exact
against the oracle's replay of the policy; every cached slot holds exactly
the host page's valid tokens; the attention output is the sparse attention
over the selection (2e-3 for 16-bit inputs, 1e-5 for fp32).
"""
import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer, storage_to_torch, torch_to_bits
from parity_util import ATOL

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(kvlib):
    kv.kv_debug_config(-1, 2_000_000_000)
    kv.kv_device_status()
    yield


def _selections(spec, ctx, steps, K, seed, drift=0.35):
    """Seeded fp32 scores of a drifting query and their top-K selections."""
    rng = np.random.default_rng(seed)
    B, Hq, maxP, ps = spec.batch, spec.num_q_heads, spec.max_pages, spec.page_size
    base = rng.standard_normal((B, Hq, maxP))
    out = []
    for _ in range(steps):
        base = base + drift * rng.standard_normal(base.shape)
        s = np.round(base, 2).astype(np.float32)
        for b in range(B):
            s[b, :, -(-int(ctx[b]) // ps):] = -np.inf
        idx = oracle.topk(s.astype(np.float64), ctx, ps, K)
        out.append((idx, s))
    return out


def _check_slots(layer, wl):
    """Every cached slot holds the valid tokens of its host page, bit for bit."""
    spec = wl.spec
    ps, C = spec.page_size, layer.window.cache_pages
    sp = layer.win_slot_page.cpu().numpy()
    wk = torch_to_bits(layer.win_k)
    wv = torch_to_bits(layer.win_v)
    hk = wl.k_cache.view(wk.dtype)
    hv = wl.v_cache.view(wv.dtype)
    for b in range(spec.batch):
        L = int(wl.context_lens[b])
        for kvh in range(spec.num_kv_heads):
            for s in range(C):
                p = int(sp[b, kvh, s])
                if p < 0:
                    continue
                n = min(ps, L - p * ps)
                phys = wl.block_table[b, p]
                assert np.array_equal(wk[b * C + s, kvh, :n], hk[phys, kvh, :n]), (b, kvh, s, p)
                assert np.array_equal(wv[b * C + s, kvh, :n], hv[phys, kvh, :n]), (b, kvh, s, p)


@pytest.mark.parametrize("dtype,hq,hkv,ps,kv_loc,C", [
    ("bf16", 8, 2, 16, "host", 20),   # G = 4, tensor-core attention
    ("f16", 4, 2, 64, "host", 12),    # G = 2, CUDA-core attention, 64-token pages
    ("f32", 2, 2, 16, "host", 8),     # fp32, C = 2 G K
    ("bf16", 16, 2, 16, "hbm", 48),   # G = 8, window in front of HBM K/V
    ("bf16", 8, 2, 128, "host", 20),  # 128-token pages
    ("bf16", 32, 2, 16, "host", 80),  # G = 16: two head chunks fetch shared pages
    ("f32", 8, 1, 32, "host", 40),    # fp32, G = 8: two chunks of 4 heads, 32-token pages
])
def test_window_policy_and_output_match_oracle(dtype, hq, hkv, ps, kv_loc, C):
    K = 4
    spec = W.tiny_spec(dtype=dtype, batch=2, hq=hq, hkv=hkv, context=ps * 30 + 7, ps=ps,
                       index=110 + hq + ps)
    wl = W.generate(spec, context_lens=[ps * 30 + 7, ps * 17])
    layer = DecodeLayer(wl, kv_loc=kv_loc, topk=K)
    layer.enable_window(C)
    ow = oracle.Window(spec.batch, hkv, spec.max_pages, C)
    for step, (idx, s) in enumerate(_selections(spec, wl.context_lens, 8, K, seed=hq + ps)):
        layer.window_attn(indices=torch.from_numpy(idx).cuda(), scores=torch.from_numpy(s).cuda())
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        _, ost = ow.step(idx, s.astype(np.float64), wl.context_lens, ps)
        assert np.array_equal(layer.win_slot_page.cpu().numpy(), ow.slot_page), step
        assert np.array_equal(layer.win_page_slot.cpu().numpy(), ow.page_slot), step
        assert np.array_equal(layer.win_stats.cpu().numpy(), ost), step
        ref = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                               wl.context_lens, wl.scale, indices=idx)
        err = np.abs(layer.out.cpu().numpy() - ref).max()
        assert err <= ATOL[dtype], (step, err)
    _check_slots(layer, wl)


def test_window_refreshes_the_growing_last_page():
    # tokens appended to the host cache between steps reach the window: the
    # last page is fetched again whenever it is needed
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=8, hkv=2, context=16 * 12, ps=16, index=120)
    wl = W.generate(spec, context_lens=[16 * 5 + 3, 16 * 3])
    K = 3
    layer = DecodeLayer(wl, kv_loc="host", topk=K)
    layer.enable_window(2 * 4 * K)
    for step in range(12):
        kn, vn = W.new_tokens(spec, step)
        layer.append(storage_to_torch(kn, "bf16").cuda(), storage_to_torch(vn, "bf16").cuda(),
                     update_index=False)
        k2, v2, _, _ = oracle.append_token("bf16", kn, vn, wl.k_cache, wl.v_cache,
                                           wl.block_table, wl.context_lens)
        wl.k_cache, wl.v_cache = k2, v2
        wl.context_lens = wl.context_lens + 1
        # the oracle's selection with the last page forced in, and its scores
        mn, mx = oracle.minmax_build("bf16", wl.k_cache, wl.block_table, wl.context_lens)
        s = oracle.scores("bf16", wl.q, mn, mx, wl.block_table, wl.context_lens, 16)
        idx = oracle.topk_forced(s, wl.context_lens, 16, K, 0, 16)
        layer.window_attn(indices=torch.from_numpy(idx).cuda(),
                          scores=torch.from_numpy(s.astype(np.float32)).cuda())
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        ref = oracle.attention("bf16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                               wl.context_lens, wl.scale, indices=idx)
        assert np.abs(layer.out.cpu().numpy() - ref).max() <= ATOL["bf16"], step
    _check_slots(layer, wl)


def test_window_rejects_a_window_smaller_than_one_step():
    spec = W.tiny_spec(dtype="bf16", batch=1, hq=8, hkv=2, context=16 * 20, ps=16, index=121)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, kv_loc="host", topk=5)
    layer.enable_window(40)
    small = kv.make_window(19, layer.win_k, layer.win_v, layer.win_slot_page,
                           layer.win_page_slot)        # G * K = 20
    rc = kv.kv_sparse_decode_attn_window(layer.shape, layer.q, layer.k_cache, layer.v_cache,
                                         layer.block_table, layer.context_lens, layer.indices, 5,
                                         layer.scores, layer.scale, layer.out, small,
                                         layer.workspace, layer.workspace.numel(), check=False)
    assert rc == kv.KV_ERR_INVALID_ARG
    host_win = kv.make_window(40, layer.k_cache, layer.v_cache, layer.win_slot_page,
                              layer.win_page_slot)     # window arrays must be device memory
    rc = kv.kv_sparse_decode_attn_window(layer.shape, layer.q, layer.k_cache, layer.v_cache,
                                         layer.block_table, layer.context_lens, layer.indices, 5,
                                         layer.scores, layer.scale, layer.out, host_win,
                                         layer.workspace, layer.workspace.numel(), check=False)
    assert rc == kv.KV_ERR_LOCATION


def test_window_full_size_llama_128k_host_sampled():
    # the 128k-token host-resident Llama-3.1-8B layer, 6 decode steps of a
    # drifting query; every query head runs on the oracle's own selection
    # (the window's state still follows it), so the oracle sees no GPU output
    spec = W.WORKLOADS["llama3.1-8b-b1-ctx128k-host"]
    wl = W.generate(spec)
    K = spec.topk
    layer = DecodeLayer(wl, topk=K)
    layer.build_index()
    C = 2 * spec.group * K
    layer.enable_window(C)
    mn, mx = oracle.minmax_build("bf16", wl.k_cache, wl.block_table, wl.context_lens)
    qs = W.drifting_queries(spec, wl.q, 6, 0.3)
    hits = []
    for step, q in enumerate(qs):
        layer.q.copy_(storage_to_torch(q, "bf16").cuda())
        layer.score()
        layer.select()
        ref_s = oracle.scores("bf16", q, mn, mx, wl.block_table, wl.context_lens, 16)
        ref_idx = oracle.topk(ref_s, wl.context_lens, 16, K)
        sel = ref_idx.copy()                                 # every group: the oracle's
        layer.window_attn(indices=torch.from_numpy(sel).cuda())
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        rows = list(range(spec.num_q_heads))                 # every kv-head group
        ref = oracle.attention("bf16", q, wl.k_cache, wl.v_cache, wl.block_table,
                               wl.context_lens, wl.scale, indices=sel, rows=rows)
        out = layer.out.cpu().numpy()
        for r in rows:
            assert np.abs(out[0, r] - ref[0, r]).max() <= ATOL["bf16"], (step, r)
        st = layer.win_stats.cpu().numpy()
        need, hit, fetched = st[..., 0], st[..., 1], st[..., 2]
        assert (hit <= need).all()
        assert ((fetched >= need - hit) & (fetched <= need - hit + 1)).all()
        hits.append(hit.sum() / max(1, need.sum()))
    assert hits[0] == 0.0 and min(hits[1:]) > 0.0, hits     # the window is reused
