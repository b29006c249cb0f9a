"""GPU parity of kv_topk_select_forced (sink and local pages forced into the
selection) against the fp64 oracle.

On identical fp32 scores the selection is exact.  Through the pipeline the
forced pages must match exactly and the rest may differ only by boundary pages
(the usual top-K exemption, taken on the oracle's scores with the forced
pages at +inf); sparse attention over the oracle's selection keeps its bar.
"""
import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer
from parity_util import ATOL, check_minmax, check_topk_with_exemption

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(kvlib):
    kv.kv_debug_config(-1, 2_000_000_000)
    kv.kv_device_status()
    yield


def _forced_mask(P, L, ps, sink, local):
    lo = np.arange(P) * ps
    hi = np.minimum(L, lo + ps)
    return ((sink > 0) & (lo < sink)) | ((local > 0) & (hi > L - local))


def _gpu_forced(s, ctx, ps, K, sink, local):
    B, Hq, P = s.shape
    shape = kv.make_shape(B, Hq, 1, 128, ps, P, B * P, "f32")
    idx = torch.empty((B, Hq, K), dtype=torch.int32, device="cuda")
    kv.kv_topk_select_forced(shape, torch.from_numpy(s).cuda(), torch.from_numpy(ctx).cuda(), K,
                             sink, local, idx)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    return idx.cpu().numpy()


@pytest.mark.parametrize("P,ps,K,sink,local", [
    (40, 16, 8, 4, 64),      # 1 sink page + 4-5 local pages, 3 free slots
    (40, 16, 3, 4, 64),      # more forced than k: lowest-index forced pages
    (40, 16, 40, 4, 64),     # every page
    (33, 64, 5, 4, 64),      # 64-token pages: the local window is 1-2 pages
    (300, 16, 17, 16, 1),    # sink exactly one page, local = the last token's page
    (2048, 16, 261, 4, 64),  # Llama-3.1-8B 32k shape with k = 256 + 5 forced
    (12000, 16, 300, 4, 64),  # keys beyond the shared-memory cache
])
def test_forced_selection_exact_on_identical_scores(P, ps, K, sink, local):
    rng = np.random.default_rng(P + 7 * K + sink)
    B, Hq = 2, 3
    s = np.round(rng.standard_normal((B, Hq, P)), 1).astype(np.float32)   # heavy ties
    s[1, 1] = 0.0
    ctx = np.array([P * ps, max(1, (P // 2) * ps - 5)], dtype=np.int32)
    for b in range(B):
        s[b, :, -(-int(ctx[b]) // ps):] = -np.inf
    got = _gpu_forced(s, ctx, ps, K, sink, local)
    ref = oracle.topk_forced(s.astype(np.float64), ctx, ps, K, sink, local)
    assert np.array_equal(got, ref)
    # the forced pages are all in (or the selection is all forced pages)
    for b in range(B):
        L = int(ctx[b])
        Pb = -(-L // ps)
        forced = np.flatnonzero(_forced_mask(Pb, L, ps, sink, local))
        for h in range(Hq):
            sel = set(got[b, h][got[b, h] >= 0].tolist())
            if forced.size <= K:
                assert set(forced.tolist()) <= sel
            else:
                assert sel == set(forced[:K].tolist())


def test_zero_forced_equals_plain_topk():
    rng = np.random.default_rng(5)
    s = rng.standard_normal((2, 4, 500)).astype(np.float32)
    ctx = np.array([500 * 16, 250 * 16 - 3], dtype=np.int32)
    s[1, :, 250:] = -np.inf
    shape = kv.make_shape(2, 4, 1, 128, 16, 500, 1000, "f32")
    idx = torch.empty((2, 4, 37), dtype=torch.int32, device="cuda")
    kv.kv_topk_select(shape, torch.from_numpy(s).cuda(), torch.from_numpy(ctx).cuda(), 37, idx)
    got = _gpu_forced(s, ctx, 16, 37, 0, 0)
    torch.cuda.synchronize()
    assert np.array_equal(got, idx.cpu().numpy())


@pytest.mark.parametrize("dtype,ps,kv_loc", [("bf16", 16, "hbm"), ("f16", 64, "hbm"),
                                             ("bf16", 16, "host")])
def test_forced_pipeline_against_oracle(dtype, ps, kv_loc):
    sink, local = 4, 64
    spec = W.tiny_spec(dtype=dtype, batch=2, hq=8, hkv=2, context=ps * 24 + 7, ps=ps,
                       index=70 + ps)
    wl = W.generate(spec, context_lens=[ps * 24 + 7, ps * 9])
    forced_max = 1 + -(-local // ps) + 1
    K = 4 + forced_max
    layer = DecodeLayer(wl, kv_loc=kv_loc, topk=K)
    layer.build_index()
    layer.score()
    layer.select(sink_tokens=sink, local_tokens=local)
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    mn, mx = check_minmax(layer, wl)
    ref_s = oracle.scores(dtype, wl.q, mn, mx, wl.block_table, wl.context_lens, ps)
    ref_idx = oracle.topk_forced(ref_s, wl.context_lens, ps, K, sink, local)
    mod = ref_s.copy()
    for b in range(spec.batch):
        L = int(wl.context_lens[b])
        Pb = -(-L // ps)
        mod[b, :, :Pb][:, _forced_mask(Pb, L, ps, sink, local)] = np.inf
    gpu_idx = layer.indices.cpu().numpy()
    check_topk_with_exemption(gpu_idx, ref_idx, mod, wl.context_lens, ps, K)
    layer.sparse_attn(indices=torch.from_numpy(ref_idx).cuda())
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ref_o = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                             wl.context_lens, wl.scale, indices=ref_idx)
    assert np.abs(layer.out.cpu().numpy() - ref_o).max() <= ATOL[dtype]
