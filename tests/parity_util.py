"""Comparison helpers shared by the GPU parity tests (tolerances, bit views,
the top-K boundary exemption)."""
import numpy as np

import oracle

from offloaded_kv_cache_gb300 import workloads as W

ATOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


def f64_to_bits(x, dtype):
    x = np.asarray(x)
    if dtype == "f32":
        return x.astype(np.float32).view(np.uint32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    return (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def referenced_pages(wl, rows=None):
    ps = wl.spec.page_size
    out = set()
    for b in (range(wl.spec.batch) if rows is None else rows):
        for p in range(-(-int(wl.context_lens[b]) // ps)):
            out.add(int(wl.block_table[b, p]))
    return sorted(out)


def check_minmax(layer, wl, rows=None):
    dtype = wl.spec.dtype
    sl = slice(None) if rows is None else rows
    mn, mx = oracle.minmax_build(dtype, wl.k_cache, wl.block_table[sl], wl.context_lens[sl])
    gpu = layer.minmax_bits()
    pages = referenced_pages(wl, rows)
    assert np.array_equal(gpu[pages, :, 0], f64_to_bits(mn[pages], dtype))
    assert np.array_equal(gpu[pages, :, 1], f64_to_bits(mx[pages], dtype))
    return mn, mx


def score_tolerance(dtype, q, mn, mx, bt, ctx, ps):
    # 1e-5 * sum_c |max(q_c mn_c, q_c mx_c)| per (b, h, p)
    qf = W.storage_to_f64(q, dtype)
    B, Hq, d = qf.shape
    Hkv = mn.shape[1]
    G = Hq // Hkv
    tol = np.zeros((B, Hq, bt.shape[1]))
    for b in range(B):
        P = -(-int(ctx[b]) // ps)
        phys = bt[b, :P]
        for h in range(Hq):
            a = qf[b, h][None, :] * mn[phys, h // G]
            c = qf[b, h][None, :] * mx[phys, h // G]
            tol[b, h, :P] = 1e-5 * np.abs(np.maximum(a, c)).sum(axis=1) + 1e-30
    return tol


def check_scores(gpu_scores, ref_scores, tol, ctx, ps):
    for b in range(ref_scores.shape[0]):
        P = -(-int(ctx[b]) // ps)
        g = gpu_scores[b, :, :P].astype(np.float64)
        assert (np.abs(g - ref_scores[b, :, :P]) <= tol[b, :, :P]).all()
        assert np.isneginf(gpu_scores[b, :, P:]).all()


def check_topk_with_exemption(gpu_idx, ref_idx, ref_scores, ctx, ps, K):
    for b in range(ref_idx.shape[0]):
        P = -(-int(ctx[b]) // ps)
        keff = min(K, P)
        for h in range(ref_idx.shape[1]):
            g = gpu_idx[b, h]
            r = ref_idx[b, h]
            assert (g[keff:] == -1).all() and (r[keff:] == -1).all()
            gs, rs = set(g[:keff].tolist()), set(r[:keff].tolist())
            assert list(g[:keff]) == sorted(gs) and len(gs) == keff
            if gs == rs:
                continue
            s = ref_scores[b, h, :P]
            tau = np.sort(s)[::-1][keff - 1]
            boundary = lambda p: abs(s[p] - tau) < 1e-6 * abs(tau) + 1e-30
            extra, missing = gs - rs, rs - gs
            assert len(extra) == len(missing)
            assert all(boundary(p) for p in extra | missing), (b, h, extra, missing)
