"""GPU parity of the mean-key page index against the fp64 oracle.

Bars:
  * mean table: bit-exact -- every entry is the exact mean of the page's valid
    keys rounded once to the storage type, as the oracle computes it with
    integer arithmetic -- for every storage type, on the workloads' values and
    on adversarial pages (keys spanning every binade of the type, sums that
    cancel, ties, signed zeros, partial pages);
  * scores: |gpu - oracle| <= 1e-5 * sum_c |q_c m_c| (+ sum_c |q_c| |dm_c|,
    dm the table difference, which the table bar makes zero);
  * top-K through the pipeline: sets differ only by pages whose oracle score
    is within the two pages' score tolerances of the K-th score;
  * sparse attention over the oracle's selection: the usual 2e-3 / 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer, storage_to_torch, torch_to_bits
from parity_util import ATOL, referenced_pages

pytestmark = pytest.mark.gpu

MANT = {"f32": 23, "f16": 10, "bf16": 7}
EMIN = {"f32": -126, "f16": -14, "bf16": -126}


@pytest.fixture(autouse=True)
def _lib(kvlib):
    kv.kv_debug_config(-1, 2_000_000_000)
    kv.kv_device_status()
    yield


def bits_to_f64(bits, dtype):
    bits = np.asarray(bits)
    if dtype == "f32":
        return bits.astype(np.uint32).view(np.float32).astype(np.float64)
    if dtype == "f16":
        return bits.astype(np.uint16).view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp(v, dtype):
    # spacing of the storage type at v, with the fixed subnormal spacing below
    # the smallest normal
    e = np.floor(np.log2(np.maximum(np.abs(v), 1e-300)))
    return np.exp2(np.maximum(e, EMIN[dtype]) - MANT[dtype])


def check_mean_table(layer, wl, rows=None):
    """Returns (oracle table, gpu table as fp64) after checking the bar."""
    spec = wl.spec
    dtype = spec.dtype
    sl = slice(None) if rows is None else rows
    ref = oracle.mean_build(dtype, wl.k_cache, wl.block_table[sl], wl.context_lens[sl])
    gpu = bits_to_f64(layer.mean_bits(), dtype)
    pages = referenced_pages(wl, rows)
    r, g = ref[pages], gpu[pages]
    # bit for bit, signed zeros included
    assert np.array_equal(g, r) and np.array_equal(np.signbit(g), np.signbit(r))
    return ref, gpu


def score_tol(dtype, q, ref_mean, gpu_mean, bt, ctx, ps):
    qf = W.storage_to_f64(q, dtype)
    B, Hq, d = qf.shape
    Hkv = ref_mean.shape[1]
    G = Hq // Hkv
    maxP = bt.shape[1]
    tol = np.zeros((B, Hq, maxP))
    for b in range(B):
        P = -(-int(ctx[b]) // ps)
        ph = bt[b, :P]
        for h in range(Hq):
            m = ref_mean[ph, h // G]                      # [P][d]
            dm = np.abs(gpu_mean[ph, h // G] - m)
            tol[b, h, :P] = 1e-5 * np.abs(qf[b, h] * m).sum(axis=1) + np.abs(qf[b, h]) @ dm.T
    return tol


def check_topk_tolerant(gpu_idx, ref_idx, ref_s, tol, ctx, ps, K):
    for b in range(ref_idx.shape[0]):
        P = -(-int(ctx[b]) // ps)
        keff = min(K, P)
        for h in range(ref_idx.shape[1]):
            g, r = gpu_idx[b, h], ref_idx[b, h]
            assert (g[keff:] == -1).all() and list(g[:keff]) == sorted(g[:keff])
            gs, rs = set(g[:keff].tolist()), set(r[:keff].tolist())
            if gs == rs:
                continue
            s, t = ref_s[b, h, :P], tol[b, h, :P]
            kth = int(np.argsort(-s, kind="stable")[keff - 1])
            extra, missing = gs - rs, rs - gs
            assert len(extra) == len(missing)
            for p in extra | missing:
                assert abs(s[p] - s[kth]) <= t[p] + t[kth] + 1e-30, (b, h, p)


def run_mean_pipeline(wl, K, kv_loc=None):
    spec = wl.spec
    dtype, ps = spec.dtype, spec.page_size
    layer = DecodeLayer(wl, kv_loc=kv_loc, topk=K)
    layer.build_mean_index()
    layer.score_mean()
    layer.select()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ref_m, gpu_m = check_mean_table(layer, wl)
    ref_s = oracle.mean_scores(dtype, wl.q, ref_m, wl.block_table, wl.context_lens, ps)
    gm = np.where(np.isnan(ref_m), 0.0, gpu_m)
    tol = score_tol(dtype, wl.q, np.nan_to_num(ref_m), gm, wl.block_table, wl.context_lens, ps)
    gs = layer.scores.cpu().numpy().astype(np.float64)
    for b in range(spec.batch):
        P = -(-int(wl.context_lens[b]) // ps)
        assert (np.abs(gs[b, :, :P] - ref_s[b, :, :P]) <= tol[b, :, :P]).all()
        assert np.isneginf(gs[b, :, P:]).all()
    ref_idx = oracle.topk(ref_s, wl.context_lens, ps, K)
    check_topk_tolerant(layer.indices.cpu().numpy(), ref_idx, ref_s, tol, wl.context_lens, ps, K)
    layer.sparse_attn(indices=torch.from_numpy(ref_idx).cuda())
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ref_o = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                             wl.context_lens, wl.scale, indices=ref_idx)
    assert np.abs(layer.out.cpu().numpy() - ref_o).max() <= ATOL[dtype]
    return layer


@pytest.mark.parametrize("dtype,hq,hkv,ps", [
    ("bf16", 8, 2, 16),    # G = 4: tensor-core score
    ("f16", 16, 2, 16),    # G = 8: tensor-core score
    ("bf16", 4, 4, 64),    # G = 1: CUDA-core score
    ("f16", 4, 2, 16),     # G = 2
    ("f32", 4, 1, 16),     # fp32: CUDA-core score
    ("bf16", 24, 2, 64),   # G = 12: three chunks of 4 heads
])
def test_mean_index_pipeline(dtype, hq, hkv, ps):
    spec = W.tiny_spec(dtype=dtype, batch=3, hq=hq, hkv=hkv, context=ps * 37 + 5, ps=ps,
                       index=90 + hq + ps)
    wl = W.generate(spec, context_lens=[ps * 37 + 5, ps * 11, 3])
    run_mean_pipeline(wl, 6)


def test_mean_index_host_pinned():
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=8, hkv=2, context=16 * 40 + 9, ps=16, index=95)
    wl = W.generate(spec, context_lens=[16 * 40 + 9, 16 * 7])
    layer = run_mean_pipeline(wl, 5, kv_loc="host")
    assert not layer.k_cache.is_cuda


def _wide_keys(rng, dtype, shape):
    """Keys whose magnitudes span every binade of the type, in the storage
    type; a page's first and last tokens cancel each other around the rest."""
    lo, hi = {"f16": (-24, 15), "bf16": (-133, 127), "f32": (-149, 127)}[dtype]
    e = rng.integers(lo, hi + 1, shape)
    x = np.ldexp(rng.uniform(1.0, 2.0, shape), e) * rng.choice([-1.0, 1.0], shape)
    cap = 6e4 if dtype == "f16" else 3e38
    x = np.clip(x, -cap, cap)
    big = np.ldexp(1.5, hi - 2)
    x[..., 0, :] = big * np.sign(x[..., 0, :])
    x[..., -1, :] = -x[..., 0, :]
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "f32":
        return x.astype(np.float32)
    return W.f32_to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("ps", [16, 64])
def test_mean_table_is_exact_on_adversarial_pages(dtype, ps):
    # every page of every row gets wide-range keys; the rows' lengths leave
    # partial last pages (n = 1, a ragged n, a full page)
    rng = np.random.default_rng(4000 + ps)
    ctx = [ps * 5 + 1, ps * 3 + ps // 2 + 3, ps * 2]
    spec = W.tiny_spec(dtype=dtype, batch=3, hq=4, hkv=2, context=max(ctx), ps=ps,
                       index=4000 + ps)
    wl = W.generate(spec, context_lens=ctx)
    wl.k_cache[...] = _wide_keys(rng, dtype, wl.k_cache.shape)
    # hand-made channels: f16 subnormals next to +-6e4, exact ties, signed zeros
    ph = int(wl.block_table[0, 0])
    special = {
        "f16": [65504.0, 2.0 ** -24, 3 * 2.0 ** -24, -65504.0],
        "bf16": [2.0 ** 120, 2.0 ** -130, 2.0 ** -100, -(2.0 ** 120)],
        "f32": [2.0 ** 100, 2.0 ** -149, 1.0, -(2.0 ** 100)],
    }[dtype]
    col = np.zeros(ps)
    col[:4] = special
    wl.k_cache[ph, 0, :, 0] = W.to_storage(col.astype(np.float32), dtype) if dtype != "f16" \
        else col.astype(np.float16)
    wl.k_cache[ph, 0, :, 1] = W.to_storage(np.full(ps, -0.0, dtype=np.float32), dtype) \
        if dtype != "f16" else np.full(ps, -0.0, dtype=np.float16)
    tie = np.zeros(ps)         # mean 1.5 smallest subnormals: a tie, to the even 2
    tie[0] = 1.5 * ps * {"f16": 2.0 ** -24, "bf16": 2.0 ** -133, "f32": 2.0 ** -149}[dtype]
    wl.k_cache[ph, 0, :, 2] = W.to_storage(tie.astype(np.float32), dtype) if dtype != "f16" \
        else tie.astype(np.float16)
    layer = DecodeLayer(wl, topk=2)
    layer.build_mean_index()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ref, gpu = check_mean_table(layer, wl)
    r0 = ref[ph, 0]
    assert np.signbit(r0[1]) and r0[1] == 0.0             # all -0 keys: -0
    assert r0[2] == 2 * {"f16": 2.0 ** -24, "bf16": 2.0 ** -133, "f32": 2.0 ** -149}[dtype]
    # refresh of the last pages after the keys change agrees too
    wl.k_cache[...] = _wide_keys(rng, dtype, wl.k_cache.shape)
    layer.k_cache.copy_(storage_to_torch(wl.k_cache, dtype).cuda())
    layer.build_mean_index(last_only=True)
    torch.cuda.synchronize()
    full = oracle.mean_build(dtype, wl.k_cache, wl.block_table, wl.context_lens)
    gpu = bits_to_f64(layer.mean_bits(), dtype)
    for b, L in enumerate(ctx):
        p_last = int(wl.block_table[b, (L - 1) // ps])
        assert np.array_equal(gpu[p_last], full[p_last])
        assert np.array_equal(np.signbit(gpu[p_last]), np.signbit(full[p_last]))


def test_mean_refresh_after_appends():
    spec = W.tiny_spec(dtype="f16", batch=3, hq=8, hkv=2, context=16 * 6, ps=16, index=96)
    wl = W.generate(spec, context_lens=[16, 40, 1])
    layer = DecodeLayer(wl, topk=3)
    layer.build_mean_index()
    for s in range(20):
        kn, vn = W.new_tokens(spec, s)
        layer.append(storage_to_torch(kn, "f16").cuda(), storage_to_torch(vn, "f16").cuda())
        layer.build_mean_index(last_only=True)
        k2, v2, _, _ = oracle.append_token("f16", kn, vn, wl.k_cache, wl.v_cache,
                                           wl.block_table, wl.context_lens)
        wl.k_cache, wl.v_cache = k2, v2
        wl.context_lens = wl.context_lens + 1
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    assert np.array_equal(layer.context_lens.cpu().numpy(), wl.context_lens)
    check_mean_table(layer, wl)


def test_mean_index_full_size_llama_32k_sampled():
    spec = W.WORKLOADS["llama3.1-8b-b4-ctx32k"]
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=spec.topk)
    layer.build_mean_index()
    layer.score_mean()
    layer.select()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    ps = spec.page_size
    gpu_s = layer.scores.cpu().numpy()
    gpu_idx = layer.indices.cpu().numpy()
    for b in (0, spec.batch - 1):
        sl = slice(b, b + 1)
        ref_m, gpu_m = check_mean_table(layer, wl, rows=[b])
        ref_s = oracle.mean_scores("bf16", wl.q[sl], ref_m, wl.block_table[sl],
                                   wl.context_lens[sl], ps)
        gm = np.where(np.isnan(ref_m), 0.0, gpu_m)
        tol = score_tol("bf16", wl.q[sl], np.nan_to_num(ref_m), gm, wl.block_table[sl],
                        wl.context_lens[sl], ps)
        assert (np.abs(gpu_s[sl].astype(np.float64) - ref_s) <= tol).all()
        ref_idx = oracle.topk(ref_s, wl.context_lens[sl], ps, spec.topk)
        check_topk_tolerant(gpu_idx[sl], ref_idx, ref_s, tol, wl.context_lens[sl], ps, spec.topk)
