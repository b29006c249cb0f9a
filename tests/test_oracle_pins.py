"""Pins of the fp64 oracle against what the pages and mathematics fix.

Every check here is independent of the oracle's own code: library routines
(numpy, torch SDPA in fp64), brute force on tiny inputs, closed forms,
invariants and hand-worked fixtures.  Each is chosen so that a plausible slip in
the oracle (a dropped scale, a swapped min/max, a wrong GQA head, a block-table
index taken as physical, a tie broken the wrong way, an unmasked partial page)
fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- decode

def test_decode_f16_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 10) & 31) != 31
    vals = bits.view(np.float16)
    got = oracle.decode("f16", vals)
    ref = vals.astype(np.float64)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(ref[finite]))


def test_decode_bf16_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    got = oracle.decode("bf16", bits)
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(ref[finite]))


def test_decode_f32_random():
    x = _rng(1).standard_normal(1000).astype(np.float32)
    assert np.array_equal(oracle.decode("f32", x), x.astype(np.float64))


# ---------------------------------------------------------------- min / max index

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_page_minmax_matches_numpy_on_nonzero_values(dtype):
    rng = _rng(2)
    for ps, n in [(16, 16), (16, 5), (64, 64), (64, 1)]:
        x = rng.standard_normal((ps, 8)).astype(np.float32) + 0.01
        x[x == 0] = 1.0
        page = W.to_storage(x, dtype)
        mn, mx = oracle.page_minmax(dtype, page, n)
        ref = W.storage_to_f64(page, dtype)[:n]
        assert np.array_equal(mn, ref.min(axis=0))
        assert np.array_equal(mx, ref.max(axis=0))


def test_page_minmax_signed_zero_total_order():
    # -0.0 < +0.0 in totalOrder: the min must carry the sign, the max must not,
    # whichever token comes first.
    page = np.array([[0.0, -0.0, -0.0, 0.0, 1.0],
                     [-0.0, 0.0, -0.0, 0.0, -0.0],
                     [0.0, -0.0, -0.0, 0.0, 0.0]], dtype=np.float32)
    mn, mx = oracle.page_minmax("f32", page)
    assert list(np.signbit(mn)) == [True, True, True, False, True]
    assert list(np.signbit(mx)) == [False, False, True, False, False]
    assert mx[4] == 1.0


def test_page_minmax_ignores_tokens_past_the_last_valid_one():
    page = np.full((16, 4), 1e30, dtype=np.float32)
    page[8:] *= -1
    page[:3] = np.arange(12, dtype=np.float32).reshape(3, 4)
    mn, mx = oracle.page_minmax("f32", page, 3)
    assert np.array_equal(mn, page[0])
    assert np.array_equal(mx, page[2])


def test_minmax_build_invariants_and_block_table_indirection():
    spec = W.tiny_spec(dtype="bf16", batch=3, hq=4, hkv=2, context=70, ps=16, index=3)
    wl = W.generate(spec, context_lens=[70, 33, 16])
    mn, mx = oracle.minmax_build("bf16", wl.k_cache, wl.block_table, wl.context_lens)
    k = W.storage_to_f64(wl.k_cache, "bf16")
    for b in range(spec.batch):
        L = int(wl.context_lens[b])
        for p in range(-(-L // spec.page_size)):
            n = min(spec.page_size, L - p * spec.page_size)
            phys = wl.block_table[b, p]
            for kvh in range(spec.num_kv_heads):
                toks = k[phys, kvh, :n]
                # bound holds and is attained (mn and mx are members of the page)
                assert (toks >= mn[phys, kvh]).all() and (toks <= mx[phys, kvh]).all()
                assert np.array_equal(mn[phys, kvh], toks.min(axis=0))
                assert np.array_equal(mx[phys, kvh], toks.max(axis=0))
    # pages no row references stay untouched
    used = {int(wl.block_table[b, p]) for b in range(3)
            for p in range(-(-int(wl.context_lens[b]) // 16))}
    unused = [i for i in range(spec.num_phys_pages) if i not in used]
    assert unused and np.isnan(mn[unused]).all()


def test_minmax_identical_keys_collapse():
    page = np.tile(np.linspace(-3, 3, 32, dtype=np.float32), (16, 1))
    mn, mx = oracle.page_minmax("f32", page)
    assert np.array_equal(mn, page[0]) and np.array_equal(mx, page[0])


# ---------------------------------------------------------------- page score

def test_page_score_hand_worked_fixture():
    fx = json.load(open(os.path.join(GOLDEN, "quest_bound_example.json")))
    s = oracle.page_score(np.array(fx["q"]), np.array(fx["mn"]), np.array(fx["mx"]))
    assert s == fx["score"]


def test_page_score_is_an_upper_bound_and_tight_on_extreme_keys():
    rng = _rng(4)
    for trial in range(50):
        d, n = 16, int(rng.integers(1, 17))
        keys = rng.standard_normal((n, d))
        q = rng.standard_normal(d)
        mn, mx = keys.min(axis=0), keys.max(axis=0)
        s = oracle.page_score(q, mn, mx)
        assert s >= (keys @ q).max() - 1e-12
        # add the corner key that picks, per channel, the extreme matching q's sign
        corner = np.where(q >= 0, mx, mn)
        keys2 = np.vstack([keys, corner])
        s2 = oracle.page_score(q, keys2.min(axis=0), keys2.max(axis=0))
        assert s2 == pytest.approx((keys2 @ q).max(), rel=1e-12, abs=1e-12)


def test_page_score_equals_dot_for_single_or_identical_keys():
    rng = _rng(5)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    assert oracle.page_score(q, k, k) == pytest.approx(float(q @ k), rel=1e-13, abs=1e-12)


def test_scores_driver_gqa_head_and_block_table_by_brute_force():
    # Score of (b, h, p) must equal max_t q_h . k_t over the page of kv head h // G
    # when the page contains its own corner key; each page here is built so.
    spec = W.tiny_spec(dtype="f32", batch=2, hq=6, hkv=2, context=40, ps=16, index=6)
    wl = W.generate(spec, context_lens=[40, 23])
    k = wl.k_cache.copy()
    q = wl.q.astype(np.float64)
    G = spec.group
    # Give head 0 of every group a corner key (token 0 of each page): the score is then
    # tight for that head only, and a wrong head mapping breaks the equality.
    for b in range(2):
        L = int(wl.context_lens[b])
        for p in range(-(-L // 16)):
            n = min(16, L - p * 16)
            phys = wl.block_table[b, p]
            for kvh in range(2):
                toks = k[phys, kvh, 1:n].astype(np.float64) if n > 1 else np.zeros((0, 128))
                h = kvh * G
                if len(toks):
                    corner = np.where(q[b, h] >= 0, toks.max(axis=0), toks.min(axis=0))
                    k[phys, kvh, 0] = corner.astype(np.float32)
    mn, mx = oracle.minmax_build("f32", k, wl.block_table, wl.context_lens)
    s = oracle.scores("f32", wl.q, mn, mx, wl.block_table, wl.context_lens, 16)
    for b in range(2):
        L = int(wl.context_lens[b])
        P = -(-L // 16)
        assert np.isneginf(s[b, :, P:]).all()
        for p in range(P):
            n = min(16, L - p * 16)
            phys = wl.block_table[b, p]
            for h in range(6):
                toks = k[phys, h // G, :n].astype(np.float64)
                best = (toks @ q[b, h]).max()
                assert s[b, h, p] >= best - 1e-9
                if h % G == 0 and n > 1:
                    assert s[b, h, p] == pytest.approx(best, rel=1e-12, abs=1e-9)


# ---------------------------------------------------------------- top-K

def _brute_topk(s, K):
    """The unique K-subset whose every member beats every non-member
    (higher score, or equal score and lower index)."""
    P = len(s)
    keff = min(K, P)
    found = []
    for sub in itertools.combinations(range(P), keff):
        ins = set(sub)
        ok = all((s[i] > s[j]) or (s[i] == s[j] and i < j)
                 for i in ins for j in range(P) if j not in ins)
        if ok:
            found.append(sub)
    assert len(found) == 1
    return list(found[0]) + [-1] * (K - keff)


def test_topk_brute_force_all_subsets_with_ties():
    rng = _rng(7)
    for trial in range(60):
        P = int(rng.integers(1, 11))
        K = int(rng.integers(1, 12))
        s = rng.integers(0, 4, size=P).astype(np.float64)  # many ties
        assert list(oracle.topk_row(s, K)) == _brute_topk(list(s), K)


def test_topk_matches_stable_argsort():
    rng = _rng(8)
    for P, K in [(256, 32), (2048, 256), (1000, 999), (5, 9)]:
        s = np.round(rng.standard_normal(P), 2)  # ties at the boundary are likely
        ref = np.sort(np.argsort(-s, kind="stable")[:min(K, P)])
        ref = np.concatenate([ref, -np.ones(K - len(ref), dtype=np.int64)])
        assert np.array_equal(oracle.topk_row(s, K), ref)


def test_topk_all_equal_and_boundary_ties():
    assert list(oracle.topk_row(np.zeros(10), 4)) == [0, 1, 2, 3]
    assert list(oracle.topk_row(np.array([1.0, 3, 3, 3, 2]), 2)) == [1, 2]
    assert list(oracle.topk_row(np.array([-np.inf, 1.0]), 1)) == [1]
    assert list(oracle.topk_row(np.array([2.0, 1.0]), 4)) == [0, 1, -1, -1]


def test_forced_selection_hand_worked_pages():
    # 16-token pages.  len 100 (P = 7), sink 4, local 64: the sink is in page
    # 0; tokens 36..99 are in pages 2..6.  With k = 7 every page is taken; with
    # k = 6 the one page left out is page 1, the only unforced one.
    s = np.arange(7, dtype=np.float64)[None, None, :] * -1.0      # page 0 scores highest
    ctx = np.array([100], dtype=np.int32)
    assert list(oracle.topk_forced(s, ctx, 16, 6, 4, 64)[0, 0]) == [0, 2, 3, 4, 5, 6]
    # len 70 (P = 5), local 64 -> tokens 6..69: every page is forced; k = 3
    # keeps the three lowest-index ones
    ctx = np.array([70], dtype=np.int32)
    assert list(oracle.topk_forced(s[:, :, :5], ctx, 16, 3, 0, 64)[0, 0]) == [0, 1, 2]
    # len 64 (P = 4), local 16: only the last page; sink 17 -> pages 0 and 1;
    # one free slot goes to the best of page 2 (score -2) alone
    ctx = np.array([64], dtype=np.int32)
    assert list(oracle.topk_forced(s[:, :, :4], ctx, 16, 4, 17, 16)[0, 0]) == [0, 1, 2, 3]
    assert list(oracle.topk_forced(s[:, :, :4], ctx, 16, 3, 17, 16)[0, 0]) == [0, 1, 3]
    # local 1: the page of the last token only (token 63 is in page 3)
    assert list(oracle.topk_forced(s[:, :, :4], ctx, 16, 1, 0, 1)[0, 0]) == [3]
    # sink 16 fills page 0 exactly and does not reach page 1
    s2 = np.array([[[-5.0, -4.0, 0.0, 1.0]]])
    assert list(oracle.topk_forced(s2, ctx, 16, 2, 16, 0)[0, 0]) == [0, 3]


def test_forced_selection_matches_sort_with_forced_pages_at_plus_infinity():
    # Library route: stable argsort of the scores with every forced page's
    # score replaced by +inf picks the same set, for k below, at and above the
    # number of forced pages, and reduces to plain top-K with nothing forced.
    rng = _rng(50)
    for trial in range(60):
        ps = [16, 64][trial % 2]
        P = int(rng.integers(1, 40))
        L = int(rng.integers((P - 1) * ps + 1, P * ps + 1))
        sink = int(rng.choice([0, 1, 4, 16, 40, 64]))
        local = int(rng.choice([0, 1, 64, 200]))
        k = int(rng.integers(1, P + 3))
        sc = np.round(rng.standard_normal(P), 1)
        got = oracle.topk_forced(sc[None, None, :], np.array([L], np.int32), ps, k, sink,
                                 local)[0, 0]
        tok_lo = np.arange(P) * ps
        tok_hi = np.minimum(L, tok_lo + ps)
        forced = ((sink > 0) & (tok_lo < sink)) | ((local > 0) & (tok_hi > L - local))
        mod = np.where(forced, np.inf, sc)
        pick = np.sort(np.argsort(-mod, kind="stable")[:min(k, P)])
        ref = np.full(k, -1)
        ref[:pick.size] = pick
        assert np.array_equal(got, ref), (trial, P, L, sink, local, k)
        if sink == 0 and local == 0:
            assert np.array_equal(got, oracle.topk_row(sc, k))


# ---------------------------------------------------------------- attention

def _gather_dense(wl, b, h):
    spec = wl.spec
    L = int(wl.context_lens[b])
    P = -(-L // spec.page_size)
    kvh = h // spec.group
    ks = [W.storage_to_f64(wl.k_cache[wl.block_table[b, p], kvh], spec.dtype) for p in range(P)]
    vs = [W.storage_to_f64(wl.v_cache[wl.block_table[b, p], kvh], spec.dtype) for p in range(P)]
    return np.concatenate(ks)[:L], np.concatenate(vs)[:L]


def _sdpa(q, k, v, scale):
    qt = torch.from_numpy(q)[None, None, None, :]
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[0, 0, 0].numpy()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_dense_attention_matches_torch_sdpa_fp64(dtype):
    spec = W.tiny_spec(dtype=dtype, batch=2, hq=4, hkv=2, context=77, ps=16, index=9)
    wl = W.generate(spec, context_lens=[77, 16])
    out = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                           wl.context_lens, wl.scale)
    q = W.storage_to_f64(wl.q, dtype)
    for b in range(2):
        for h in range(4):
            k, v = _gather_dense(wl, b, h)
            ref = _sdpa(q[b, h], k, v, wl.scale)
            assert np.abs(out[b, h] - ref).max() <= 1e-12


def test_all_pages_selected_equals_dense_exactly():
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=4, hkv=1, context=50, ps=16, index=10)
    wl = W.generate(spec, context_lens=[50, 31])
    dense = oracle.attention("bf16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                             wl.context_lens, wl.scale)
    idx = np.tile(np.arange(spec.max_pages, dtype=np.int32), (2, 4, 1))
    idx[1, :, 2:] = -1  # row 1 has 2 pages; pad the rest
    sparse = oracle.attention("bf16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                              wl.context_lens, wl.scale, indices=idx)
    assert np.array_equal(dense, sparse)


def test_sparse_attention_matches_sdpa_over_selected_tokens():
    spec = W.tiny_spec(dtype="f16", batch=1, hq=2, hkv=1, context=90, ps=16, index=11)
    wl = W.generate(spec)
    idx = np.array([[[0, 3, 5], [1, 2, -1]]], dtype=np.int32)   # page 5 is partial (10 tokens)
    out = oracle.attention("f16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                           wl.context_lens, wl.scale, indices=idx)
    q = W.storage_to_f64(wl.q, "f16")
    for h in range(2):
        k, v = _gather_dense(wl, 0, h)
        toks = [t for p in idx[0, h] if p >= 0 for t in range(p * 16, min(90, p * 16 + 16))]
        ref = _sdpa(q[0, h], k[toks], v[toks], wl.scale)
        assert np.abs(out[0, h] - ref).max() <= 1e-12


def test_identical_keys_give_mean_of_values():
    spec = W.tiny_spec(dtype="f32", batch=1, hq=1, hkv=1, context=37, ps=16, index=12)
    wl = W.generate(spec)
    wl.k_cache[:] = wl.k_cache[0, 0, 0]
    out = oracle.attention("f32", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                           wl.context_lens, wl.scale)
    _, v = _gather_dense(wl, 0, 0)
    assert np.abs(out[0, 0] - v.mean(axis=0)).max() <= 1e-12


def test_single_token_context_returns_its_value():
    spec = W.tiny_spec(dtype="bf16", batch=1, hq=2, hkv=2, context=1, ps=16, index=13)
    wl = W.generate(spec)
    out = oracle.attention("bf16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                           wl.context_lens, wl.scale)
    for h in range(2):
        v = W.storage_to_f64(wl.v_cache[wl.block_table[0, 0], h, 0], "bf16")
        assert np.array_equal(out[0, h], v)


def test_partial_last_page_is_masked():
    spec = W.tiny_spec(dtype="f32", batch=1, hq=1, hkv=1, context=20, ps=16, index=14)
    wl = W.generate(spec)
    phys = wl.block_table[0, 1]
    wl.k_cache[phys, 0, 4:] = 1e3 * wl.q[0, 0]      # would dominate if not masked
    wl.v_cache[phys, 0, 4:] = 1e6
    out = oracle.attention("f32", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                           wl.context_lens, wl.scale)
    k, v = _gather_dense(wl, 0, 0)
    assert np.abs(out[0, 0] - _sdpa(wl.q[0, 0].astype(np.float64), k, v, wl.scale)).max() <= 1e-12
    assert np.abs(out[0, 0]).max() < 10


def test_page_permutation_invariance():
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=2, hkv=1, context=64, ps=16, index=15)
    wl = W.generate(spec, context_lens=[64, 40])
    out1 = oracle.attention("bf16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                            wl.context_lens, wl.scale)
    perm = _rng(16).permutation(spec.num_phys_pages)
    inv = np.argsort(perm)
    k2 = wl.k_cache[perm]
    v2 = wl.v_cache[perm]
    bt2 = inv[wl.block_table].astype(np.int32)
    out2 = oracle.attention("bf16", wl.q, k2, v2, bt2, wl.context_lens, wl.scale)
    assert np.array_equal(out1, out2)


def test_linearity_in_values():
    spec = W.tiny_spec(dtype="f32", batch=1, hq=2, hkv=1, context=48, ps=16, index=17)
    wl = W.generate(spec)
    rng = _rng(18)
    v1 = rng.integers(-8, 8, wl.v_cache.shape).astype(np.float32)
    v2 = rng.integers(-8, 8, wl.v_cache.shape).astype(np.float32)
    f = lambda v: oracle.attention("f32", wl.q, wl.k_cache, v, wl.block_table,
                                   wl.context_lens, wl.scale)
    assert np.abs(f(3 * v1 - 2 * v2) - (3 * f(v1) - 2 * f(v2))).max() <= 1e-11


def test_planted_logit_gap_returns_planted_value():
    spec = W.tiny_spec(dtype="f32", batch=1, hq=1, hkv=1, context=64, ps=16, index=19)
    wl = W.generate(spec)
    q = wl.q[0, 0].astype(np.float64)
    t = 37
    phys = wl.block_table[0, t // 16]
    wl.k_cache[phys, 0, t % 16] = (60.0 * q / np.linalg.norm(q)).astype(np.float32)
    out = oracle.attention("f32", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                           wl.context_lens, wl.scale)
    assert np.abs(out[0, 0] - wl.v_cache[phys, 0, t % 16]).max() < 1e-9


def test_scale_is_applied():
    # A wrong or missing scale changes the softmax temperature; SDPA with the
    # same explicit scale pins it (checked at two scales).
    spec = W.tiny_spec(dtype="f32", batch=1, hq=1, hkv=1, context=30, ps=16, index=20)
    wl = W.generate(spec)
    k, v = _gather_dense(wl, 0, 0)
    for sc in (0.02, 0.5):
        out = oracle.attention("f32", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                               wl.context_lens, sc)
        assert np.abs(out[0, 0] - _sdpa(wl.q[0, 0].astype(np.float64), k, v, sc)).max() <= 1e-12


def test_rows_subset_matches_full():
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=4, hkv=2, context=40, ps=16, index=21)
    wl = W.generate(spec)
    full = oracle.attention("bf16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                            wl.context_lens, wl.scale)
    part = oracle.attention("bf16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                            wl.context_lens, wl.scale, rows=[1, 6])
    assert np.array_equal(part[0, 1], full[0, 1]) and np.array_equal(part[1, 2], full[1, 2])
    assert np.isnan(part[0, 0]).all()


# ---------------------------------------------------------------- shapes

def test_workload_byte_counts_printed_by_the_pages():
    fx = json.load(open(os.path.join(GOLDEN, "page_sizes.json")))
    opt = W.WORKLOADS["opt6.7b-b32-ctx544"]
    per_tok = opt.batch * opt.num_kv_heads * opt.head_dim * opt.elem_bytes
    assert per_tok == fx["opt6.7b_layer_k_bytes_one_token"]["value"]
    assert per_tok * 512 == fx["opt6.7b_layer_k_bytes_512_tokens"]["value"]
    lo, hi = fx["opt6.7b_layer_k_bytes_544_tokens_upper"]["range_mib"]
    assert lo * 2**20 <= per_tok * opt.context <= hi * 2**20
    ll = W.WORKLOADS["llama3.1-8b-b1-ctx128k-host"]
    e = fx["llama3.1_8b_kv_bytes_128k_all_layers_min"]
    assert ll.kv_bytes() * e["layers"] > e["value"]
    assert ll.kv_bytes() == 512 * 2**20
    l3 = W.WORKLOADS["llama3.1-8b-b4-ctx32k"]
    e = fx["llama3_8b_kv_bytes_b8_100k_all_layers_approx"]
    b8 = l3.with_(batch=8, context=100_000)
    assert 0.9 * e["value"] <= b8.kv_bytes() * e["layers"] <= 1.1 * e["value"]


def test_planted_tokens_carry_the_largest_logits_in_the_fp32_workload():
    # Generator check: the 8 planted tokens have k = 4 q/|q|, so q.k = 4|q| and they
    # hold the 8 largest logits.  (The Quest page bound does not lift their pages
    # into the top-32 at d = 128: it is dominated by the per-channel extremes of the
    # other 15 random keys of the page.  That is a property of the method on this
    # recipe, recorded in the design notes, not something to pin.)
    wl = W.generate(W.WORKLOADS["fp32-b1-ctx4k"])
    spec = wl.spec
    q = wl.q[0, 0].astype(np.float64)
    keys = np.concatenate([wl.k_cache[wl.block_table[0, p], 0] for p in range(spec.max_pages)])
    logits = keys.astype(np.float64) @ q
    top8 = np.sort(logits)[-8:]
    assert np.allclose(top8, 4 * np.linalg.norm(q), rtol=1e-6)


# ---------------------------------------------------------------- decode append

def _token(wl, b, t):
    """K and V rows [Hkv][d] of token t of sequence b, read through the block table."""
    ps = wl.spec.page_size
    phys = wl.block_table[b, t // ps]
    return wl.k_cache[phys, :, t % ps], wl.v_cache[phys, :, t % ps]


@pytest.mark.parametrize("dtype,ps", [("bf16", 16), ("f16", 64), ("f32", 16)])
def test_append_token_by_token_rebuilds_the_cache_and_its_index(dtype, ps):
    # Appending every token of a workload one step at a time, into caches and
    # min/max tables that start as garbage, must give back the workload's
    # caches at every valid position and exactly the bulk index build.
    spec = W.tiny_spec(dtype=dtype, batch=3, hq=4, hkv=2, context=3 * ps + 5, ps=ps, index=40)
    lens = [3 * ps + 5, ps, 7]
    wl = W.generate(spec, context_lens=lens)
    rng = _rng(41)
    k = W.to_storage(rng.standard_normal(wl.k_cache.shape).astype(np.float32) * 50, dtype)
    v = W.to_storage(rng.standard_normal(wl.v_cache.shape).astype(np.float32) * 50, dtype)
    mn = rng.standard_normal((spec.num_phys_pages, 2, spec.head_dim)) * 50
    mx = mn + 1.0
    done = spec.max_pages * ps            # a length the append leaves alone
    for t in range(max(lens)):
        ctx = np.array([t if t < L else done for L in lens], dtype=np.int32)
        kn = np.zeros((3, 2, spec.head_dim), dtype=k.dtype)
        vn = np.zeros_like(kn)
        for b in range(3):
            if t < lens[b]:
                kn[b], vn[b] = _token(wl, b, t)
        k, v, mn, mx = oracle.append_token(dtype, kn, vn, k, v, wl.block_table, ctx, mn, mx)
    ref_mn, ref_mx = oracle.minmax_build(dtype, wl.k_cache, wl.block_table, wl.context_lens)
    for b, L in enumerate(lens):
        for t in range(L):
            kt, vt = _token(wl, b, t)
            phys = wl.block_table[b, t // ps]
            assert np.array_equal(k[phys, :, t % ps].view(np.uint8), kt.view(np.uint8))
            assert np.array_equal(v[phys, :, t % ps].view(np.uint8), vt.view(np.uint8))
        for p in range(-(-L // ps)):
            phys = wl.block_table[b, p]
            assert np.array_equal(mn[phys], ref_mn[phys]) and np.array_equal(mx[phys], ref_mx[phys])


def test_append_updates_min_max_in_closed_form():
    # For a page holding t >= 1 tokens, appending key x gives
    # min' = min(min, x) and max' = max(max, x) channel by channel; into an
    # empty slot 0 it gives min' = max' = x (the page is that one token).
    spec = W.tiny_spec(dtype="f32", batch=2, hq=2, hkv=1, context=40, ps=16, index=42)
    wl = W.generate(spec, context_lens=[21, 32])
    mn, mx = oracle.minmax_build("f32", wl.k_cache, wl.block_table, wl.context_lens)
    rng = _rng(43)
    kn = (rng.standard_normal((2, 1, 128)) * 2 + 0.01).astype(np.float32)
    vn = rng.standard_normal((2, 1, 128)).astype(np.float32)
    _, _, mn2, mx2 = oracle.append_token("f32", kn, vn, wl.k_cache, wl.v_cache, wl.block_table,
                                         wl.context_lens, mn, mx)
    p0 = wl.block_table[0, 1]                         # sequence 0: slot 5 of page 1
    assert np.array_equal(mn2[p0, 0], np.minimum(mn[p0, 0], kn[0, 0]))
    assert np.array_equal(mx2[p0, 0], np.maximum(mx[p0, 0], kn[0, 0]))
    p1 = wl.block_table[1, 2]                         # sequence 1: slot 0 of page 2
    assert np.array_equal(mn2[p1, 0], kn[1, 0].astype(np.float64))
    assert np.array_equal(mx2[p1, 0], kn[1, 0].astype(np.float64))
    # entries of other pages are untouched
    others = [i for i in range(spec.num_phys_pages) if i not in (p0, p1)]
    assert np.array_equal(mn2[others], mn[others], equal_nan=True)


def test_append_writes_one_row_per_sequence_and_skips_out_of_range_lengths():
    spec = W.tiny_spec(dtype="bf16", batch=3, hq=2, hkv=2, context=48, ps=16, index=44)
    wl = W.generate(spec, context_lens=[48, 10, 1])
    kn, vn = W.new_tokens(spec, 0)
    ctx = np.array([48, 10, -1], dtype=np.int32)       # full row, a middle slot, invalid
    k2, v2, _, _ = oracle.append_token("bf16", kn, vn, wl.k_cache, wl.v_cache, wl.block_table, ctx)
    changed_k = np.argwhere((k2 != wl.k_cache).any(axis=-1))
    changed_v = np.argwhere((v2 != wl.v_cache).any(axis=-1))
    phys = wl.block_table[1, 0]
    expect = {(int(phys), h, 10) for h in range(2)}
    assert {tuple(map(int, r)) for r in changed_k} <= expect
    assert {tuple(map(int, r)) for r in changed_v} <= expect
    assert np.array_equal(k2[phys, :, 10], kn[1]) and np.array_equal(v2[phys, :, 10], vn[1])


def test_attention_after_appending_to_an_empty_sequence_is_the_new_value():
    spec = W.tiny_spec(dtype="f16", batch=1, hq=4, hkv=2, context=32, ps=16, index=45)
    wl = W.generate(spec)
    kn, vn = W.new_tokens(spec, 3)
    k2, v2, _, _ = oracle.append_token("f16", kn, vn, wl.k_cache, wl.v_cache, wl.block_table,
                                       np.array([0], dtype=np.int32))
    out = oracle.attention("f16", wl.q, k2, v2, wl.block_table, np.array([1], dtype=np.int32),
                           wl.scale)
    for h in range(4):
        assert np.array_equal(out[0, h], vn[0, h // 2].astype(np.float64))


# ---------------------------------------------------------------- mean-key index

def _all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    vals = (bits[finite] << 16).view(np.float32).astype(np.float64)
    order = np.argsort(vals, kind="stable")
    return vals[order], bits[finite][order]


def _bf16_nearest_even(x):
    """Brute force: the nearest finite bf16 value, ties to the even pattern."""
    vals, bits = _all_bf16_values()
    keep = np.concatenate([[True], np.diff(vals) != 0])        # one of +0/-0
    vals, bits = vals[keep], bits[keep]
    out = np.empty_like(x)
    for i, v in enumerate(x.reshape(-1)):
        j = np.searchsorted(vals, v)
        cands = [c for c in (j - 1, j) if 0 <= c < vals.size]
        best = min(cands, key=lambda c: (abs(vals[c] - v), int(bits[c]) & 1))
        out.reshape(-1)[i] = vals[best]
    return out


def test_round_to_dtype_matches_library_and_brute_force():
    rng = _rng(80)
    x = np.concatenate([rng.standard_normal(400) * 10.0 ** rng.integers(-3, 4, 400),
                        [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8),  # bf16 ties
                         1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,                    # f16 ties
                         1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, 0.0,               # f32 ties
                         3e-6, -7.7e-7, 2.0 ** -25, 3 * 2.0 ** -25, 5e-5,           # f16 subnormal
                         1e-40, -3.3e-39, 2.0 ** -134, 3 * 2.0 ** -134]])          # f32/bf16 subnormal
    assert np.array_equal(oracle.round_to_dtype("f16", x), x.astype(np.float16).astype(np.float64))
    assert np.array_equal(oracle.round_to_dtype("f32", x), x.astype(np.float32).astype(np.float64))
    assert np.array_equal(oracle.round_to_dtype("bf16", x), _bf16_nearest_even(x))
    # the ties themselves: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7 -> 1 (even)
    assert oracle.round_to_dtype("bf16", np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert oracle.round_to_dtype("bf16", np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_page_mean_matches_numpy_mean_then_rounding(dtype):
    rng = _rng(81)
    for ps, n in [(16, 16), (16, 7), (64, 64), (64, 33), (16, 1)]:
        x = rng.standard_normal((ps, 128)).astype(np.float32)
        page = W.to_storage(x, dtype)
        got = oracle.page_mean(dtype, page, n)
        m = W.storage_to_f64(page, dtype)[:n].mean(axis=0)
        if dtype == "f16":
            ref = m.astype(np.float16).astype(np.float64)
        elif dtype == "f32":
            ref = m.astype(np.float32).astype(np.float64)
        else:
            ref = _bf16_nearest_even(m)
        assert np.array_equal(got, ref), (ps, n)


def _format_table(dtype):
    """Every finite value of a 16-bit format as exact fp64, sorted, with its
    bit pattern (-0.0 dropped: +0.0 stands for zero)."""
    bits = np.arange(65536, dtype=np.uint32)
    if dtype == "bf16":
        finite = ((bits >> 7) & 0xFF) != 0xFF
        vals = (bits[finite] << 16).view(np.float32).astype(np.float64)
    else:
        finite = ((bits >> 10) & 0x1F) != 0x1F
        vals = bits[finite].astype(np.uint16).view(np.float16).astype(np.float64)
    b = bits[finite]
    keep = ~((vals == 0) & (b >= 0x8000))
    order = np.argsort(vals[keep], kind="stable")
    return vals[keep][order], b[keep][order]


def _exact_mean_rounded(dtype, xs, table=None):
    """The mean of xs (exact stored values) from rational arithmetic, rounded
    to the nearest value of the type by brute force over its neighbours, ties
    to the even bit pattern; an exact zero is +0 unless every x is -0, a
    non-zero mean that rounds to zero keeps its sign."""
    from fractions import Fraction
    import math
    mu = sum(Fraction(float(x)) for x in xs) / len(xs)
    if mu == 0:
        return -0.0 if all(x == 0 and math.copysign(1.0, x) < 0 for x in xs) else 0.0
    if dtype == "f32":
        c = np.float32(float(mu))
        cands = {c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))}
        cands = [(float(v), int(np.float32(v).view(np.uint32))) for v in cands if np.isfinite(v)]
    else:
        vals, bits = table
        j = int(np.searchsorted(vals, float(mu)))
        cands = [(float(vals[i]), int(bits[i])) for i in range(j - 2, j + 2) if 0 <= i < vals.size]
    best = min(cands, key=lambda vb: (abs(Fraction(vb[0]) - mu), vb[1] & 1))
    v = best[0]
    return math.copysign(0.0, float(mu)) if v == 0 else v


def _wide_values(rng, dtype, n):
    """n stored values whose magnitudes span the type's whole range, with
    cancelling pairs, as a storage array [n]."""
    lo, hi = {"f16": (-24, 15), "bf16": (-133, 127), "f32": (-149, 127)}[dtype]
    e = rng.integers(lo, hi + 1, n)
    x = np.ldexp(rng.uniform(1.0, 2.0, n), e) * rng.choice([-1.0, 1.0], n)
    if n >= 3:                       # a large pair that cancels exactly, around the rest
        x[0] = np.ldexp(1.5, hi - 2) * np.sign(x[0])
        x[-1] = -x[0]
    x = np.clip(x, -6e4 if dtype == "f16" else -3e38, 6e4 if dtype == "f16" else 3e38)
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "f32":
        return x.astype(np.float32)
    return W.f32_to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_page_mean_is_the_correctly_rounded_exact_mean_on_wide_pages(dtype):
    # keys spanning every binade of the type, cancelling pairs, partial pages:
    # an fp32 (or fp64) running sum is not exact here, the exact mean is
    rng = _rng(83)
    table = None if dtype == "f32" else _format_table(dtype)
    for n in (1, 2, 3, 5, 16, 33, 64, 128):
        cols = np.stack([_wide_values(rng, dtype, n) for _ in range(24)], axis=1)   # [n][24]
        got = oracle.page_mean(dtype, cols, n)
        vals = W.storage_to_f64(cols, dtype)
        for c in range(cols.shape[1]):
            ref = _exact_mean_rounded(dtype, vals[:, c], table)
            assert got[c] == ref and np.signbit(got[c]) == np.signbit(ref), (n, c)


def test_page_mean_hand_worked_edge_cases():
    import math
    f16 = lambda *v: np.array(v, dtype=np.float16).reshape(-1, 1)
    mean = lambda a, dt="f16": float(oracle.page_mean(dt, a, a.shape[0])[0])
    # the f16 extremes cancel; a third of the smallest subnormal rounds to +0
    assert mean(f16(65504, -65504, 2.0 ** -24)) == 0.0
    # two thirds of it rounds up to the smallest subnormal
    assert mean(f16(65504, -65504, 2.0 ** -23)) == 2.0 ** -24
    # halfway between two subnormals: ties to the even one
    assert mean(f16(2.0 ** -24, 2.0 ** -23)) == 2.0 ** -23     # 1.5 units -> 2 units
    assert mean(f16(2.0 ** -24, 0.0)) == 0.0                   # 0.5 units -> 0
    # signed zeros: -0 only when every key is -0; a negative mean keeps its sign
    assert math.copysign(1.0, mean(f16(-0.0, -0.0))) < 0
    assert math.copysign(1.0, mean(f16(-0.0, 0.0))) > 0
    assert math.copysign(1.0, mean(f16(1.0, -1.0))) > 0
    assert math.copysign(1.0, mean(f16(-(2.0 ** -24), 0.0, 0.0))) < 0
    # bf16: 2^100 cancels, the 2^-100 terms between survive exactly
    b = W.f32_to_bf16_bits(np.array([2.0 ** 100, 2.0 ** -100, 2.0 ** -100, -(2.0 ** 100)],
                                    dtype=np.float32)).reshape(-1, 1)
    assert mean(b, "bf16") == 2.0 ** -101
    # fp32: 2^60 + 1 - 2^60 = 1, over 3 tokens; 1/3 to the nearest fp32
    f = np.array([2.0 ** 80, 1.0, -(2.0 ** 80)], dtype=np.float32).reshape(-1, 1)
    assert mean(f, "f32") == float(np.float32(1.0 / 3.0))


def test_mean_build_indirection_partial_pages_and_identical_keys():
    spec = W.tiny_spec(dtype="f16", batch=3, hq=4, hkv=2, context=70, ps=16, index=82)
    wl = W.generate(spec, context_lens=[70, 33, 16])
    phys = wl.block_table[1, 2]                      # page 2 of row 1 holds 1 token
    wl.k_cache[phys, :, 1:] = np.float16(1e4)        # garbage past the valid token
    mean = oracle.mean_build("f16", wl.k_cache, wl.block_table, wl.context_lens)
    k = W.storage_to_f64(wl.k_cache, "f16")
    for b in range(3):
        L = int(wl.context_lens[b])
        for p in range(-(-L // 16)):
            n = min(16, L - p * 16)
            ph = wl.block_table[b, p]
            ref = k[ph, :, :n].mean(axis=1).astype(np.float16).astype(np.float64)
            assert np.array_equal(mean[ph], ref)
    assert np.array_equal(mean[phys], k[phys, :, 0])     # one token: the mean is the key
    used = {int(wl.block_table[b, p]) for b in range(3)
            for p in range(-(-int(wl.context_lens[b]) // 16))}
    unused = [i for i in range(spec.num_phys_pages) if i not in used]
    assert np.isnan(mean[unused]).all()


def test_mean_scores_gqa_head_and_block_table_by_brute_force():
    spec = W.tiny_spec(dtype="bf16", batch=2, hq=6, hkv=2, context=50, ps=16, index=83)
    wl = W.generate(spec, context_lens=[50, 17])
    mean = oracle.mean_build("bf16", wl.k_cache, wl.block_table, wl.context_lens)
    s = oracle.mean_scores("bf16", wl.q, mean, wl.block_table, wl.context_lens, 16)
    q = W.storage_to_f64(wl.q, "bf16")
    for b in range(2):
        P = -(-int(wl.context_lens[b]) // 16)
        for h in range(6):
            for p in range(spec.max_pages):
                if p >= P:
                    assert s[b, h, p] == -np.inf
                    continue
                ref = float(np.dot(q[b, h], mean[wl.block_table[b, p], h // 3]))
                assert abs(s[b, h, p] - ref) <= 1e-12 * (1 + abs(ref))


def test_mean_score_of_a_single_token_page_is_q_dot_k():
    spec = W.tiny_spec(dtype="bf16", batch=1, hq=2, hkv=1, context=17, ps=16, index=84)
    wl = W.generate(spec)
    mean = oracle.mean_build("bf16", wl.k_cache, wl.block_table, wl.context_lens)
    s = oracle.mean_scores("bf16", wl.q, mean, wl.block_table, wl.context_lens, 16)
    kk = W.storage_to_f64(wl.k_cache[wl.block_table[0, 1], 0, 0], "bf16")
    for h in range(2):
        qq = W.storage_to_f64(wl.q[0, h], "bf16")
        assert abs(s[0, h, 1] - float(np.dot(qq, kk))) <= 1e-12 * (1 + abs(s[0, h, 1]))


# ---------------------------------------------------------------- page window

def _window_scenario(seed, steps, B=2, Hq=4, Hkv=2, maxP=40, K=5, C=14, ps=16, drift=0.3):
    """Selections and scores of a slowly drifting query: each step keeps most
    of the previous step's high-scoring pages."""
    rng = _rng(seed)
    base = rng.standard_normal((B, Hq, maxP))
    ctx = np.array([maxP * ps - 3, (maxP - 9) * ps], dtype=np.int32)
    out = []
    for _ in range(steps):
        base = base + drift * rng.standard_normal(base.shape)
        s = np.round(base, 2)
        for b in range(B):
            s[b, :, -(-int(ctx[b]) // ps):] = -np.inf
        idx = oracle.topk(s, ctx, ps, K)
        out.append((idx, s))
    return ctx, out


def _needed(idx, ctx, ps, b, kvh, G):
    P = -(-int(ctx[b]) // ps)
    sel = idx[b, kvh * G:(kvh + 1) * G].reshape(-1)
    return {int(p) for p in sel if 0 <= p < P}


def test_window_repeated_selection_hits_everything():
    ctx, steps = _window_scenario(90, 1)
    idx, s = steps[0]
    w = oracle.Window(2, 2, 40, 14)
    _, st1 = w.step(idx, s, ctx, 16)
    assert (st1[..., 1] == 0).all() and (st1[..., 2] == st1[..., 0]).all()
    fetch, st2 = w.step(idx, s, ctx, 16)
    assert (st2[..., 1] == st2[..., 0]).all() and (st2[..., 3] == 0).all()
    for b in range(2):
        P = -(-int(ctx[b]) // 16)
        for kvh in range(2):
            need = _needed(idx, ctx, 16, b, kvh, 2)
            # only the growing last page is fetched again, and only if needed
            assert [p for p, _ in fetch[b][kvh]] == ([P - 1] if P - 1 in need else [])


def test_window_invariants_and_lookahead_eviction_by_brute_force():
    # The policy's defining properties, checked on every step of a drifting
    # sequence (not its implementation: no eviction order or slot assignment
    # is recomputed here): every page the step needs is in the window
    # afterwards; pages that stay keep their slots; only as many pages are
    # evicted as the misses need beyond the free slots; none of them is
    # needed; each evicted page has a look-ahead score (the group's best
    # score for it this step, stale pages -inf) no higher than any page that
    # stays without being needed; the misses land in the freed slots.
    ctx, steps = _window_scenario(91, 12)
    C, G, ps = 14, 2, 16
    w = oracle.Window(2, 2, 40, C)
    evictions = 0
    for idx, s in steps:
        before = w.slot_page.copy()
        fetch, st = w.step(idx, s, ctx, ps)
        for b in range(2):
            P = -(-int(ctx[b]) // ps)
            for kvh in range(2):
                need = _needed(idx, ctx, ps, b, kvh, G)
                old, new = before[b, kvh], w.slot_page[b, kvh]
                cached_old = {int(p) for p in old if p >= 0}
                cached_new = {int(p) for p in new if p >= 0}
                misses = need - cached_old
                free = {i for i in range(C) if old[i] < 0}
                assert need <= cached_new
                kept = [i for i in range(C) if old[i] >= 0 and int(old[i]) in cached_new]
                assert all(new[i] == old[i] for i in kept)
                evicted = cached_old - cached_new
                assert not evicted & need
                assert len(evicted) == max(0, len(misses) - len(free))
                evictions += len(evicted)

                def look_ahead(p):
                    return -np.inf if p >= P else max(float(s[b, h, p])
                                                      for h in range(kvh * G, kvh * G + G))
                stay_unneeded = cached_old - evicted - need
                for e in evicted:
                    for k in stay_unneeded:
                        assert look_ahead(e) <= look_ahead(k)
                miss_slots = {i for i in range(C) if new[i] >= 0 and int(new[i]) in misses}
                freed = free | {i for i in range(C) if old[i] >= 0 and int(old[i]) in evicted}
                assert len(miss_slots) == len(misses) and miss_slots <= freed
                # the two maps are inverse to each other
                for slot, p in enumerate(new):
                    if p >= 0:
                        assert w.page_slot[b, kvh, p] == slot
                assert (w.page_slot[b, kvh] >= 0).sum() == len(cached_new)
                # every miss is fetched; of the pages already there only the
                # row's last page (which may have grown) is fetched again
                fetched = {p for p, _ in fetch[b][kvh]}
                assert misses <= fetched and fetched - misses <= {P - 1} & need
                assert tuple(st[b, kvh]) == (len(need), len(need) - len(misses), len(fetched),
                                             len(evicted))
    assert evictions > 0  # the scenario exercises the eviction at all


def test_window_large_enough_never_evicts():
    ctx, steps = _window_scenario(92, 10)
    w = oracle.Window(2, 2, 40, 40)
    seen = [[set(), set()], [set(), set()]]
    for idx, s in steps:
        _, st = w.step(idx, s, ctx, 16)
        assert (st[..., 3] == 0).all()
        for b in range(2):
            for kvh in range(2):
                seen[b][kvh] |= _needed(idx, ctx, 16, b, kvh, 2)
                assert {int(p) for p in w.slot_page[b, kvh] if p >= 0} == seen[b][kvh]


def test_window_evicts_stale_pages_first_and_refuses_overflow():
    # slots hold pages 0 and 5; the row now has 4 pages, so page 5 is stale
    # (-inf) and goes before page 0 although page 0 scores lowest of the rest
    w = oracle.Window(1, 1, 8, 2)
    w.slot_page[0, 0] = [0, 5]
    w.page_slot[0, 0, 0], w.page_slot[0, 0, 5] = 0, 1
    s = np.array([[[-5.0, 1.0, 2.0, 3.0, -np.inf, -np.inf, -np.inf, -np.inf]]])
    _, st = w.step(np.array([[[3, -1]]], dtype=np.int32), s, np.array([4 * 16], np.int32), 16)
    assert list(w.slot_page[0, 0]) == [0, 3] and tuple(st[0, 0]) == (1, 0, 1, 1)
    assert w.page_slot[0, 0, 5] == -1 and w.page_slot[0, 0, 3] == 1
    # two misses: page 0 (lowest score, not needed) is evicted next
    _, st = w.step(np.array([[[1, 3]]], dtype=np.int32), s, np.array([4 * 16], np.int32), 16)
    assert list(w.slot_page[0, 0]) == [1, 3] and tuple(st[0, 0]) == (2, 1, 2, 1)
    with pytest.raises(ValueError):
        w.step(np.array([[[0, 1, 2]]], dtype=np.int32), s, np.array([4 * 16], np.int32), 16)
