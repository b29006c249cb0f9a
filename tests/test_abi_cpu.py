"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "kvsparse.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(kvlib):
    names = declared_functions()
    assert {"kv_page_minmax_build", "kv_page_score", "kv_topk_select", "kv_sparse_decode_attn",
            "kv_dense_decode_attn", "kv_device_status", "kv_status_string"} <= set(names)
    for n in names:
        assert hasattr(kvlib, n), n


def test_shape_struct_layout():
    assert ctypes.sizeof(kv.kv_shape) == 40
    assert kv.kv_shape.num_phys_pages.offset == 24
    assert kv.kv_shape.kv_loc.offset == 36


def test_status_strings(kvlib):
    for code, name in [(0, "KV_OK"), (-1, "KV_ERR_INVALID_ARG"), (-2, "KV_ERR_UNSUPPORTED"),
                       (-3, "KV_ERR_LOCATION"), (-4, "KV_ERR_WORKSPACE"), (-5, "KV_ERR_CUDA"),
                       (-6, "KV_ERR_DEVICE_TIMEOUT"), (-7, "KV_ERR_BOUNDS")]:
        assert kv.kv_status_string(code) == name
    assert kv.kv_status_string(-99) == "KV_ERR_UNKNOWN"


def _shape(**kw):
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                max_pages_per_seq=4, num_phys_pages=8, dtype="bf16", kv_loc="hbm")
    base.update(kw)
    return kv.make_shape(**base)


FAKE = 0x10000  # 16-byte aligned address that is never dereferenced


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), kv.KV_ERR_UNSUPPORTED),
    (dict(page_size=48), kv.KV_ERR_UNSUPPORTED),
    (dict(page_size=256), kv.KV_ERR_UNSUPPORTED),
    (dict(dtype=7), kv.KV_ERR_UNSUPPORTED),
    (dict(num_q_heads=6, num_kv_heads=4), kv.KV_ERR_INVALID_ARG),
    (dict(batch=0), kv.KV_ERR_INVALID_ARG),
    (dict(max_pages_per_seq=0), kv.KV_ERR_INVALID_ARG),
    (dict(num_phys_pages=0), kv.KV_ERR_INVALID_ARG),
    (dict(kv_loc=5), kv.KV_ERR_INVALID_ARG),
])
def test_bad_shapes_rejected_by_every_entry_point(kvlib, kw, code):
    s = _shape(**kw)
    assert kv.kv_page_minmax_build(s, FAKE, FAKE, FAKE, FAKE, check=False) == code
    assert kv.kv_page_score(s, FAKE, FAKE, FAKE, FAKE, FAKE, check=False) == code
    assert kv.kv_page_mean_build(s, FAKE, FAKE, FAKE, FAKE, check=False) == code
    assert kv.kv_page_mean_refresh(s, FAKE, FAKE, FAKE, FAKE, check=False) == code
    assert kv.kv_page_score_mean(s, FAKE, FAKE, FAKE, FAKE, FAKE, check=False) == code
    assert kv.kv_append_token(s, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                              check=False) == code
    assert kv.kv_topk_select(s, FAKE, FAKE, 4, FAKE, check=False) == code
    assert kv.kv_topk_select_forced(s, FAKE, FAKE, 4, 4, 64, FAKE, check=False) == code
    assert kv.kv_dense_decode_attn(s, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, FAKE, 1 << 20,
                                   check=False) == code
    assert kv.kv_sparse_decode_attn(s, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 0.1, FAKE, FAKE,
                                    1 << 20, check=False) == code
    assert kv.kv_attn_workspace_bytes(s, 0) == 0


def test_null_and_misaligned_pointers_rejected(kvlib):
    s = _shape()
    assert kv.kv_page_minmax_build(s, FAKE, FAKE, FAKE, None, check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_page_minmax_build(s, FAKE, FAKE, FAKE, FAKE + 8, check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_page_score(s, FAKE + 4, FAKE, FAKE, FAKE, FAKE, check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_page_mean_build(s, FAKE, FAKE, FAKE, FAKE + 8, check=False) == \
        kv.KV_ERR_INVALID_ARG
    assert kv.kv_page_mean_refresh(s, FAKE, FAKE, FAKE, None, check=False) == \
        kv.KV_ERR_INVALID_ARG
    assert kv.kv_page_score_mean(s, FAKE, FAKE + 4, FAKE, FAKE, FAKE, check=False) == \
        kv.KV_ERR_INVALID_ARG
    assert kv.kv_page_score(s, FAKE, FAKE, FAKE + 2, FAKE, FAKE, check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_append_token(s, None, FAKE, FAKE, FAKE, FAKE, FAKE, check=False) == \
        kv.KV_ERR_INVALID_ARG
    assert kv.kv_append_token(s, FAKE, FAKE + 4, FAKE, FAKE, FAKE, FAKE, check=False) == \
        kv.KV_ERR_INVALID_ARG
    assert kv.kv_append_token(s, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, check=False) == \
        kv.KV_ERR_INVALID_ARG
    assert kv.kv_append_token(s, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE + 8,
                              check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_topk_select(s, FAKE, FAKE, 0, FAKE, check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_topk_select(s, FAKE, FAKE, 4, None, check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_topk_select_forced(s, FAKE, FAKE, 4, -1, 64, FAKE, check=False) == \
        kv.KV_ERR_INVALID_ARG
    assert kv.kv_topk_select_forced(s, FAKE, FAKE, 4, 4, -64, FAKE, check=False) == \
        kv.KV_ERR_INVALID_ARG
    assert kv.kv_dense_decode_attn(s, FAKE, FAKE, FAKE, FAKE, FAKE, float("nan"), FAKE, FAKE, 64,
                                   check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_dense_decode_attn(s, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, None, FAKE, 64,
                                   check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_sparse_decode_attn(s, FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, 0.1, FAKE, FAKE,
                                    64, check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_sparse_decode_attn(s, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0.1, FAKE, FAKE,
                                    64, check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_debug_config(-1, 0, check=False) == kv.KV_ERR_INVALID_ARG
    io = kv.kv_step_io()
    assert kv.kv_decode_step(s, io, check=False) == kv.KV_ERR_INVALID_ARG


def test_workspace_sizes_follow_the_plan(kvlib):
    # dense workspace holds split partials only; sparse adds the union lists
    for name in W.WORKLOAD_ORDER:
        spec = W.WORKLOADS[name]
        s = kv.make_shape(spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                          spec.page_size, spec.max_pages, spec.num_phys_pages, spec.dtype,
                          spec.kv_loc)
        dense = kv.kv_attn_workspace_bytes(s, 0)
        assert dense % 256 == 0
        if spec.topk:
            sparse = kv.kv_attn_workspace_bytes(s, spec.topk)
            G = spec.group
            gc = 8 if G % 8 == 0 else 4 if G % 4 == 0 else 2 if G % 2 == 0 else 1
            if spec.dtype == "f32":
                gc = 4 if G % 4 == 0 else 2 if G % 2 == 0 else 1
            umax = min(gc * spec.topk, spec.max_pages)
            groups = spec.batch * spec.num_kv_heads * (G // gc)
            assert sparse >= 2 * groups * umax * 4 + groups * 4
        assert kv.kv_topk_workspace_bytes(s, max(1, spec.topk)) == 0


def test_launch_plans_keep_their_invariants(kvlib):
    # seeded random shapes through the planner (the occupancy estimate when
    # no device is present): every split count covers its pages with at most
    # 512 per CTA and at most 1024 CTAs per (sequence, kv head, head chunk),
    # and the workspace holds the split partials, the union lists and, for
    # the page window, the fetch bits
    rng = np.random.default_rng(20261202)
    for _ in range(300):
        dtype = ["f32", "f16", "bf16"][rng.integers(3)]
        hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.choice([1, 2, 3, 4, 8, 16]))
        ps = int(rng.choice([16, 32, 64, 128]))
        B = int(rng.integers(1, 65))
        maxP = int(rng.choice([1, 7, 34, 256, 2048, 8192, 70000]))
        k = int(rng.choice([0, 1, 32, 256, 512, 5000]))
        s = kv.make_shape(B, hkv * g, hkv, 128, ps, maxP, B * maxP, dtype)
        S = kv.kv_attn_num_splits(s, k)
        if S == 0:  # refused (e.g. more cache rows than 32-bit TMA coordinates address)
            assert kv.kv_attn_workspace_bytes(s, k) == 0
            continue
        gc = (4 if g % 4 == 0 else 2 if g % 2 == 0 else 1) if dtype == "f32" else \
             (8 if g % 8 == 0 else 4 if g % 4 == 0 else 2 if g % 2 == 0 else 1)
        work = min(gc * k, maxP) if k > 0 else maxP
        assert 1 <= S <= 1024, (dtype, hkv, g, ps, B, maxP, k, S)
        assert -(-work // S) <= 512, (work, S)
        ws = kv.kv_attn_workspace_bytes(s, k)
        rows = B * hkv * g
        need = S * rows * (128 + 2) * 4 if S > 1 else 0
        if k > 0:
            groups = B * hkv * (g // gc)
            need += 2 * groups * work * 4 + groups * 4
        assert ws >= need, (ws, need)
        if k > 0:
            C = min(g * k, maxP) + 5
            wws = kv.kv_window_workspace_bytes(s, k, C)
            bits = B * hkv * -(-maxP // 32) * 4
            if wws:  # 0: the window's shared-memory bound refuses this shape
                assert wws >= bits + 2 * B * hkv * (g // gc) * work * 4
