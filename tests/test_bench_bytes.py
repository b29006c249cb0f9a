"""The benchmark's algorithmic byte counts, the numerator of its GB/s and of
the roofline's achieved bandwidth, against totals worked out by hand.

Dense: K and V of every valid token, q, the fp32 output, one block-table
entry per page and the context lengths.  Sparse step: the page index read by
the score, the scores written and read, the selection written and read, and
the attention's q, output and K/V of the union of each GQA group's selected
pages, counting only the valid tokens of a ragged last page (the selection
and the index are Quest's, KVDrive section 2.2; the union read once per
group is this library's reading of the GQA case).
"""
import importlib.util
import os

import numpy as np

from offloaded_kv_cache_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_dense_bytes_of_the_opt_workload():
    bm = _bench()
    spec = W.WORKLOADS["opt6.7b-b32-ctx544"]
    ctx = np.full(32, 544)
    # K+V 2*32*(32*544)*128*2 = 285,212,672; q 32*32*128*2 = 262,144;
    # out 32*32*128*4 = 524,288; block table 32*34*4 = 4,352; lengths 128
    assert bm.dense_bytes(spec, ctx) == 286_003_584


def test_sparse_bytes_count_each_group_union_once_and_ragged_tails():
    bm = _bench()
    # one sequence of 40 tokens in 16-token pages (16, 16, 8 valid tokens),
    # two q heads on one kv head; head 0 picks pages 0 and 2, head 1 page 2
    spec = W.tiny_spec(dtype="bf16", batch=1, hq=2, hkv=1, context=40, ps=16, topk=2)
    idx = np.array([[[0, 2], [2, -1]]], dtype=np.int32)
    step, attn = bm.sparse_bytes(spec, np.array([40]), idx)
    # union {0, 2}: K+V of 16 + 8 tokens = 2*24*128*2 = 12,288
    # attention: + selection read 16 + q 512 + out 1,024 = 13,840
    assert attn == 13_840
    # step: + index 3*1*2*128*2 = 1,536 + q 512 + scores 2*1*2*3*4 = 48
    #       + selection written 16
    assert step == 15_952
    # the mean-key index is one row per page instead of two
    step_mean, _ = bm.sparse_bytes(spec, np.array([40]), idx, table_rows=1)
    assert step_mean == 15_952 - 768


def test_sparse_bytes_keep_groups_apart():
    bm = _bench()
    # two kv heads, two q heads each; heads 1 and 2 pick the same page but
    # belong to different groups, so it is read once for each kv head
    spec = W.tiny_spec(dtype="f16", batch=1, hq=4, hkv=2, context=64, ps=16, topk=1)
    idx = np.array([[[1], [3], [3], [3]]], dtype=np.int32)
    _, attn = bm.sparse_bytes(spec, np.array([64]), idx)
    # group 0: pages {1, 3}; group 1: page {3}; 16 valid tokens each
    kv = 3 * 2 * 16 * 128 * 2
    assert attn == kv + 4 * 4 + 4 * 128 * 2 + 4 * 128 * 4


def test_sparse_bytes_with_the_selection_lists():
    bm = _bench()
    # the case above through kv_select_pages: the unions are written as
    # 8-byte entries and read by the attention; the select reads one
    # block-table entry per scored page; the scores stay on chip
    spec = W.tiny_spec(dtype="bf16", batch=1, hq=2, hkv=1, context=40, ps=16, topk=2)
    idx = np.array([[[0, 2], [2, -1]]], dtype=np.int32)
    step, attn = bm.sparse_bytes(spec, np.array([40]), idx, lists=True, scores_in_memory=False)
    # attention: lists 2 * 8 = 16 + K/V 12,288 + q 512 + out 1,024
    assert attn == 13_840
    # step: + index 1,536 + block table 3 * 4 = 12 + q 512 + selection 16
    #       + lists written 16
    assert step == 15_932
    # with the scores through memory (the page-score kernel first): + 48
    step2, _ = bm.sparse_bytes(spec, np.array([40]), idx, lists=True, scores_in_memory=True)
    assert step2 == 15_932 + 48
