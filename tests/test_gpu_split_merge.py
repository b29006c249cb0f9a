"""Merging the split partials of the attention against the fp64 oracle.

When one (sequence, kv head, head chunk) is split over several CTAs, each
split keeps its own running maximum, weight sum and weighted V sum, and the
combine kernel rescales and adds them (the streaming softmax of KVDrive,
section 2.3 step (3), carried across splits).  Cases: 2, 3, 13-16, more than
32 and more than 64 splits (the combine's preloaded first 16 or 64 partials,
then its rounds of 32 weights), 16-bit data on tensor cores and on CUDA
cores, fp32; a workspace filled with garbage before the first call; repeated
calls on one workspace, which must agree bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from offloaded_kv_cache_gb300 import kvsparse as kv
from offloaded_kv_cache_gb300 import workloads as W
from offloaded_kv_cache_gb300.pipeline import DecodeLayer
from parity_util import ATOL

pytestmark = pytest.mark.gpu

# (dtype, batch, q heads, kv heads, context, page size, k, least splits)
CASES = [
    ("bf16", 1, 4, 1, 65536, 16, 1024, 33),   # one group over many CTAs
    ("f16", 1, 2, 1, 32768, 16, 512, 33),     # CUDA-core consumers, 2 heads a CTA
    ("f32", 1, 4, 1, 32768, 32, 256, 33),
    ("bf16", 4, 32, 8, 4096, 16, 64, 2),      # the 32k workload's shape of plan
    ("bf16", 8, 16, 4, 2048, 16, 48, 2),
    ("f16", 16, 8, 8, 1024, 16, 16, 2),
    ("f32", 8, 8, 8, 2048, 16, 32, 2),
]


@pytest.fixture(autouse=True)
def _lib(kvlib):
    kv.kv_debug_config(-1, 2_000_000_000)
    yield


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c[:7])))
def test_split_merge_matches_the_oracle(case):
    dtype, batch, hq, hkv, context, ps, k, least = case
    spec = W.tiny_spec(dtype=dtype, batch=batch, hq=hq, hkv=hkv, context=context, ps=ps,
                       topk=k, index=4100 + CASES.index(case))
    # ragged rows: the first is full, the others end inside a page
    ctx = [context] + [context - 1 - 37 * i for i in range(1, batch)]
    wl = W.generate(spec, context_lens=ctx)
    layer = DecodeLayer(wl, topk=k)
    S = kv.kv_attn_num_splits(layer.shape, k)
    assert S >= least, S

    mn, mx = oracle.minmax_build(dtype, wl.k_cache, wl.block_table, wl.context_lens)
    s = oracle.scores(dtype, wl.q, mn, mx, wl.block_table, wl.context_lens, ps)
    idx = oracle.topk(s, wl.context_lens, ps, k)
    ref = oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                           wl.context_lens, wl.scale, indices=idx)

    layer.workspace.fill_(0xFF)  # nothing may depend on the workspace's old contents
    idx_d = torch.from_numpy(idx).cuda()
    outs = []
    for _ in range(3):
        layer.sparse_attn(indices=idx_d)
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        outs.append(layer.out.cpu().numpy().copy())
    err = np.abs(outs[0] - ref).max()
    assert err <= ATOL[dtype], (S, err)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_dense_call_between_sparse_calls_leaves_the_merge_intact():
    # the dense call's partials share the workspace with the sparse call's
    # union lists; each call writes all it reads
    spec = W.tiny_spec(dtype="bf16", batch=1, hq=4, hkv=1, context=16384, ps=16, topk=256,
                       index=4199)
    wl = W.generate(spec)
    layer = DecodeLayer(wl, topk=256)
    assert kv.kv_attn_num_splits(layer.shape, 256) > 1
    mn, mx = oracle.minmax_build("bf16", wl.k_cache, wl.block_table, wl.context_lens)
    s = oracle.scores("bf16", wl.q, mn, mx, wl.block_table, wl.context_lens, 16)
    idx = oracle.topk(s, wl.context_lens, 16, 256)
    ref = oracle.attention("bf16", wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                           wl.context_lens, wl.scale, indices=idx)
    idx_d = torch.from_numpy(idx).cuda()
    for _ in range(2):
        layer.sparse_attn(indices=idx_d)
        layer.dense_step()
        layer.sparse_attn(indices=idx_d)
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        assert np.abs(layer.out.cpu().numpy() - ref).max() <= ATOL["bf16"]
