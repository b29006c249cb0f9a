"""ctypes binding of libkvsparse (include/kvsparse.h): argument marshalling only.

Every function has the C name and argument order.  Pointer arguments take a
torch tensor (its data_ptr), a plain integer address or None; `stream` takes a
torch.cuda.Stream, a raw cudaStream_t integer or None (legacy default stream).
A non-zero status raises KvError unless check=False, in which case the status
integer is returned.  All work happens in the CUDA library: if it is missing,
loading fails loudly (there is no fallback of any kind).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvsparse.so")

KV_F32, KV_F16, KV_BF16 = 0, 1, 2
KV_LOC_HBM, KV_LOC_HOST_PINNED = 0, 1
KV_OK = 0
KV_ERR_INVALID_ARG = -1
KV_ERR_UNSUPPORTED = -2
KV_ERR_LOCATION = -3
KV_ERR_WORKSPACE = -4
KV_ERR_CUDA = -5
KV_ERR_DEVICE_TIMEOUT = -6
KV_ERR_BOUNDS = -7

DTYPE_CODE = {"f32": KV_F32, "f16": KV_F16, "bf16": KV_BF16}
LOC_CODE = {"hbm": KV_LOC_HBM, "host": KV_LOC_HOST_PINNED}


class kv_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("num_phys_pages", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("kv_loc", ctypes.c_int32)]


class kv_window(ctypes.Structure):
    _fields_ = [("cache_pages", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("cache_k", ctypes.c_void_p), ("cache_v", ctypes.c_void_p),
                ("slot_page", ctypes.c_void_p), ("page_slot", ctypes.c_void_p),
                ("stats", ctypes.c_void_p)]


class kv_step_io(ctypes.Structure):
    _fields_ = [("q_host", ctypes.c_void_p), ("context_lens_host", ctypes.c_void_p),
                ("out_host", ctypes.c_void_p), ("q", ctypes.c_void_p),
                ("context_lens", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("minmax", ctypes.c_void_p),
                ("scores", ctypes.c_void_p), ("indices", ctypes.c_void_p),
                ("k", ctypes.c_int32), ("scale", ctypes.c_float),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class KvError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} ({code})")
        self.code = code


_lib = None


def load(path: str = LIB_PATH):
    """Load libkvsparse.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    S = ctypes.POINTER(kv_shape)
    i32, sz, f32 = ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    sig = {
        "kv_page_minmax_build": (ctypes.c_int, [S, P, P, P, P, P]),
        "kv_append_token": (ctypes.c_int, [S, P, P, P, P, P, P, P, P, P]),
        "kv_page_score": (ctypes.c_int, [S, P, P, P, P, P, P]),
        "kv_page_mean_build": (ctypes.c_int, [S, P, P, P, P, P]),
        "kv_page_mean_refresh": (ctypes.c_int, [S, P, P, P, P, P]),
        "kv_page_score_mean": (ctypes.c_int, [S, P, P, P, P, P, P]),
        "kv_topk_workspace_bytes": (sz, [S, i32]),
        "kv_topk_select": (ctypes.c_int, [S, P, P, i32, P, P, sz, P]),
        "kv_topk_select_forced": (ctypes.c_int, [S, P, P, i32, i32, i32, P, P, sz, P]),
        "kv_attn_workspace_bytes": (sz, [S, i32]),
        "kv_select_workspace_bytes": (sz, [S, i32]),
        "kv_select_pages": (ctypes.c_int, [S, P, P, P, P, i32, i32, i32, P, P, sz, P]),
        "kv_sparse_decode_attn_selected": (ctypes.c_int, [S, P, P, P, P, P, i32, f32, P, P, sz,
                                                          P]),
        "kv_attn_num_splits": (i32, [S, i32]),
        "kv_sparse_decode_attn": (ctypes.c_int, [S, P, P, P, P, P, P, i32, f32, P, P, sz, P]),
        "kv_dense_decode_attn": (ctypes.c_int, [S, P, P, P, P, P, f32, P, P, sz, P]),
        "kv_window_workspace_bytes": (sz, [S, i32, i32]),
        "kv_window_reset": (ctypes.c_int, [S, ctypes.POINTER(kv_window), P]),
        "kv_sparse_decode_attn_window": (ctypes.c_int, [S, P, P, P, P, P, P, i32, P, f32, P,
                                                        ctypes.POINTER(kv_window), P, sz, P]),
        "kv_decode_step": (ctypes.c_int, [S, ctypes.POINTER(kv_step_io), P]),
        "kv_device_status": (ctypes.c_int, [P]),
        "kv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "kv_debug_config": (ctypes.c_int, [i32, ctypes.c_uint64]),
        "kv_debug_split_mode": (ctypes.c_int, [i32]),
        "kv_stream_read_probe": (ctypes.c_int, [P, sz, P, i32, P]),
        "kv_stream_read_probe_shape": (ctypes.c_int, [P, sz, P, i32, i32, i32, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def make_window(cache_pages, cache_k, cache_v, slot_page, page_slot, stats=None) -> kv_window:
    return kv_window(int(cache_pages), 0, _ptr(cache_k), _ptr(cache_v), _ptr(slot_page),
                     _ptr(page_slot), _ptr(stats))


def kv_window_workspace_bytes(shape, k, cache_pages) -> int:
    return int(load().kv_window_workspace_bytes(ctypes.byref(shape), int(k), int(cache_pages)))


def kv_window_reset(shape, win, stream=None, check=True):
    rc = load().kv_window_reset(ctypes.byref(shape), ctypes.byref(win), _stream(stream))
    return _ret(rc, "kv_window_reset", check)


def kv_sparse_decode_attn_window(shape, q, k_cache, v_cache, block_table, context_lens, indices,
                                 k, scores, scale, out, win, workspace, workspace_bytes,
                                 stream=None, check=True):
    rc = load().kv_sparse_decode_attn_window(
        ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(context_lens), _ptr(indices), int(k), _ptr(scores), float(scale), _ptr(out),
        None if win is None else ctypes.byref(win), _ptr(workspace), int(workspace_bytes),
        _stream(stream))
    return _ret(rc, "kv_sparse_decode_attn_window", check)


def kv_decode_step(shape, io, stream=None, check=True):
    rc = load().kv_decode_step(ctypes.byref(shape), ctypes.byref(io), _stream(stream))
    return _ret(rc, "kv_decode_step", check)


def make_shape(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages_per_seq,
               num_phys_pages, dtype, kv_loc="hbm") -> kv_shape:
    dt = DTYPE_CODE.get(dtype, dtype)
    loc = LOC_CODE.get(kv_loc, kv_loc)
    return kv_shape(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages_per_seq,
                    num_phys_pages, dt, loc)


def _ret(rc, where, check):
    if check and rc != KV_OK:
        raise KvError(rc, where)
    return rc


def status_string(code: int) -> str:
    return load().kv_status_string(int(code)).decode()


def kv_page_minmax_build(shape, k_cache, block_table, context_lens, minmax, stream=None,
                         check=True):
    rc = load().kv_page_minmax_build(ctypes.byref(shape), _ptr(k_cache), _ptr(block_table),
                                     _ptr(context_lens), _ptr(minmax), _stream(stream))
    return _ret(rc, "kv_page_minmax_build", check)


def kv_append_token(shape, k_new, v_new, k_cache, v_cache, block_table, context_lens,
                    context_lens_out=None, minmax=None, stream=None, check=True):
    rc = load().kv_append_token(ctypes.byref(shape), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                _ptr(v_cache), _ptr(block_table), _ptr(context_lens),
                                _ptr(context_lens_out), _ptr(minmax), _stream(stream))
    return _ret(rc, "kv_append_token", check)


def kv_page_score(shape, q, minmax, block_table, context_lens, scores, stream=None, check=True):
    rc = load().kv_page_score(ctypes.byref(shape), _ptr(q), _ptr(minmax), _ptr(block_table),
                              _ptr(context_lens), _ptr(scores), _stream(stream))
    return _ret(rc, "kv_page_score", check)


def kv_page_mean_build(shape, k_cache, block_table, context_lens, mean, stream=None, check=True):
    rc = load().kv_page_mean_build(ctypes.byref(shape), _ptr(k_cache), _ptr(block_table),
                                   _ptr(context_lens), _ptr(mean), _stream(stream))
    return _ret(rc, "kv_page_mean_build", check)


def kv_page_mean_refresh(shape, k_cache, block_table, context_lens, mean, stream=None,
                         check=True):
    rc = load().kv_page_mean_refresh(ctypes.byref(shape), _ptr(k_cache), _ptr(block_table),
                                     _ptr(context_lens), _ptr(mean), _stream(stream))
    return _ret(rc, "kv_page_mean_refresh", check)


def kv_page_score_mean(shape, q, mean, block_table, context_lens, scores, stream=None,
                       check=True):
    rc = load().kv_page_score_mean(ctypes.byref(shape), _ptr(q), _ptr(mean), _ptr(block_table),
                                   _ptr(context_lens), _ptr(scores), _stream(stream))
    return _ret(rc, "kv_page_score_mean", check)


def kv_topk_workspace_bytes(shape, k) -> int:
    return int(load().kv_topk_workspace_bytes(ctypes.byref(shape), int(k)))


def kv_topk_select(shape, scores, context_lens, k, indices, workspace=None, workspace_bytes=0,
                   stream=None, check=True):
    rc = load().kv_topk_select(ctypes.byref(shape), _ptr(scores), _ptr(context_lens), int(k),
                               _ptr(indices), _ptr(workspace), int(workspace_bytes),
                               _stream(stream))
    return _ret(rc, "kv_topk_select", check)


def kv_topk_select_forced(shape, scores, context_lens, k, sink_tokens, local_tokens, indices,
                          workspace=None, workspace_bytes=0, stream=None, check=True):
    rc = load().kv_topk_select_forced(ctypes.byref(shape), _ptr(scores), _ptr(context_lens),
                                      int(k), int(sink_tokens), int(local_tokens), _ptr(indices),
                                      _ptr(workspace), int(workspace_bytes), _stream(stream))
    return _ret(rc, "kv_topk_select_forced", check)


def kv_attn_workspace_bytes(shape, k) -> int:
    return int(load().kv_attn_workspace_bytes(ctypes.byref(shape), int(k)))


def kv_attn_num_splits(shape, k) -> int:
    return int(load().kv_attn_num_splits(ctypes.byref(shape), int(k)))


def kv_sparse_decode_attn(shape, q, k_cache, v_cache, block_table, context_lens, indices, k,
                          scale, out, workspace=None, workspace_bytes=0, stream=None,
                          check=True):
    rc = load().kv_sparse_decode_attn(ctypes.byref(shape), _ptr(q), _ptr(k_cache),
                                      _ptr(v_cache), _ptr(block_table), _ptr(context_lens),
                                      _ptr(indices), int(k), float(scale), _ptr(out),
                                      _ptr(workspace), int(workspace_bytes), _stream(stream))
    return _ret(rc, "kv_sparse_decode_attn", check)


def kv_select_workspace_bytes(shape, k) -> int:
    return int(load().kv_select_workspace_bytes(ctypes.byref(shape), int(k)))


def kv_select_pages(shape, q, minmax, block_table, context_lens, k, sink_tokens, local_tokens,
                    indices, workspace, workspace_bytes, stream=None, check=True):
    rc = load().kv_select_pages(ctypes.byref(shape), _ptr(q), _ptr(minmax), _ptr(block_table),
                                _ptr(context_lens), int(k), int(sink_tokens), int(local_tokens),
                                _ptr(indices), _ptr(workspace), int(workspace_bytes),
                                _stream(stream))
    return _ret(rc, "kv_select_pages", check)


def kv_sparse_decode_attn_selected(shape, q, k_cache, v_cache, block_table, context_lens, k,
                                   scale, out, workspace, workspace_bytes, stream=None,
                                   check=True):
    rc = load().kv_sparse_decode_attn_selected(ctypes.byref(shape), _ptr(q), _ptr(k_cache),
                                               _ptr(v_cache), _ptr(block_table),
                                               _ptr(context_lens), int(k), float(scale),
                                               _ptr(out), _ptr(workspace), int(workspace_bytes),
                                               _stream(stream))
    return _ret(rc, "kv_sparse_decode_attn_selected", check)


def kv_dense_decode_attn(shape, q, k_cache, v_cache, block_table, context_lens, scale, out,
                         workspace=None, workspace_bytes=0, stream=None, check=True):
    rc = load().kv_dense_decode_attn(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(block_table), _ptr(context_lens), float(scale),
                                     _ptr(out), _ptr(workspace), int(workspace_bytes),
                                     _stream(stream))
    return _ret(rc, "kv_dense_decode_attn", check)


def kv_device_status(stream=None) -> int:
    return int(load().kv_device_status(_stream(stream)))


def kv_status_string(code: int) -> str:
    return status_string(code)


def kv_debug_config(skip_page: int, wait_limit_ns: int, check=True):
    rc = load().kv_debug_config(int(skip_page), int(wait_limit_ns))
    return _ret(rc, "kv_debug_config", check)


def kv_debug_split_mode(mode: int, check=True):
    """Attention over kv_select_pages' lists: -1 the plan chooses; 0 per-group
    splits; 1 equal chunks of all groups' lists where possible; 2 the kernel
    chooses for every call the shapes allow."""
    rc = load().kv_debug_split_mode(int(mode))
    return _ret(rc, "kv_debug_split_mode", check)


def kv_stream_read_probe(src, nbytes, sink, stream=None, check=True):
    """Streaming 16-byte reads of `nbytes` from src (device or pinned host);
    sink is a device int64 tensor with one word per thread block."""
    rc = load().kv_stream_read_probe(_ptr(src), int(nbytes), _ptr(sink), int(sink.numel()),
                                     _stream(stream))
    return _ret(rc, "kv_stream_read_probe", check)


def kv_stream_read_probe_shape(src, nbytes, sink, blocks, threads, loads_in_flight, stream=None,
                               check=True):
    """kv_stream_read_probe with its launch shape given; sink holds one int64
    word per block."""
    rc = load().kv_stream_read_probe_shape(_ptr(src), int(nbytes), _ptr(sink), int(blocks),
                                           int(threads), int(loads_in_flight), _stream(stream))
    return _ret(rc, "kv_stream_read_probe_shape", check)
