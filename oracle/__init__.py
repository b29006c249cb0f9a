"""fp64 CPU oracle for paged decode attention with Quest-style page selection.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The oracle shares no code
with the CUDA path and never calls it; the product path never calls this.

The arithmetic lives in ``kv_oracle.c`` (plain C, fp64, one loop per
definition).  This module compiles it with gcc on first use and marshals numpy
arrays into it; it performs none of the method's arithmetic itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_LOCK = threading.Lock()
_lib = None

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}

_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc, -O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _LOCK:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.okv_decode.restype = ctypes.c_double
            lib.okv_decode.argtypes = [ctypes.c_int, _vp, ctypes.c_int64]
            lib.okv_page_minmax.restype = None
            lib.okv_page_minmax.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp,
                                            ctypes.c_int64, _f64p, _f64p]
            lib.okv_minmax_build.restype = None
            lib.okv_minmax_build.argtypes = [ctypes.c_int] + [ctypes.c_int] * 5 + [
                _vp, _i32p, _i32p, _f64p, _f64p]
            lib.okv_round_to_dtype.restype = ctypes.c_double
            lib.okv_round_to_dtype.argtypes = [ctypes.c_int, ctypes.c_double]
            lib.okv_page_mean.restype = None
            lib.okv_page_mean.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp,
                                          ctypes.c_int64, _f64p]
            lib.okv_mean_build.restype = None
            lib.okv_mean_build.argtypes = [ctypes.c_int] + [ctypes.c_int] * 5 + [
                _vp, _i32p, _i32p, _f64p]
            lib.okv_mean_scores.restype = None
            lib.okv_mean_scores.argtypes = [ctypes.c_int] * 7 + [_vp, _f64p, _i32p, _i32p, _f64p]
            lib.okv_append.restype = None
            lib.okv_append.argtypes = [ctypes.c_int] * 6 + [_vp, _vp, _vp, _vp, _i32p, _i32p,
                                                            _f64p, _f64p]
            lib.okv_page_score.restype = ctypes.c_double
            lib.okv_page_score.argtypes = [ctypes.c_int, _f64p, _f64p, _f64p]
            lib.okv_scores.restype = None
            lib.okv_scores.argtypes = [ctypes.c_int] * 7 + [
                _vp, _f64p, _f64p, _i32p, _i32p, _f64p]
            lib.okv_topk_row.restype = None
            lib.okv_topk_row.argtypes = [ctypes.c_int, _f64p, ctypes.c_int, _i32p]
            lib.okv_topk.restype = None
            lib.okv_topk.argtypes = [ctypes.c_int] * 4 + [_i32p, _f64p, ctypes.c_int, _i32p]
            lib.okv_topk_forced.restype = None
            lib.okv_topk_forced.argtypes = [ctypes.c_int] * 4 + [
                _i32p, _f64p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p]
            lib.okv_window_step.restype = ctypes.c_int
            lib.okv_window_step.argtypes = [ctypes.c_int] * 6 + [
                _i32p, _i32p, ctypes.c_int, _f64p, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p]
            lib.okv_attention_row.restype = None
            lib.okv_attention_row.argtypes = [ctypes.c_int] * 5 + [
                ctypes.c_double, _vp, ctypes.c_int64, _vp, _vp, ctypes.c_int, _i32p,
                ctypes.c_int, _i32p, ctypes.c_int, _f64p]
            lib.okv_attention.restype = None
            lib.okv_attention.argtypes = [ctypes.c_int] * 7 + [
                ctypes.c_double, _vp, _vp, _vp, _i32p, _i32p, _i32p, ctypes.c_int, _i32p,
                ctypes.c_int, ctypes.c_int, _f64p]
            lib.okv_max_threads.restype = ctypes.c_int
            lib.okv_max_threads.argtypes = []
            _lib = lib
    return _lib


def _c(a, dtype=None):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctype)


def max_threads() -> int:
    return int(_load().okv_max_threads())


def decode(dtype: str, arr: np.ndarray) -> np.ndarray:
    """Exact fp64 value of every stored element (element by element, in C)."""
    lib = _load()
    a = _c(arr)
    flat = a.reshape(-1)
    out = np.empty(flat.size, dtype=np.float64)
    base = flat.ctypes.data
    code = DTYPE_CODE[dtype]
    for i in range(flat.size):
        out[i] = lib.okv_decode(code, base, i)
    return out.reshape(a.shape)


def page_minmax(dtype: str, page: np.ndarray, n: int | None = None):
    """Channel-wise min/max over the first n tokens of a [ps][d] page."""
    lib = _load()
    a = _c(page)
    ps, d = a.shape
    n = ps if n is None else n
    mn = np.empty(d)
    mx = np.empty(d)
    lib.okv_page_minmax(DTYPE_CODE[dtype], d, n, a.ctypes.data, 0, _ptr(mn, _f64p),
                        _ptr(mx, _f64p))
    return mn, mx


def minmax_build(dtype: str, k_cache: np.ndarray, block_table: np.ndarray,
                 context_lens: np.ndarray):
    """fp64 tables mn, mx of shape [N_phys][Hkv][d]; untouched entries are NaN."""
    lib = _load()
    k = _c(k_cache)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    nphys, hkv, ps, d = k.shape
    B, maxP = bt.shape
    mn = np.full((nphys, hkv, d), np.nan)
    mx = np.full((nphys, hkv, d), np.nan)
    lib.okv_minmax_build(DTYPE_CODE[dtype], B, hkv, d, ps, maxP, k.ctypes.data, _ptr(bt, _i32p),
                         _ptr(ctx, _i32p), _ptr(mn, _f64p), _ptr(mx, _f64p))
    return mn, mx


def round_to_dtype(dtype: str, x) -> np.ndarray:
    """Nearest storage-type values (ties to even), as exact fp64 values."""
    lib = _load()
    a = np.asarray(x, dtype=np.float64)
    out = np.empty(a.shape)
    flat, of = a.reshape(-1), out.reshape(-1)
    code = DTYPE_CODE[dtype]
    for i in range(flat.size):
        of[i] = lib.okv_round_to_dtype(code, float(flat[i]))
    return out


def page_mean(dtype: str, page: np.ndarray, n: int | None = None) -> np.ndarray:
    """Channel-wise mean of the first n tokens of a [ps][d] page, rounded to dtype."""
    lib = _load()
    a = _c(page)
    ps, d = a.shape
    n = ps if n is None else n
    out = np.empty(d)
    lib.okv_page_mean(DTYPE_CODE[dtype], d, n, a.ctypes.data, 0, _ptr(out, _f64p))
    return out


def mean_build(dtype: str, k_cache: np.ndarray, block_table: np.ndarray,
               context_lens: np.ndarray) -> np.ndarray:
    """[N_phys][Hkv][d] rounded page means (fp64 values); untouched entries NaN."""
    lib = _load()
    k = _c(k_cache)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    nphys, hkv, ps, d = k.shape
    B, maxP = bt.shape
    mean = np.full((nphys, hkv, d), np.nan)
    lib.okv_mean_build(DTYPE_CODE[dtype], B, hkv, d, ps, maxP, k.ctypes.data, _ptr(bt, _i32p),
                       _ptr(ctx, _i32p), _ptr(mean, _f64p))
    return mean


def mean_scores(dtype: str, q: np.ndarray, mean: np.ndarray, block_table: np.ndarray,
                context_lens: np.ndarray, page_size: int) -> np.ndarray:
    """[B][Hq][max_pages] fp64 q . mean scores (-inf past each row's last page)."""
    lib = _load()
    q = _c(q)
    mean = _c(mean, np.float64)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    B, Hq, d = q.shape
    Hkv = mean.shape[1]
    maxP = bt.shape[1]
    out = np.empty((B, Hq, maxP))
    lib.okv_mean_scores(DTYPE_CODE[dtype], B, Hq, Hkv, d, page_size, maxP, q.ctypes.data,
                        _ptr(mean, _f64p), _ptr(bt, _i32p), _ptr(ctx, _i32p), _ptr(out, _f64p))
    return out


def append_token(dtype: str, k_new: np.ndarray, v_new: np.ndarray, k_cache: np.ndarray,
                 v_cache: np.ndarray, block_table: np.ndarray, context_lens: np.ndarray,
                 mn: np.ndarray | None = None, mx: np.ndarray | None = None):
    """Append one token per sequence at position context_lens[b].

    Returns new copies (k_cache, v_cache, mn, mx); mn/mx are the fp64 tables of
    minmax_build with the appended pages' entries recomputed (None when not
    given).  k_new / v_new are [B][Hkv][d] in the cache's storage type.
    """
    lib = _load()
    k = np.array(k_cache, copy=True, order="C")
    v = np.array(v_cache, copy=True, order="C")
    kn = _c(k_new)
    vn = _c(v_new)
    assert kn.dtype == k.dtype and vn.dtype == v.dtype
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    nphys, hkv, ps, d = k.shape
    B, maxP = bt.shape
    assert kn.shape == (B, hkv, d) and vn.shape == (B, hkv, d)
    if mn is not None:
        mn = np.array(mn, dtype=np.float64, copy=True, order="C")
        mx = np.array(mx, dtype=np.float64, copy=True, order="C")
        mn_p, mx_p = _ptr(mn, _f64p), _ptr(mx, _f64p)
    else:
        mn_p = mx_p = None
    lib.okv_append(DTYPE_CODE[dtype], B, hkv, d, ps, maxP, kn.ctypes.data, vn.ctypes.data,
                   k.ctypes.data, v.ctypes.data, _ptr(bt, _i32p), _ptr(ctx, _i32p), mn_p, mx_p)
    return k, v, mn, mx


def page_score(q: np.ndarray, mn: np.ndarray, mx: np.ndarray) -> float:
    lib = _load()
    q = _c(q, np.float64)
    mn = _c(mn, np.float64)
    mx = _c(mx, np.float64)
    return float(lib.okv_page_score(q.size, _ptr(q, _f64p), _ptr(mn, _f64p), _ptr(mx, _f64p)))


def scores(dtype: str, q: np.ndarray, mn: np.ndarray, mx: np.ndarray, block_table: np.ndarray,
           context_lens: np.ndarray, page_size: int) -> np.ndarray:
    """[B][Hq][max_pages] fp64 page scores (-inf past each row's last page)."""
    lib = _load()
    q = _c(q)
    mn = _c(mn, np.float64)
    mx = _c(mx, np.float64)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    B, Hq, d = q.shape
    Hkv = mn.shape[1]
    maxP = bt.shape[1]
    out = np.empty((B, Hq, maxP))
    lib.okv_scores(DTYPE_CODE[dtype], B, Hq, Hkv, d, page_size, maxP, q.ctypes.data,
                   _ptr(mn, _f64p), _ptr(mx, _f64p), _ptr(bt, _i32p), _ptr(ctx, _i32p),
                   _ptr(out, _f64p))
    return out


def topk_row(scores_row: np.ndarray, k: int) -> np.ndarray:
    lib = _load()
    s = _c(scores_row, np.float64)
    out = np.empty(k, dtype=np.int32)
    lib.okv_topk_row(s.size, _ptr(s, _f64p), k, _ptr(out, _i32p))
    return out


def topk(scores_arr: np.ndarray, context_lens: np.ndarray, page_size: int, k: int) -> np.ndarray:
    """[B][Hq][k] ascending selected logical pages, -1 padded."""
    lib = _load()
    s = _c(scores_arr, np.float64)
    ctx = _c(context_lens, np.int32)
    B, Hq, maxP = s.shape
    out = np.empty((B, Hq, k), dtype=np.int32)
    lib.okv_topk(B, Hq, page_size, maxP, _ptr(ctx, _i32p), _ptr(s, _f64p), k, _ptr(out, _i32p))
    return out


def topk_forced(scores_arr: np.ndarray, context_lens: np.ndarray, page_size: int, k: int,
                sink_tokens: int, local_tokens: int) -> np.ndarray:
    """[B][Hq][k] ascending selection with the sink and local pages forced in."""
    lib = _load()
    s = _c(scores_arr, np.float64)
    ctx = _c(context_lens, np.int32)
    B, Hq, maxP = s.shape
    out = np.empty((B, Hq, k), dtype=np.int32)
    lib.okv_topk_forced(B, Hq, page_size, maxP, _ptr(ctx, _i32p), _ptr(s, _f64p), k,
                        int(sink_tokens), int(local_tokens), _ptr(out, _i32p))
    return out


class Window:
    """State of the GPU-resident page window, one group per (sequence, kv head)."""

    def __init__(self, batch: int, num_kv_heads: int, max_pages: int, cache_pages: int):
        self.C = cache_pages
        self.slot_page = np.full((batch, num_kv_heads, cache_pages), -1, dtype=np.int32)
        self.page_slot = np.full((batch, num_kv_heads, max_pages), -1, dtype=np.int32)

    def step(self, indices: np.ndarray, scores_arr: np.ndarray, context_lens: np.ndarray,
             page_size: int):
        """One decode step; returns (fetch list [(page, slot)] per group, stats
        [B][Hkv][4] = needed, hits, fetched, evicted)."""
        lib = _load()
        idx = _c(indices, np.int32)
        s = _c(scores_arr, np.float64)
        ctx = _c(context_lens, np.int32)
        B, Hq, K = idx.shape
        _, Hkv, C = self.slot_page.shape
        maxP = self.page_slot.shape[2]
        fpage = np.full((B, Hkv, C), -1, dtype=np.int32)
        fslot = np.full((B, Hkv, C), -1, dtype=np.int32)
        fcount = np.zeros((B, Hkv), dtype=np.int32)
        stats = np.zeros((B, Hkv, 4), dtype=np.int32)
        rc = lib.okv_window_step(B, Hq, Hkv, page_size, maxP, C, _ptr(ctx, _i32p),
                                 _ptr(idx, _i32p), K, _ptr(s, _f64p),
                                 _ptr(self.slot_page, _i32p), _ptr(self.page_slot, _i32p),
                                 _ptr(fpage, _i32p), _ptr(fslot, _i32p), _ptr(fcount, _i32p),
                                 _ptr(stats, _i32p))
        if rc != 0:
            raise ValueError("a group needs more pages than the window holds")
        fetch = [[list(zip(fpage[b, h, :fcount[b, h]].tolist(),
                           fslot[b, h, :fcount[b, h]].tolist()))
                  for h in range(Hkv)] for b in range(B)]
        return fetch, stats


def attention(dtype: str, q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
              block_table: np.ndarray, context_lens: np.ndarray, scale: float,
              indices: np.ndarray | None = None, rows=None, nthreads: int = 0) -> np.ndarray:
    """Decode attention [B][Hq][d] in fp64 (dense when indices is None).

    rows: optional iterable of flattened (b * Hq + h) rows to compute; other
    rows of the result are NaN.
    """
    lib = _load()
    q = _c(q)
    k = _c(k_cache)
    v = _c(v_cache)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    B, Hq, d = q.shape
    nphys, Hkv, ps, _ = k.shape
    maxP = bt.shape[1]
    out = np.full((B, Hq, d), np.nan)
    if indices is not None:
        idx = _c(indices, np.int32)
        K = idx.shape[-1]
        idx_p = _ptr(idx, _i32p)
    else:
        K = 0
        idx_p = None
    if rows is not None:
        r = _c(np.asarray(list(rows), dtype=np.int32))
        rows_p, nrows = _ptr(r, _i32p), r.size
    else:
        rows_p, nrows = None, 0
    lib.okv_attention(DTYPE_CODE[dtype], B, Hq, Hkv, d, ps, maxP, float(scale), q.ctypes.data,
                      k.ctypes.data, v.ctypes.data, _ptr(bt, _i32p), _ptr(ctx, _i32p), idx_p, K,
                      rows_p, nrows, int(nthreads), _ptr(out, _f64p))
    return out
