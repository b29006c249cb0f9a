"""Device buffers and the decode steps of one paged-attention layer.

`DecodeLayer` owns the device (or pinned host) copies of one workload and the
outputs and workspaces the C ABI needs, and runs the path through the ctypes
binding:

    build_index()  -> kv_page_minmax_build
    build_mean_index(), score_mean() -> kv_page_mean_build, kv_page_score_mean
    append()       -> kv_append_token
    sparse_step()  -> kv_page_score, kv_topk_select, kv_sparse_decode_attn
    sparse_step_fused() -> kv_select_pages, kv_sparse_decode_attn_selected
    enable_window(C), window_attn() -> kv_window_reset, kv_sparse_decode_attn_window
    dense_step()   -> kv_dense_decode_attn
    host_step()    -> kv_decode_step (host q / lengths in, out back)

PyTorch is used for allocation, host<->device copies and streams only; every
step of the computation runs in libkvsparse's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import kvsparse as kv
from .workloads import Workload

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def storage_to_torch(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Host tensor with exactly the stored bits of `a`."""
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def torch_to_bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits of a tensor as an unsigned numpy array."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


class DecodeLayer:
    def __init__(self, wl: Workload, kv_loc: str | None = None, topk: int | None = None,
                 device: str = "cuda", kv_copies: int = 1):
        spec = wl.spec
        self.wl = wl
        self.spec = spec
        self.kv_loc = kv_loc or spec.kv_loc
        self.topk = spec.topk if topk is None else topk
        self.device = torch.device(device)
        self.scale = wl.scale
        self.shape = kv.make_shape(spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                                   spec.page_size, spec.max_pages, spec.num_phys_pages, spec.dtype,
                                   self.kv_loc)
        dev = self.device
        self.q = storage_to_torch(wl.q, spec.dtype).to(dev)
        self.block_table = torch.from_numpy(wl.block_table).to(dev)
        self.context_lens = torch.from_numpy(wl.context_lens).to(dev)
        # kv_copies > 1 keeps rotated copies of the caches so that a timing
        # loop can cycle through more bytes than the L2 holds
        self.k_copies, self.v_copies = [], []
        kt = storage_to_torch(wl.k_cache, spec.dtype)
        vt = storage_to_torch(wl.v_cache, spec.dtype)
        for _ in range(kv_copies):
            if self.kv_loc == "host":
                kh = torch.empty(kt.shape, dtype=kt.dtype, pin_memory=True)
                vh = torch.empty(vt.shape, dtype=vt.dtype, pin_memory=True)
                kh.copy_(kt)
                vh.copy_(vt)
                self.k_copies.append(kh)
                self.v_copies.append(vh)
            else:
                self.k_copies.append(kt.to(dev))
                self.v_copies.append(vt.to(dev))
        self.k_cache, self.v_cache = self.k_copies[0], self.v_copies[0]
        tdt = TORCH_DTYPE[spec.dtype]
        self.minmax = torch.zeros((spec.num_phys_pages, spec.num_kv_heads, 2, spec.head_dim),
                                  dtype=tdt, device=dev)
        self.scores = torch.empty((spec.batch, spec.num_q_heads, spec.max_pages),
                                  dtype=torch.float32, device=dev)
        k = max(1, self.topk)
        self.indices = torch.empty((spec.batch, spec.num_q_heads, k), dtype=torch.int32,
                                   device=dev)
        self.out = torch.empty((spec.batch, spec.num_q_heads, spec.head_dim),
                               dtype=torch.float32, device=dev)
        self.mean = None  # the mean-key index, allocated by build_mean_index()
        self.ws_dense_bytes = kv.kv_attn_workspace_bytes(self.shape, 0)
        self.ws_sparse_bytes = kv.kv_attn_workspace_bytes(self.shape, k) if self.topk else 0
        self.ws_topk_bytes = kv.kv_topk_workspace_bytes(self.shape, k)
        self.ws_select_bytes = kv.kv_select_workspace_bytes(self.shape, k) if self.topk else 0
        nbytes = max(self.ws_dense_bytes, self.ws_sparse_bytes, self.ws_topk_bytes,
                     self.ws_select_bytes, 16)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    # --- the GPU-resident page window -----------------------------------------
    def enable_window(self, cache_pages: int, stream=None):
        """Allocate and empty a window of cache_pages slots per (sequence, kv head)."""
        spec = self.spec
        C = int(cache_pages)
        tdt = TORCH_DTYPE[spec.dtype]
        shp = (spec.batch * C, spec.num_kv_heads, spec.page_size, spec.head_dim)
        self.win_k = torch.zeros(shp, dtype=tdt, device=self.device)
        self.win_v = torch.zeros(shp, dtype=tdt, device=self.device)
        self.win_slot_page = torch.empty((spec.batch, spec.num_kv_heads, C), dtype=torch.int32,
                                         device=self.device)
        self.win_page_slot = torch.empty((spec.batch, spec.num_kv_heads, spec.max_pages),
                                         dtype=torch.int32, device=self.device)
        self.win_stats = torch.zeros((spec.batch, spec.num_kv_heads, 4), dtype=torch.int32,
                                     device=self.device)
        self.window = kv.make_window(C, self.win_k, self.win_v, self.win_slot_page,
                                     self.win_page_slot, self.win_stats)
        nbytes = kv.kv_window_workspace_bytes(self.shape, max(1, self.topk), C)
        if nbytes > self.workspace.numel():
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        kv.kv_window_reset(self.shape, self.window, self._st(stream))

    def window_attn(self, indices=None, scores=None, stream=None):
        stream = self._st(stream)
        idx = self.indices if indices is None else indices
        sc = self.scores if scores is None else scores
        kv.kv_sparse_decode_attn_window(self.shape, self.q, self.k_cache, self.v_cache,
                                        self.block_table, self.context_lens, idx, idx.shape[-1],
                                        sc, self.scale, self.out, self.window, self.workspace,
                                        self.workspace.numel(), stream)

    def window_step(self, stream=None):
        stream = self._st(stream)
        self.score(stream)
        self.select(stream)
        self.window_attn(stream=stream)

    def use_copy(self, i: int):
        self.k_cache = self.k_copies[i % len(self.k_copies)]
        self.v_cache = self.v_copies[i % len(self.v_copies)]

    # --- steps (on torch's current stream unless one is given) ---------------
    @staticmethod
    def _st(stream):
        return torch.cuda.current_stream() if stream is None else stream

    def build_index(self, stream=None):
        stream = self._st(stream)
        kv.kv_page_minmax_build(self.shape, self.k_cache, self.block_table, self.context_lens,
                                self.minmax, stream)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, advance: bool = True,
               update_index: bool = True, stream=None):
        """Append one token per sequence (k_new, v_new: [B][Hkv][d] on the device).

        advance: context_lens grows by one in place; else the lengths stay and a
        repeated call rewrites the same slot.
        """
        stream = self._st(stream)
        kv.kv_append_token(self.shape, k_new, v_new, self.k_cache, self.v_cache, self.block_table,
                           self.context_lens, self.context_lens if advance else None,
                           self.minmax if update_index else None, stream)

    def build_mean_index(self, stream=None, last_only=False):
        stream = self._st(stream)
        if self.mean is None:
            spec = self.spec
            self.mean = torch.zeros((spec.num_phys_pages, spec.num_kv_heads, spec.head_dim),
                                    dtype=TORCH_DTYPE[spec.dtype], device=self.device)
        fn = kv.kv_page_mean_refresh if last_only else kv.kv_page_mean_build
        fn(self.shape, self.k_cache, self.block_table, self.context_lens, self.mean, stream)

    def score_mean(self, stream=None):
        stream = self._st(stream)
        kv.kv_page_score_mean(self.shape, self.q, self.mean, self.block_table, self.context_lens,
                              self.scores, stream)

    def score(self, stream=None):
        stream = self._st(stream)
        kv.kv_page_score(self.shape, self.q, self.minmax, self.block_table, self.context_lens,
                         self.scores, stream)

    def select(self, stream=None, sink_tokens: int = 0, local_tokens: int = 0):
        """Top-K pages per query head; sink_tokens / local_tokens force the pages
        holding the first and the most recent tokens into the selection."""
        stream = self._st(stream)
        if sink_tokens or local_tokens:
            kv.kv_topk_select_forced(self.shape, self.scores, self.context_lens, self.topk,
                                     sink_tokens, local_tokens, self.indices, self.workspace,
                                     self.workspace.numel(), stream)
        else:
            kv.kv_topk_select(self.shape, self.scores, self.context_lens, self.topk,
                              self.indices, self.workspace, self.workspace.numel(), stream)

    def sparse_attn(self, indices=None, stream=None):
        stream = self._st(stream)
        idx = self.indices if indices is None else indices
        kv.kv_sparse_decode_attn(self.shape, self.q, self.k_cache, self.v_cache, self.block_table,
                                 self.context_lens, idx, idx.shape[-1], self.scale, self.out,
                                 self.workspace, self.workspace.numel(), stream)

    def select_fused(self, stream=None, sink_tokens: int = 0, local_tokens: int = 0):
        """Page score, top-K and the group unions in one call (kv_select_pages):
        the selection lands in `indices`, the unions in the workspace for
        sparse_attn_selected()."""
        stream = self._st(stream)
        kv.kv_select_pages(self.shape, self.q, self.minmax, self.block_table, self.context_lens,
                           self.topk, sink_tokens, local_tokens, self.indices, self.workspace,
                           self.workspace.numel(), stream)

    def sparse_attn_selected(self, stream=None):
        """Attention over the pages the last select_fused() chose."""
        stream = self._st(stream)
        kv.kv_sparse_decode_attn_selected(self.shape, self.q, self.k_cache, self.v_cache,
                                          self.block_table, self.context_lens, self.topk,
                                          self.scale, self.out, self.workspace,
                                          self.workspace.numel(), stream)

    def sparse_step_fused(self, stream=None):
        stream = self._st(stream)
        self.select_fused(stream)
        self.sparse_attn_selected(stream)

    def sparse_step(self, stream=None):
        stream = self._st(stream)
        self.score(stream)
        self.select(stream)
        self.sparse_attn(stream=stream)

    def dense_step(self, stream=None):
        stream = self._st(stream)
        kv.kv_dense_decode_attn(self.shape, self.q, self.k_cache, self.v_cache, self.block_table,
                                self.context_lens, self.scale, self.out, self.workspace,
                                self.workspace.numel(), stream)

    def host_io(self, q_host: torch.Tensor, ctx_host: torch.Tensor, out_host: torch.Tensor,
                sparse: bool):
        """The kv_step_io of one decode step on these host buffers."""
        k = self.topk if sparse else 0
        return kv.kv_step_io(
            q_host.data_ptr(), ctx_host.data_ptr(), out_host.data_ptr(), self.q.data_ptr(),
            self.context_lens.data_ptr(), self.out.data_ptr(), self.k_cache.data_ptr(),
            self.v_cache.data_ptr(), self.block_table.data_ptr(),
            self.minmax.data_ptr() if sparse else None, self.scores.data_ptr() if sparse else None,
            self.indices.data_ptr() if sparse else None, k, self.scale,
            self.workspace.data_ptr(), self.workspace.numel())

    def host_step(self, io, stream=None):
        kv.kv_decode_step(self.shape, io, self._st(stream))

    # --- host views --------------------------------------------------------
    def minmax_bits(self) -> np.ndarray:
        return torch_to_bits(self.minmax)

    def mean_bits(self) -> np.ndarray:
        return torch_to_bits(self.mean)
