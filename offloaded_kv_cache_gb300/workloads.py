"""Seeded synthetic decode-attention workloads over a paged KV cache.

This module only *draws inputs*: it holds none of the arithmetic of the method
(no min/max index, no page score, no selection, no attention).  Both the CUDA
path and the fp64 oracle consume exactly the arrays produced here, so the two
sides see identical dtype bits.

Shapes follow the workloads the KV-offloading pages evaluate on:

* OPT-6.7B, 512 prompt + 32 generated tokens, batch 32 (Dual-Blade,
  "Effect" paragraph and per-layer I/O sizes paragraph);
* Llama-3.1-8B at 32k and 128k context (KVDrive, Introduction; DirectKV,
  Experimental design);
* a 70B-class GQA layer with 64-token pages (the tiered-offload blog,
  page-granularity advice).

Layout (shared with the C ABI):

* ``q``            ``[B][Hq][d]``
* ``k_cache``      ``[N_phys][Hkv][ps][d]`` (same for ``v_cache``)
* ``block_table``  ``[B][max_pages]`` int32, logical page -> physical page
* ``context_lens`` ``[B]`` int32

Element storage: fp32 as ``float32``, fp16 as ``float16`` and bf16 as the raw
``uint16`` bit pattern.  Values are drawn as float32 N(0,1) from numpy's PCG64
(one independent stream per chunk, spawned from the workload seed so the
result does not depend on the thread count) and rounded once to the storage
type with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

SEED_BASE = 20261202

DTYPES = ("f32", "f16", "bf16")
_ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    """Shape and value recipe of one decode-attention workload."""

    name: str
    dtype: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    context: int
    page_size: int
    topk: int            # 0: dense only
    kv_loc: str          # "hbm" or "host"
    value_scale: float   # q, K, V ~ N(0, value_scale^2)
    plant: str           # "none", "tokens" or "pages"
    plant_count: int = 0         # planted tokens (plant == "tokens")
    plant_frac: float = 0.0      # fraction of pages per (b, kv head) (plant == "pages")
    plant_cos: float = 0.8       # cosine of a planted key to its group's query direction
    index: int = 0               # seed offset

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_pages(self) -> int:
        return -(-self.context // self.page_size)

    @property
    def num_phys_pages(self) -> int:
        return self.batch * self.max_pages

    @property
    def elem_bytes(self) -> int:
        return _ELEM_BYTES[self.dtype]

    def kv_bytes(self) -> int:
        """Bytes of K plus V over every valid token (the dense read)."""
        return 2 * self.batch * self.num_kv_heads * self.context * self.head_dim * self.elem_bytes

    def with_(self, **kw) -> "WorkloadSpec":
        return dataclasses.replace(self, **kw)


# The five workloads.  Names say what each is; the index only offsets the seed.
WORKLOADS = {
    "fp32-b1-ctx4k": WorkloadSpec(
        name="fp32-b1-ctx4k", dtype="f32", batch=1, num_q_heads=1, num_kv_heads=1,
        head_dim=128, context=4096, page_size=16, topk=32, kv_loc="hbm",
        value_scale=1.0, plant="tokens", plant_count=8, index=0),
    "opt6.7b-b32-ctx544": WorkloadSpec(
        name="opt6.7b-b32-ctx544", dtype="f16", batch=32, num_q_heads=32, num_kv_heads=32,
        head_dim=128, context=544, page_size=16, topk=0, kv_loc="hbm",
        value_scale=1.0 / math.sqrt(128.0), plant="none", index=1),
    "llama3.1-8b-b4-ctx32k": WorkloadSpec(
        name="llama3.1-8b-b4-ctx32k", dtype="bf16", batch=4, num_q_heads=32, num_kv_heads=8,
        head_dim=128, context=32768, page_size=16, topk=256, kv_loc="hbm",
        value_scale=1.0, plant="pages", plant_frac=0.01, index=2),
    "llama3.1-8b-b1-ctx128k-host": WorkloadSpec(
        name="llama3.1-8b-b1-ctx128k-host", dtype="bf16", batch=1, num_q_heads=32,
        num_kv_heads=8, head_dim=128, context=131072, page_size=16, topk=512, kv_loc="host",
        value_scale=1.0, plant="pages", plant_frac=0.01, index=3),
    "70b-gqa-b8-ctx64k-ps64": WorkloadSpec(
        name="70b-gqa-b8-ctx64k-ps64", dtype="bf16", batch=8, num_q_heads=64, num_kv_heads=8,
        head_dim=128, context=65536, page_size=64, topk=128, kv_loc="hbm",
        value_scale=1.0, plant="pages", plant_frac=0.005, index=4),
}
WORKLOAD_ORDER = list(WORKLOADS)


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_table: np.ndarray
    context_lens: np.ndarray

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.spec.head_dim)


# ----------------------------------------------------------------------------
# rounding to the storage type (round to nearest, ties to even)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (RNE) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f32":
        return x.copy()
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact value of stored elements as float64 (a view helper for tests)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def storage_np_dtype(dtype: str):
    return {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]


# ----------------------------------------------------------------------------
# chunked, thread-parallel normal draws
# ----------------------------------------------------------------------------

_CHUNK = 1 << 22


def _normal_storage(seed_seq: np.random.SeedSequence, n: int, scale: float, dtype: str,
                    threads: int | None = None) -> np.ndarray:
    """n values ~ N(0, scale^2) rounded to ``dtype``; one PCG64 stream per chunk."""
    out = np.empty(n, dtype=storage_np_dtype(dtype))
    nchunks = max(1, -(-n // _CHUNK))
    children = seed_seq.spawn(nchunks)

    def work(i):
        lo = i * _CHUNK
        hi = min(n, lo + _CHUNK)
        g = np.random.Generator(np.random.PCG64(children[i]))
        x = g.standard_normal(hi - lo, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[lo:hi] = to_storage(x, dtype)

    if nchunks == 1:
        work(0)
    else:
        nt = threads or min(16, os.cpu_count() or 1)
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def _unit(v: np.ndarray) -> np.ndarray:
    return v / np.linalg.norm(v, axis=-1, keepdims=True)


def generate(spec: WorkloadSpec, context_lens=None, threads: int | None = None) -> Workload:
    """Draw one workload.

    ``context_lens`` overrides the per-row lengths (each must be in
    [1, max_pages * page_size]); by default every row has ``spec.context``.
    """
    B, Hq, Hkv, d, ps = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.page_size
    maxP = spec.max_pages
    nphys = spec.num_phys_pages
    root = np.random.SeedSequence(spec.seed)
    s_q, s_k, s_v, s_perm, s_plant = root.spawn(5)

    q = _normal_storage(s_q, B * Hq * d, spec.value_scale, spec.dtype, threads).reshape(B, Hq, d)
    k = _normal_storage(s_k, nphys * Hkv * ps * d, spec.value_scale, spec.dtype,
                        threads).reshape(nphys, Hkv, ps, d)
    v = _normal_storage(s_v, nphys * Hkv * ps * d, spec.value_scale, spec.dtype,
                        threads).reshape(nphys, Hkv, ps, d)

    # Physical pages are a seeded permutation, so the block table is not the identity.
    g_perm = np.random.Generator(np.random.PCG64(s_perm))
    block_table = g_perm.permutation(nphys).astype(np.int32).reshape(B, maxP)

    if context_lens is None:
        ctx = np.full(B, spec.context, dtype=np.int32)
    else:
        ctx = np.asarray(context_lens, dtype=np.int32).copy()
        assert ctx.shape == (B,)
        assert (ctx >= 1).all() and (ctx <= maxP * ps).all()

    g = np.random.Generator(np.random.PCG64(s_plant))
    qf = storage_to_f64(q, spec.dtype)
    if spec.plant == "tokens":
        # k = 4 * q / |q| at a few seeded token positions (single-head recipe; with
        # several heads the group's mean direction is used).
        for b in range(B):
            for kvh in range(Hkv):
                qg = qf[b, kvh * spec.group:(kvh + 1) * spec.group]
                u = _unit(_unit(qg).mean(axis=0))
                pos = g.choice(int(ctx[b]), size=min(spec.plant_count, int(ctx[b])), replace=False)
                for t in pos:
                    phys = block_table[b, t // ps]
                    k[phys, kvh, t % ps] = to_storage((4.0 * u).astype(np.float32), spec.dtype)
    elif spec.plant == "pages":
        # A fraction of pages per (b, kv head) hold keys aligned with the group's
        # unit mean query direction u: k = |k_orig| (c u + sqrt(1 - c^2) w), w a
        # random unit vector orthogonal to u, for every token of the page.
        c = spec.plant_cos
        s_perp = math.sqrt(max(0.0, 1.0 - c * c))
        for b in range(B):
            P_b = -(-int(ctx[b]) // ps)
            n_plant = int(round(spec.plant_frac * P_b))
            for kvh in range(Hkv):
                qg = qf[b, kvh * spec.group:(kvh + 1) * spec.group]
                u = _unit(_unit(qg).mean(axis=0))
                pages = g.choice(P_b, size=n_plant, replace=False) if n_plant else []
                for p in pages:
                    phys = block_table[b, p]
                    ko = storage_to_f64(k[phys, kvh], spec.dtype)          # [ps][d]
                    w = g.standard_normal((ps, d))
                    w -= (w @ u)[:, None] * u[None, :]
                    w = _unit(w)
                    kn = np.linalg.norm(ko, axis=1, keepdims=True)
                    newk = kn * (c * u[None, :] + s_perp * w)
                    k[phys, kvh] = to_storage(newk.astype(np.float32), spec.dtype)
    return Workload(spec=spec, q=q, k_cache=k, v_cache=v, block_table=block_table,
                    context_lens=ctx)


def new_tokens(spec: WorkloadSpec, step: int = 0):
    """Seeded K and V rows of one appended decode token per sequence.

    Returns (k_new, v_new), each [B][Hkv][d] in the storage type, drawn like the
    cache (N(0, value_scale^2), rounded once); ``step`` selects the draw.
    """
    B, Hkv, d = spec.batch, spec.num_kv_heads, spec.head_dim
    root = np.random.SeedSequence([spec.seed, 0x0A99E7D, step])
    s_k, s_v = root.spawn(2)
    k = _normal_storage(s_k, B * Hkv * d, spec.value_scale, spec.dtype, 1).reshape(B, Hkv, d)
    v = _normal_storage(s_v, B * Hkv * d, spec.value_scale, spec.dtype, 1).reshape(B, Hkv, d)
    return k, v


def drifting_queries(spec: WorkloadSpec, q0: np.ndarray, steps: int, sigma: float):
    """Queries of `steps` consecutive decode steps starting at q0 ([B][Hq][d]
    storage values): each step adds N(0, (sigma * value_scale)^2) noise to the
    previous step's fp32 values and rounds once, so consecutive steps select
    overlapping pages (the temporal locality a page window exploits)."""
    root = np.random.SeedSequence([spec.seed, 0xD41F7, steps])
    g = np.random.Generator(np.random.PCG64(root))
    x = storage_to_f64(q0, spec.dtype).astype(np.float32)
    out = []
    for _ in range(steps):
        x = x + np.float32(sigma * spec.value_scale) * g.standard_normal(x.shape, dtype=np.float32)
        out.append(to_storage(x, spec.dtype))
    return out


def tiny_spec(dtype="bf16", batch=2, hq=4, hkv=2, d=128, context=100, ps=16, topk=3,
              scale=1.0, plant="none", index=100, **kw) -> WorkloadSpec:
    """A small workload for parity tests (several pages, ragged last page)."""
    return WorkloadSpec(name=f"tiny-{dtype}-b{batch}-h{hq}x{hkv}-ctx{context}-ps{ps}", dtype=dtype,
                        batch=batch, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                        context=context, page_size=ps, topk=topk, kv_loc="hbm",
                        value_scale=scale, plant=plant, index=index, **kw)
