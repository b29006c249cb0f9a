"""Decode-attention benchmark: KV GB/s, % of the bandwidth roofline, queries/s.

One step = one pass of the decode path of one layer over one batch of the
workload: dense attention for a dense-only workload; for a workload with a
page budget, kv_select_pages (page scoring, top-K selection and the group
unions in one call) and kv_sparse_decode_attn_selected (sparse attention and
the split combine).  The same step through the separate calls, the dense
pass, the index builds, the decode append, two other sparse workloads and a
batch of mixed context lengths are timed beside it and reported as
sub-objects.  The default workload is the largest that fits one GPU, a
70B-class GQA layer with 2 GiB of K/V.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Under torchrun each rank runs an independent replica of the workload on its
own GPU (the path has no exchange step); the job value is the units all ranks
processed over the slowest rank's time.  `--impl reference` times the fp64 CPU
oracle on this machine's host cores, as it stands, on a bounded sample of the
same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

DEFAULT_WORKLOAD = "70b-gqa-b8-ctx64k-ps64"
# sparse workloads also measured (shorter) beside the default one
SIDE_WORKLOADS = ("llama3.1-8b-b4-ctx32k", "llama3.1-8b-b1-ctx128k-host")
METRIC = "decode-attn KV GB/s and % of HBM (or pinned-host) roofline; queries/sec"

# DRAM traffic per launch of the dominant kernel from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by workload, with the
# hash of the kernel sources it was taken on; a changed kernel reports null.
# "bytes" is a full-size launch; "per_alg_byte" is the ratio of DRAM bytes to
# algorithmic bytes of a launch of the same kernel on a smaller case of the
# workload (its batch in "from_batch"), applied to this launch's algorithmic
# bytes (the traffic grows with the union bytes the launch reads).
NCU_TRAFFIC = {
    # attention + combine launches of kv_sparse_decode_attn_selected at batch 4
    # (543.56 + 0.52 MB attention, 2.41 MB combine, against 543.39 MB
    # algorithmic; ncu empties the caches before each launch, so the
    # combine's partials, which stay in L2 between the two launches in a
    # timed step, count as DRAM reads here)
    "70b-gqa-b8-ctx64k-ps64": {"per_alg_byte": 1.00568, "from_batch": 4,
                               "src": "ea6a1e573e38cb3c"},
    # the same two launches at full size (189.88 MB against 188.65 MB)
    "llama3.1-8b-b4-ctx32k": {"per_alg_byte": 1.00653, "from_batch": 4,
                              "src": "ea6a1e573e38cb3c"},
}


def ncu_traffic(spec, attn_bytes, batch_override=0):
    """(DRAM bytes of one attention call from the table above, how they were
    obtained), or (None, None) when there is no record for this kernel."""
    rec = NCU_TRAFFIC.get(spec.name)
    if not rec or rec.get("src") != kernel_source_hash() or batch_override:
        return None, None
    if "bytes" in rec:
        return rec["bytes"], "ncu DRAM bytes of a full-size launch"
    how = ("full-size" if rec["from_batch"] == spec.batch else f"batch-{rec['from_batch']}")
    return (round(rec["per_alg_byte"] * attn_bytes),
            f"ncu DRAM bytes of a {how} call (attention + combine launches) per algorithmic "
            "byte, times this call's algorithmic bytes")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("kv_attn.cuh", "kv_attn_core.cu", "kv_attn_mma.cu", "kv_internal.cuh"):
        with open(os.path.join(ROOT, "offloaded_kv_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def dense_bytes(spec, ctx):
    e = spec.elem_bytes
    kv = 2 * spec.num_kv_heads * int(np.sum(ctx)) * spec.head_dim * e
    q = spec.batch * spec.num_q_heads * spec.head_dim * e
    out = spec.batch * spec.num_q_heads * spec.head_dim * 4
    pages = int(np.sum(-(-np.asarray(ctx) // spec.page_size)))
    return kv + q + out + 4 * pages + 4 * spec.batch


def sparse_bytes(spec, ctx, indices, table_rows=2, lists=False, scores_in_memory=True):
    """(step bytes, attention bytes): score + select + attention over the union
    of each (sequence, kv head) group's selected pages.  table_rows: 2 for the
    min/max index, 1 for the mean-key index.  lists=False: the separate calls
    (the attention reads the selection and builds the unions); lists=True:
    kv_select_pages writes the unions as 8-byte entries that the attention
    reads instead.  scores_in_memory: the scores pass through memory (written,
    then read by the select); the one-launch selection keeps them on chip."""
    e = spec.elem_bytes
    B, Hq, Hkv, d, ps = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.page_size
    G = spec.group
    P = -(-np.asarray(ctx) // ps)
    table = int(np.sum(P)) * Hkv * table_rows * d * e        # index read by the page score
    scores = 2 * B * Hq * spec.max_pages * 4 if scores_in_memory else 0
    idx_w = B * Hq * indices.shape[-1] * 4                   # written by top-K
    kv = 0
    upages = 0
    for b in range(B):
        for kvh in range(Hkv):
            sel = indices[b, kvh * G:(kvh + 1) * G].reshape(-1)
            for p in np.unique(sel[sel >= 0]):
                n = min(ps, int(ctx[b]) - int(p) * ps)
                kv += 2 * n * d * e
                upages += 1
    q = B * Hq * d * e
    out = B * Hq * d * 4
    if lists:
        # the select also reads each scored page's block-table entry
        bt = int(np.sum(P)) * 4
        attn = 8 * upages + kv + q + out
        return table + bt + q + scores + idx_w + 8 * upages + attn, attn
    idx_r = B * Hq * indices.shape[-1] * 4                   # read by the union step
    attn = idx_r + kv + q + out
    return table + q + scores + idx_w + attn, attn


def window_measurement(spec, wl, layer, steps=128, sigma=0.5, reps=2):
    """Decode sequence of `steps` drifting queries through the page window
    (x1 and x2 of the per-step budget G*K per (sequence, kv head)) against the
    same steps read zero-copy: per-step time, hit rate, host-link bytes.

    Each variant's whole sequence is one CUDA graph; every step also writes a
    256 MiB buffer (twice the L2) so no step reads the previous step's pages
    from L2, and that flush's own time, measured alone, is subtracted.  Hit
    rates come from an eager pass over the sequence that starts from the
    state the timed replays start from."""
    import torch
    from offloaded_kv_cache_gb300 import kvsparse as kv
    from offloaded_kv_cache_gb300 import workloads as W
    from offloaded_kv_cache_gb300.pipeline import storage_to_torch
    qs = [storage_to_torch(q, spec.dtype).cuda() for q in
          W.drifting_queries(spec, wl.q, steps, sigma)]
    q0 = layer.q
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    page_bytes = 2 * spec.page_size * spec.head_dim * spec.elem_bytes   # K + V, one kv head

    def step(t, attn):
        flush.fill_(t & 0xFF)
        if attn is None:
            return
        layer.q = qs[t]
        layer.score()
        layer.select()
        attn()

    def graph_ms(attn):
        for _ in range(2):                       # eager warm-up passes
            for t in range(steps):
                step(t, attn)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            for t in range(steps):
                step(t, attn)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * steps)

    flush_ms = graph_ms(None)
    res = {"steps": steps, "query_drift_sigma": sigma, "l2_flush_ms_subtracted": round(flush_ms, 5)}
    res["zero_copy_ms_per_step"] = round(graph_ms(lambda: layer.sparse_attn()) - flush_ms, 5)
    for mult in (1, 2):
        C = mult * spec.group * layer.topk
        layer.enable_window(C)
        ms = graph_ms(lambda: layer.window_attn()) - flush_ms
        hits = need = fetched = 0
        for t in range(steps):                   # same start state as a replay
            step(t, lambda: layer.window_attn())
            torch.cuda.synchronize()
            st = layer.win_stats.cpu().numpy()
            need += int(st[..., 0].sum())
            hits += int(st[..., 1].sum())
            fetched += int(st[..., 2].sum())
        assert kv.kv_device_status() == kv.KV_OK
        res[f"x{mult}"] = {"cache_pages": C, "hit_rate": round(hits / max(1, need), 4),
                           "needed_pages_per_step": round(need / steps, 1),
                           "fetched_pages_per_step": round(fetched / steps, 1),
                           "host_MB_per_step": round(fetched / steps * page_bytes / 1e6, 3),
                           "ms_per_step": round(ms, 5)}
    layer.q = q0
    del flush
    return res


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        self.t_on = self.t_off = None
        sel = None
        try:
            import torch
            props = torch.cuda.get_device_properties(device_index)
            bus = getattr(props, "pci_bus_id", None)
            dom = getattr(props, "pci_domain_id", 0)
            dev = getattr(props, "pci_device_id", 0)
            if bus is not None:
                sel = f"{dom:08X}:{bus:02X}:{dev:02X}.0"
        except Exception:
            sel = None
        self.sel = sel

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.sel:
            cmd += ["-i", self.sel]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        inside = [r for t, r in self.rows if self.t_on and self.t_off and self.t_on <= t <= self.t_off]
        use = inside or [r for _, r in self.rows]
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in use:
            parts = [x.strip() for x in r.split(",")]
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names[1:], parts[4:8]):
                if v.lower() in ("active", "yes", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(use),
                "window": "timed region" if inside else "whole run (timed region shorter than "
                                                        "the 100 ms sampling period)"}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(spec, wl, target_s: float, nthreads: int):
    """Times the oracle over whole (b, kv-head group) row sets, enough rows
    for about target_s seconds; returns (GB/s, queries/s, seconds, sample).
    The bytes are those the GPU metric counts for the same rows: dense, the
    groups' K/V; sparse, the groups' index rows, the K/V of each group's union
    of selected pages, q and out."""
    import oracle
    dtype = spec.dtype
    G = spec.group
    groups = [(b, kvh) for b in range(spec.batch) for kvh in range(spec.num_kv_heads)]

    def rows_of(gs):
        return [b * spec.num_q_heads + kvh * G + g for b, kvh in gs for g in range(G)]

    sel = {}

    def run(gs):
        rows = rows_of(gs)
        t0 = time.perf_counter()
        if spec.topk:
            bs = sorted({b for b, _ in gs})
            for b in bs:
                mn, mx = oracle.minmax_build(dtype, wl.k_cache, wl.block_table[b:b + 1],
                                             wl.context_lens[b:b + 1])
                s = oracle.scores(dtype, wl.q[b:b + 1], mn, mx, wl.block_table[b:b + 1],
                                  wl.context_lens[b:b + 1], spec.page_size)
                idx = oracle.topk(s, wl.context_lens[b:b + 1], spec.page_size, spec.topk)
                sel[b] = idx[0]
                rb = [r - b * spec.num_q_heads for r in rows if r // spec.num_q_heads == b]
                oracle.attention(dtype, wl.q[b:b + 1], wl.k_cache, wl.v_cache,
                                 wl.block_table[b:b + 1], wl.context_lens[b:b + 1], wl.scale,
                                 indices=idx, rows=rb, nthreads=nthreads)
        else:
            oracle.attention(dtype, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                             wl.context_lens, wl.scale, rows=rows, nthreads=nthreads)
        return time.perf_counter() - t0

    n = 1
    dt = run(groups[:1])
    while dt < target_s / 4 and n < len(groups):
        n = min(len(groups), max(n + 1, int(n * max(2.0, (target_s / 2) / max(dt, 1e-3)))))
        dt = run(groups[:n])
    gs = groups[:n]
    ctx = wl.context_lens
    e, d, ps = spec.elem_bytes, spec.head_dim, spec.page_size
    if spec.topk:
        nbytes = 0
        for b, kvh in gs:
            P = -(-int(ctx[b]) // ps)
            nbytes += P * 2 * d * e                                   # index rows
            pages = np.unique(sel[b][kvh * G:(kvh + 1) * G].reshape(-1))
            for p in pages[pages >= 0]:
                nbytes += 2 * min(ps, int(ctx[b]) - int(p) * ps) * d * e
            nbytes += G * d * (e + 4)                                 # q and out
    else:
        nbytes = sum(2 * int(ctx[b]) * d * e + G * d * (e + 4) for b, _ in gs)
    gbs = nbytes / dt / 1e9
    qps = len(rows_of(gs)) / dt
    what = (f"{n} of {len(groups)} (sequence, kv head) groups = {len(rows_of(gs))} query heads, "
            f"{'score+top-K+sparse attention' if spec.topk else 'dense attention'}, "
            f"fp64 oracle, {nthreads} threads")
    return gbs, qps, dt, what


def host_link_gbs(kv, torch, sizes=(64 << 20, 512 << 20, 2 << 30), reps=5):
    """Pinned-host read bandwidth, swept: zero-copy streaming reads of a
    cudaHostAlloc buffer (kv_stream_read_probe_shape: blocks per SM, threads,
    16-byte loads in flight per thread) and cudaMemcpyAsync host->device on 1
    to 4 streams in 64 MiB chunks, over buffers of 64 MiB to 2 GiB.  Returns
    the best of each kind with its settings, the peak (the larger) and the
    sweep."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    top = max(sizes)
    host = torch.empty(top, dtype=torch.uint8, pin_memory=True)
    host.fill_(1)
    dev = torch.empty(top, dtype=torch.uint8, device="cuda")
    sink = torch.empty(8 * sms, dtype=torch.int64, device="cuda")
    streams = [torch.cuda.Stream() for _ in range(4)]
    cur = torch.cuda.current_stream()

    def t(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for _ in range(reps):
            fn()
        b.record(cur)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    sweep = []
    for nbytes in sizes:
        for bps, threads in ((1, 256), (1, 512), (1, 1024), (2, 256), (2, 512), (2, 1024),
                             (4, 256), (4, 512), (8, 256)):
            for loads in (4, 8, 16):
                ms = t(lambda: kv.kv_stream_read_probe_shape(host, nbytes, sink, bps * sms,
                                                              threads, loads, cur))
                sweep.append({"kind": "zero_copy", "bytes": nbytes, "blocks_per_sm": bps,
                              "threads": threads, "loads_in_flight": loads,
                              "GB_s": round(nbytes / ms / 1e6, 1)})
        chunk = 64 << 20
        for ns in (1, 2, 3, 4):
            def copy():
                ev = torch.cuda.Event()
                ev.record(cur)
                for i, off in enumerate(range(0, nbytes, chunk)):
                    st = streams[i % ns]
                    st.wait_event(ev)
                    with torch.cuda.stream(st):
                        dev[off:off + chunk].copy_(host[off:off + chunk], non_blocking=True)
                for st in streams[:ns]:
                    done = torch.cuda.Event()
                    done.record(st)
                    cur.wait_event(done)
            ms = t(copy)
            sweep.append({"kind": "h2d_copy", "bytes": nbytes, "streams": ns,
                          "chunk_bytes": chunk, "GB_s": round(nbytes / ms / 1e6, 1)})
    zc = max((r for r in sweep if r["kind"] == "zero_copy"), key=lambda r: r["GB_s"])
    h2d = max((r for r in sweep if r["kind"] == "h2d_copy"), key=lambda r: r["GB_s"])
    del host, dev
    return {"zero_copy": zc["GB_s"], "zero_copy_best": zc, "h2d": h2d["GB_s"], "h2d_best": h2d,
            "peak": max(zc["GB_s"], h2d["GB_s"]), "configs": len(sweep),
            "sweep_GB_s": {"zero_copy": [r["GB_s"] for r in sweep if r["kind"] == "zero_copy"],
                           "h2d_copy": [r["GB_s"] for r in sweep if r["kind"] == "h2d_copy"]}}


def link_source(link):
    zc, h = link["zero_copy_best"], link["h2d_best"]
    return (f"pinned-host read bandwidth measured in this run, the best of a sweep of "
            f"{link['configs']} settings: zero-copy streaming read {zc['GB_s']} GB/s "
            f"({zc['blocks_per_sm']} blocks/SM x {zc['threads']} threads, "
            f"{zc['loads_in_flight']} loads in flight, {zc['bytes'] >> 20} MiB), "
            f"cudaMemcpyAsync H2D {h['GB_s']} GB/s ({h['streams']} streams, "
            f"{h['chunk_bytes'] >> 20} MiB chunks, {h['bytes'] >> 20} MiB)")


R_GRAPH = 10  # steps per captured graph (amortises the graph launch itself)


def _capture(layer, copies, fn, n):
    """A CUDA graph of n consecutive calls of fn, K/V copies rotating (after
    eager warm-up calls of every copy)."""
    import torch
    for c in range(copies):
        layer.use_copy(c)
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        for i in range(n):
            layer.use_copy(i)
            fn()
    torch.cuda.synchronize()
    return g


def run_graph_steps(layer, copies, fn, k, warm, ws=1):
    """Exactly k calls of fn on the device (graphs of R_GRAPH calls, then
    single calls), after warm calls; returns device ms for the k calls."""
    import torch
    from offloaded_kv_cache_gb300 import replicas
    stream = torch.cuda.current_stream()
    g_r = _capture(layer, copies, fn, R_GRAPH)
    g_1 = _capture(layer, copies, fn, 1)
    for _ in range(max(1, warm // R_GRAPH)):
        g_r.replay()
    torch.cuda.synchronize()
    replicas.barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(k // R_GRAPH):
        g_r.replay()
    for _ in range(k % R_GRAPH):
        g_1.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    replicas.barrier(ws)
    return e0.elapsed_time(e1)


def timed_stages(layer, copies, fns, k, warm, ws=1):
    """The step (every stage once) k times, then each stage alone k times
    (its mean duration); returns (total ms of the k steps, {stage: ms})."""
    def step_fn():
        for _, f in fns:
            f()
    total = run_graph_steps(layer, copies, step_fn, k, warm, ws)
    per = {n: run_graph_steps(layer, copies, f, k, warm, ws) / k for n, f in fns} \
        if len(fns) > 1 else {fns[0][0]: total / k}
    return total, per


STEP_NAME = ("kv_select_pages (page score + top-K + group unions) + "
             "kv_sparse_decode_attn_selected (attention + split combine)")


def scores_in_memory(layer):
    """Whether kv_select_pages passes the scores through its workspace (the
    page-score kernel first) rather than keeping them on chip."""
    from offloaded_kv_cache_gb300 import kvsparse as kv
    k = layer.topk
    return kv.kv_select_workspace_bytes(layer.shape, k) > kv.kv_attn_workspace_bytes(layer.shape, k)


def kv_copies_for(spec, cap=8):
    """Rotating K/V copies so that one pass over them exceeds 4x the L2 (at
    most `cap`)."""
    l2_bytes = 129 * 2**20
    if spec.kv_loc != "hbm":
        return 1
    return max(1, min(cap, math.ceil(4 * l2_bytes / spec.kv_bytes())))


def l2_note(spec, copies):
    """How the timed steps keep K/V out of L2, for the config record."""
    mib = spec.kv_bytes() / 2**20
    if copies == 1:
        return "K/V larger than L2"
    if copies * spec.kv_bytes() >= 4 * 129 * 2**20:
        return f"{copies} rotating K/V copies of {mib:.0f} MiB each (> 4x the 129 MB L2 in total)"
    return (f"{copies} rotating K/V copies of {mib:.0f} MiB each stay in L2; `l2_rotated` times "
            f"the step over enough copies to fill 4x the L2")


def l2_rotated(spec, wl, step_fn_of, step_bytes, reps=3):
    """For a workload whose K/V fit in L2 many times over: the step over as
    many rotating K/V copies as fill 4x the L2, one CUDA graph with a step per
    copy, so no step finds its pages in L2 (the main timed steps rotate over at
    most R_GRAPH copies and so measure the L2-resident latency)."""
    import torch
    from offloaded_kv_cache_gb300.pipeline import DecodeLayer
    copies = kv_copies_for(spec, cap=256)
    layer = DecodeLayer(wl, kv_copies=copies)
    fn = step_fn_of(layer)
    ms = run_graph_steps_n(layer, copies, fn, copies, reps)
    del layer
    torch.cuda.empty_cache()
    return {"copies": copies, "bytes_rotated": int(copies * spec.kv_bytes()),
            "ms_per_step": round(ms, 5), "GB_s": round(step_bytes / (ms * 1e-3) / 1e9, 2)}


def run_graph_steps_n(layer, copies, fn, n, reps):
    """Device ms per call of fn over one graph of n calls rotating the K/V
    copies, replayed reps times after one warm replay."""
    import torch
    g = _capture(layer, copies, fn, n)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * n)


def cpu_model() -> str:
    """The host CPU's model string (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        fields = dict(l.split(":", 1) for l in out.splitlines() if ":" in l)
        fields = {k.strip(): v.strip() for k, v in fields.items()}
        name = fields.get("Model name") or fields.get("BIOS Model name")
        if name:
            vendor = fields.get("Vendor ID", "")
            return f"{vendor} {name}".strip()
    except (OSError, subprocess.SubprocessError, ValueError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def side_workload(name, steps, warm):
    """The sparse step (score + top-K + sparse attention) of another workload,
    timed like the default one, with its attention call against its own
    roofline (HBM, or the pinned-host link measured in this run)."""
    import torch
    from offloaded_kv_cache_gb300 import kvsparse as kv
    from offloaded_kv_cache_gb300 import workloads as W
    from offloaded_kv_cache_gb300.pipeline import DecodeLayer
    spec = W.WORKLOADS[name]
    wl = W.generate(spec)
    copies = kv_copies_for(spec)
    layer = DecodeLayer(wl, kv_copies=copies)
    layer.build_index()
    layer.score()
    layer.select()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    layer.select_fused()
    torch.cuda.synchronize()
    step_bytes, attn_bytes = sparse_bytes(spec, wl.context_lens, layer.indices.cpu().numpy(),
                                          lists=True, scores_in_memory=scores_in_memory(layer))
    stages = [("select_pages", layer.select_fused), ("sparse_attn", layer.sparse_attn_selected)]
    total, per = timed_stages(layer, copies, stages, steps, warm)
    ms = total / steps
    if spec.kv_loc == "host":
        link = host_link_gbs(kv, torch)
        peak, bound = link["peak"], "host-link"
        peak_source = link_source(link)
    else:
        peak, kind = measured_peaks()
        bound, peak_source = "hbm", f"MEASURED_PEAKS.json hbm_gbs ({kind})"
    achieved = attn_bytes / (per["sparse_attn"] * 1e-3) / 1e9
    res = {"step": STEP_NAME, "steps": steps,
           "ms_per_step": round(ms, 5),
           "value": round(step_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "step_bytes": int(step_bytes),
           "stages_ms": {n: round(v, 5) for n, v in per.items()},
           "attention_call": {"bound": bound, "achieved": round(achieved, 1),
                              "peak": round(peak, 1), "unit": "GB/s",
                              "frac": round(achieved / peak, 4), "bytes": int(attn_bytes),
                              "traffic": ncu_traffic(spec, attn_bytes)[0],
                              "peak_source": peak_source},
           "l2": (f"{copies} rotating K/V copies" if copies > 1 else
                  ("K/V in pinned host memory" if spec.kv_loc == "host" else "K/V larger than L2"))}
    if spec.kv_loc == "host":
        res["host_link_sweep"] = {k: link[k] for k in ("zero_copy_best", "h2d_best", "configs",
                                                        "sweep_GB_s")}
    del layer
    torch.cuda.empty_cache()
    return res

def mixed_lengths(name, steps, warm):
    """The workload with every other row at an eighth of its context (a batch
    of sequences of different lengths): the sparse step with the plan's own
    split of the attention work over the CTAs, and with each (sequence, kv
    head) group's list split over its own CTAs (kv_debug_split_mode 0)."""
    import torch
    from offloaded_kv_cache_gb300 import kvsparse as kv
    from offloaded_kv_cache_gb300 import workloads as W
    from offloaded_kv_cache_gb300.pipeline import DecodeLayer
    spec = W.WORKLOADS[name]
    ctx = [spec.context if b % 2 == 0 else spec.context // 8 for b in range(spec.batch)]
    wl = W.generate(spec, context_lens=ctx)
    copies = kv_copies_for(spec)
    layer = DecodeLayer(wl, kv_copies=copies)
    layer.build_index()
    layer.select_fused()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK
    step_bytes, attn_bytes = sparse_bytes(spec, wl.context_lens, layer.indices.cpu().numpy(),
                                          lists=True, scores_in_memory=scores_in_memory(layer))
    stages = [("select_pages", layer.select_fused), ("sparse_attn", layer.sparse_attn_selected)]
    res = {"context_lens": f"rows alternate {spec.context} and {spec.context // 8} tokens",
           "steps": steps, "step_bytes": int(step_bytes), "attention_bytes": int(attn_bytes)}
    for label, mode in (("plan", -1), ("per_group_split", 0)):
        kv.kv_debug_split_mode(mode)
        try:
            total, per = timed_stages(layer, copies, stages, steps, warm)
        finally:
            kv.kv_debug_split_mode(-1)
        ms = total / steps
        res[label] = {"ms_per_step": round(ms, 5),
                      "GB_s": round(step_bytes / (ms * 1e-3) / 1e9, 2),
                      "attention_ms": round(per["sparse_attn"], 5),
                      "attention_GB_s": round(attn_bytes / (per["sparse_attn"] * 1e-3) / 1e9, 2)}
    assert kv.kv_device_status() == kv.KV_OK
    del layer
    torch.cuda.empty_cache()
    return res

# ---------------------------------------------------------------------------

def run_reference(args, spec_name):
    from offloaded_kv_cache_gb300 import workloads as W
    import oracle
    from offloaded_kv_cache_gb300 import replicas
    ws, rank, _ = replicas.rank_info()
    if rank != 0:
        return 0
    spec = W.WORKLOADS[spec_name]
    wl = W.generate(spec)
    oracle.build()
    cores = os.cpu_count() or 1
    budget = max(0.5, min(4.0, 150.0 / max(1, args.steps + args.warmup)))
    vals = []
    what = ""
    for i in range(args.warmup + args.steps):
        gbs, qps, dt, what = oracle_sample(spec, wl, budget, cores)
        if i >= args.warmup:
            vals.append((gbs, qps, dt))
    gbs = statistics.median(v[0] for v in vals)
    qps = statistics.median(v[1] for v in vals)
    line = {"metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * statistics.median(v[2] for v in vals), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec.name, "batch": spec.batch, "q_heads": spec.num_q_heads,
                       "kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
                       "context": spec.context, "page_size": spec.page_size,
                       "topk": spec.topk, "kv_loc": spec.kv_loc, "parallelism": "replicas"},
            "queries_per_s": round(qps, 2),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "cpu_model": cpu_model(), "sample": what},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--side-workloads", default=",".join(SIDE_WORKLOADS),
                    help="comma-separated sparse workloads also timed (shorter) and reported "
                         "under `workloads`; empty for none")
    ap.add_argument("--no-mixed", action="store_true",
                    help="skip the side measurement of a batch of mixed context lengths")
    ap.add_argument("--window-steps", type=int, default=0,
                    help="profiling aid: run this many eager page-window decode steps "
                         "(x1 window, drifting queries) on the workload and exit")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling aid: the workload with this batch size instead of its own "
                         "(a smaller case of the same kernels)")
    ap.add_argument("--kernel-pass", type=int, default=0,
                    help="profiling aid: run this many eager passes over every kernel of "
                         "the path on the workload (no timing) and exit")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    if args.impl == "reference":
        return run_reference(args, args.workload)

    import torch
    from offloaded_kv_cache_gb300 import build as kbuild
    from offloaded_kv_cache_gb300 import replicas
    from offloaded_kv_cache_gb300 import kvsparse as kv
    from offloaded_kv_cache_gb300 import workloads as W
    from offloaded_kv_cache_gb300.pipeline import DecodeLayer, storage_to_torch

    ws, rank, local = replicas.rank_info()
    replicas.init(ws, "nccl", torch.device("cuda", local))
    torch.cuda.set_device(local)
    if rank == 0:
        kbuild.build()
    replicas.barrier(ws)
    kv.load()

    spec = W.WORKLOADS[args.workload]
    if args.batch > 0:
        spec = spec.with_(batch=args.batch)
    wl = W.generate(spec)
    ctx = wl.context_lens
    copies = kv_copies_for(spec)
    layer = DecodeLayer(wl, kv_copies=copies)
    stream = torch.cuda.current_stream()
    sparse = spec.topk > 0

    if args.window_steps > 0:  # profiling aid, no timing
        layer.build_index()
        layer.enable_window(spec.group * max(1, spec.topk))
        for q in W.drifting_queries(spec, wl.q, args.window_steps, 0.5):
            layer.q = storage_to_torch(q, spec.dtype).cuda()
            layer.score()
            layer.select()
            layer.window_attn()
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        print(json.dumps({"window_steps": args.window_steps,
                          "last_step_stats": layer.win_stats.sum(dim=(0, 1)).tolist()}))
        return 0

    if args.kernel_pass > 0:  # profiling aid, no timing
        # one pass, in this order: index build, the one-call selection and the
        # attention over its lists (select, attention, combine), page score,
        # top-K, sparse attention (union, attention, combine), forced top-K,
        # mean index build and score, page-window update and attention, dense
        # attention, append
        kn, vn = W.new_tokens(spec, 0)
        kn = storage_to_torch(kn, spec.dtype).cuda()
        vn = storage_to_torch(vn, spec.dtype).cuda()
        ctx_last = (layer.context_lens - 1).contiguous()  # full rows: rewrite the last slot
        if sparse:
            layer.enable_window(spec.group * spec.topk)
        for _ in range(args.kernel_pass):
            layer.build_index()
            if sparse:
                layer.select_fused()
                layer.sparse_attn_selected()
                layer.score()
                layer.select()
                layer.sparse_attn()
                layer.select(sink_tokens=4, local_tokens=64)
                layer.build_mean_index()
                layer.score_mean()
                layer.score()
                layer.select()
                layer.window_attn()
            layer.dense_step()
            kv.kv_append_token(layer.shape, kn, vn, layer.k_cache, layer.v_cache,
                               layer.block_table, ctx_last, None, layer.minmax, stream)
        torch.cuda.synchronize()
        assert kv.kv_device_status() == kv.KV_OK
        info = {"kernel_pass": args.kernel_pass, "workload": spec.name}
        if sparse:
            layer.select_fused()
            torch.cuda.synchronize()
            idx = layer.indices.cpu().numpy()
            _, attn_b = sparse_bytes(spec, ctx, idx, lists=True,
                                     scores_in_memory=scores_in_memory(layer))
            info["sparse_attention_bytes"] = int(attn_b)
        print(json.dumps(info))
        return 0

    # index (built once per page; timed separately below)
    layer.build_index()
    if sparse:
        layer.select_fused()
    torch.cuda.synchronize()
    assert kv.kv_device_status() == kv.KV_OK

    splits = kv.kv_attn_num_splits(layer.shape, spec.topk if sparse else 0)
    if sparse:
        idx_np = layer.indices.cpu().numpy()
        sim = scores_in_memory(layer)
        step_bytes, attn_bytes = sparse_bytes(spec, ctx, idx_np, lists=True,
                                              scores_in_memory=sim)
        stages = [("select_pages", layer.select_fused),
                  ("sparse_attn", layer.sparse_attn_selected)]
        # selection (the page-score kernel too when the scores pass through
        # memory), attention, combine
        launches_per_step = (2 if sim else 1) + 1 + (1 if splits > 1 else 0)
        dominant = "sparse_attn"
    else:
        step_bytes = dense_bytes(spec, ctx)
        stages = [("dense_attn", layer.dense_step)]
        launches_per_step = 1 + (1 if splits > 1 else 0)
        attn_bytes = step_bytes
        dominant = "dense_attn"

    def run_steps(fn, k, warm):
        return run_graph_steps(layer, copies, fn, k, warm, ws)

    def timed(fns, k, warm):
        return timed_stages(layer, copies, fns, k, warm, ws)

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    clocks.mark_on()
    total_ms, per_stage = timed(stages, args.steps, args.warmup)
    clocks.mark_off()
    kern_ms = per_stage[dominant]
    t_local = replicas.max_over_ranks(total_ms, ws, "cuda")
    ms_per_step = t_local / args.steps
    value = replicas.whole_job_rate(step_bytes, ms_per_step * 1e-3, ws) / 1e9
    qps = replicas.whole_job_rate(spec.batch * spec.num_q_heads, ms_per_step * 1e-3, ws)

    # sustained window for the clock record when the timed region is short;
    # every rank runs it (its barriers must pair with the other ranks'), sized
    # from the slowest rank's time so that all ranks make the same calls
    if t_local < 500:
        clocks.mark_on()
        timed(stages, max(20, int(args.steps * 600 / max(t_local, 1e-3))), 3)
        clocks.mark_off()
    clocks.stop()

    # side measurements: dense pass for sparse workloads, index build
    extra = {}
    if sparse:
        extra["stages_ms"] = {n: round(v, 5) for n, v in per_stage.items()}
        # the same step through the separate calls: kv_page_score,
        # kv_topk_select, kv_sparse_decode_attn (which builds the unions)
        n_sep = max(3, args.steps // 4)
        sep_total, sep_per = timed([("page_score", layer.score), ("topk_select", layer.select),
                                    ("sparse_attn", lambda: layer.sparse_attn())], n_sep, 3)
        sep_bytes, sep_attn = sparse_bytes(spec, ctx, layer.indices.cpu().numpy())
        extra["separate_calls"] = {
            "ms_per_step": round(sep_total / n_sep, 5),
            "GB_s": round(sep_bytes / (sep_total / n_sep * 1e-3) / 1e9, 2),
            "stages_ms": {n: round(v, 5) for n, v in sep_per.items()}}
        layer.select_fused()
        # selection with the sink (first 4 tokens) and local (last 64 tokens)
        # pages forced in, the same budget
        f_total, _ = timed([("topk_forced", lambda: layer.select(sink_tokens=4, local_tokens=64))],
                           max(3, args.steps // 4), 3)
        extra["stages_ms"]["topk_select_forced_4_64"] = round(f_total / max(3, args.steps // 4), 5)
        layer.select()
        # the mean-key index: build, score, and the sparse step it drives
        n_side = max(3, args.steps // 4)
        layer.build_mean_index()
        mb_total, _ = timed([("mean_build", layer.build_mean_index)], n_side, 3)
        ms_total, _ = timed([("mean_score", layer.score_mean)], n_side, 3)
        layer.score_mean()
        layer.select()
        torch.cuda.synchronize()
        m_step, _ = sparse_bytes(spec, ctx, layer.indices.cpu().numpy(), table_rows=1)
        mstep_total, _ = timed([("score_mean", layer.score_mean), ("topk_select", layer.select),
                                ("sparse_attn", lambda: layer.sparse_attn())], n_side, 3)
        kb = spec.num_kv_heads * int(np.sum(ctx)) * spec.head_dim * spec.elem_bytes
        pages_all = int(np.sum(-(-ctx // spec.page_size)))
        mtab = pages_all * spec.num_kv_heads * spec.head_dim * spec.elem_bytes
        extra["mean_index"] = {
            "build_ms": round(mb_total / n_side, 5),
            "build_GB_s": round((kb + mtab) / (mb_total / n_side * 1e-3) / 1e9, 2),
            "score_ms": round(ms_total / n_side, 5),
            "score_GB_s": round(mtab / (ms_total / n_side * 1e-3) / 1e9, 2),
            "sparse_step_ms": round(mstep_total / n_side, 5),
            "sparse_step_GB_s": round(m_step / (mstep_total / n_side * 1e-3) / 1e9, 2)}
        layer.score()
        layer.select()
        d_total, _ = timed([("dense_attn", layer.dense_step)], max(3, args.steps // 4), 3)
        d_ms = d_total / max(3, args.steps // 4)
        db = dense_bytes(spec, ctx)
        extra["dense"] = {"ms_per_step": round(d_ms, 4), "GB_s": round(db / (d_ms * 1e-3) / 1e9, 2)}
        if spec.kv_loc == "host":
            extra["window"] = window_measurement(spec, wl, layer)
    ib_total, _ = timed([("index_build", layer.build_index)], max(3, args.steps // 4), 3)
    ib_ms = ib_total / max(3, args.steps // 4)
    kbytes = spec.num_kv_heads * int(np.sum(ctx)) * spec.head_dim * spec.elem_bytes
    table_bytes = int(np.sum(-(-ctx // spec.page_size))) * spec.num_kv_heads * 2 * spec.head_dim * spec.elem_bytes
    extra["index_build"] = {"ms": round(ib_ms, 4),
                            "GB_s": round((kbytes + table_bytes) / (ib_ms * 1e-3) / 1e9, 2)}

    # end to end through the public API with host buffers: q and context
    # lengths copied in, the output copied out, every step
    q_host = layer.q.cpu().pin_memory()
    ctx_host = layer.context_lens.cpu().pin_memory()
    out_host = torch.empty(layer.out.shape, dtype=torch.float32, pin_memory=True)
    h2d = q_host.numel() * q_host.element_size() + ctx_host.numel() * 4
    d2h = out_host.numel() * 4

    # one kv_decode_step call per step: q and the lengths copied in from the
    # pinned host buffers, the path, the output copied back
    ios = []
    for c in range(copies):
        layer.use_copy(c)
        ios.append(layer.host_io(q_host, ctx_host, out_host, sparse))

    for i in range(args.warmup):
        layer.host_step(ios[i % copies])
    torch.cuda.synchronize()
    replicas.barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        layer.host_step(ios[i % copies])
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = replicas.max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, "cuda")
    e2e_value = replicas.whole_job_rate(step_bytes, e_ms * 1e-3, ws) / 1e9
    assert kv.kv_device_status() == kv.KV_OK

    # decode append (one token per row, min/max updated in place).  The
    # workloads are full, so the append targets each row's last slot
    # (lengths - 1) and rewrites it on every call.
    kn, vn = W.new_tokens(spec, 0)
    kn_d = storage_to_torch(kn, spec.dtype).cuda()
    vn_d = storage_to_torch(vn, spec.dtype).cuda()
    ctx_last = (layer.context_lens - 1).contiguous()

    def append_call():
        kv.kv_append_token(layer.shape, kn_d, vn_d, layer.k_cache, layer.v_cache,
                           layer.block_table, ctx_last, None, layer.minmax,
                           torch.cuda.current_stream())

    n_app = max(3, args.steps // 4)
    a_total, _ = timed([("append", append_call)], n_app, 3)
    a_ms = a_total / n_app
    a_bytes = 8 * spec.batch * spec.num_kv_heads * spec.head_dim * spec.elem_bytes
    extra["append"] = {"ms": round(a_ms, 5), "GB_s": round(a_bytes / (a_ms * 1e-3) / 1e9, 2),
                       "bytes": a_bytes}
    assert kv.kv_device_status() == kv.KV_OK

    # a workload whose K/V the graphs' rotation leaves in L2: the step over
    # enough rotating copies to defeat it, as a side measurement
    if kv_copies_for(spec, cap=256) > R_GRAPH:
        if sparse:
            def step_of(lay):
                lay.build_index()
                lay.select_fused()
                return lambda: (lay.select_fused(), lay.sparse_attn_selected())
        else:
            def step_of(lay):
                return lay.dense_step
        extra["l2_rotated"] = l2_rotated(spec, wl, step_of, step_bytes)

    # other sparse workloads, shorter runs, after the default one
    side = {}
    for name in [n for n in args.side_workloads.split(",") if n and n != spec.name]:
        side[name] = side_workload(name, max(10, min(args.steps, 200)), args.warmup)
    if side:
        extra["workloads"] = side
    if sparse and spec.batch >= 2 and not args.no_mixed:
        extra["mixed_lengths"] = mixed_lengths(spec.name, max(10, min(args.steps, 200)),
                                               args.warmup)

    peak, peak_kind = measured_peaks()
    bound = "hbm"
    peak_source = f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"
    if spec.kv_loc == "host":
        link = host_link_gbs(kv, torch)
        peak, bound = link["peak"], "host-link"
        peak_source = link_source(link)
    achieved = attn_bytes / (kern_ms * 1e-3) / 1e9
    traffic, traffic_source = ncu_traffic(spec, attn_bytes, args.batch)
    rec = NCU_TRAFFIC.get(spec.name)
    link_traffic = rec.get("link_bytes") if rec and traffic else None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        gbs, cq, dt, what = oracle_sample(spec, wl, 2.0, cores)
        gbs1, cq1, dt1, what1 = oracle_sample(spec, wl, 2.0, 1)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "cpu_model": cpu_model(), "sample": what, "seconds": round(dt, 3), "queries_per_s": round(cq, 2),
               "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "sample": what1,
                                 "seconds": round(dt1, 3), "queries_per_s": round(cq1, 2)}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": spec.dtype, "data": "synthetic",
            "config": {"workload": spec.name, "batch": spec.batch, "q_heads": spec.num_q_heads,
                       "kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
                       "context": spec.context, "page_size": spec.page_size,
                       "topk": spec.topk, "kv_loc": spec.kv_loc, "accumulate": "f32",
                       "step": (STEP_NAME if sparse else "dense attention"),
                       "l2": l2_note(spec, copies),
                       "splits": splits,
                       "timing": ("CUDA events around exactly K steps replayed as CUDA graphs of "
                                  f"{R_GRAPH} steps; per-kernel times from graphs of each stage alone"),
                       "parallelism": f"replicas x{ws}"},
            "queries_per_s": round(qps, 1),
            "sequence_steps_per_s": round(qps / spec.num_q_heads, 1),
            "roofline": {"bound": bound, "achieved": round(achieved, 1), "peak": round(peak, 1),
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "algorithmic_bytes": int(attn_bytes),
                         **({"traffic_source": traffic_source} if traffic else {}),
                         **({"link_traffic": link_traffic} if spec.kv_loc == "host" else {}),
                         "kernel": ("kv_sparse_decode_attn_selected (attention + combine)" if sparse
                                    else "kv_dense_decode_attn (attention"
                                    + (" + combine)" if splits > 1 else ")")),
                         "peak_source": peak_source},
            "clocks": clocks.summary(),
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 5)},
            "gpu_launches": launches_per_step * args.steps,
            "cpu_baseline": cpu,
            **extra,
        }
        print(json.dumps(line), flush=True)
    replicas.finish(ws)
    return 0


if __name__ == "__main__":
    sys.exit(main())
