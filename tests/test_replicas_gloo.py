"""Multi-process bookkeeping on CPU: two ranks over gloo, as the benchmark
runs one replica per GPU.  The path has no exchange step; the ranks agree on
the slowest replica's time and report the whole job's rate."""
import os
import socket

import torch.multiprocessing as mp

from offloaded_kv_cache_gb300 import replicas as R


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, times, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    w, r, local = R.rank_info()
    R.init(w, "gloo")
    R.barrier(w)
    t = R.max_over_ranks(times[r], w)
    q.put((r, w, local, t, R.whole_job_rate(100.0, t, w)))
    R.finish(w)


def test_two_gloo_ranks_agree_on_the_slowest_replica():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [0.5, 2.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    assert [g[2] for g in got] == [0, 1]
    for _, _, _, t, rate in got:
        assert t == 2.0                  # the slower replica's time on both ranks
        assert rate == 2 * 100.0 / 2.0   # both replicas' units over that time


def test_single_rank_needs_no_process_group():
    assert R.rank_info({}) == (1, 0, 0)
    assert R.rank_info({"WORLD_SIZE": "4", "RANK": "3", "LOCAL_RANK": "1"}) == (4, 3, 1)
    R.init(1)
    R.barrier(1)
    assert R.max_over_ranks(3.5, 1) == 3.5
    assert R.whole_job_rate(10.0, 2.0, 1) == 5.0
    R.finish(1)
