"""The N > 1 path on CPU: two gloo ranks.

The path shards by sequence with no exchange step: every rank runs its own
block pool and scheduler replica on its share of the requests, and the bench
combines the ranks only through a barrier and a max over the ranks' times.
These tests run that host-side logic in two spawned processes (no GPU).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _trace(n=120, seed=7):
    """A small request trace: (arrival step, rid, prompt, max_tokens, eos)."""
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(0, 40)), rid, int(rng.integers(1, 300)), int(rng.integers(1, 90)),
             int(rng.geometric(1 / 25))) for rid in range(n)]


MML = 384


def _worker(rank, ws, port, q):
    try:
        os.environ.update(WORLD_SIZE=str(ws), RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                          MASTER_PORT=str(port))
        sys.path.insert(0, ROOT)
        import torch.distributed as dist

        import bench
        from paged_kv_cache_tables_gb300 import Scheduler

        got_ws, got_rank, _ = bench.dist_setup(None)
        assert (got_ws, got_rank) == (ws, rank)
        assert dist.get_backend() == "gloo"
        # the bench's timing reduction: every rank gets the slowest rank's time
        assert bench.max_over_ranks(1.5 + rank, ws) == 1.5 + ws - 1
        bench.barrier(ws)

        # by-sequence sharding: request i runs on rank i % ws, each rank with
        # its own pool and scheduler replica, no exchange between them
        mine = [r for r in _trace() if r[1] % ws == rank]
        sched = Scheduler(num_blocks=64, block_size=16, max_batch=8, max_num_batched_tokens=128, chunk=64,
                          max_model_len=MML)
        arrivals = sorted(mine)
        i, finished = 0, []
        for step in range(20000):
            while i < len(arrivals) and arrivals[i][0] <= step:
                _, rid, prompt, mt, eos = arrivals[i]
                sched.add(rid, prompt, mt, eos)
                i += 1
            m = sched.step()
            if m is not None:
                finished.extend(int(x) for x in m["finished_rids"])
            if i == len(arrivals) and len(finished) == len(mine):
                break
        counts = {rid: sched.request_state(rid)[1] for rid in finished}
        assert sched.stats()["free_blocks"] == 64
        gathered = [None] * ws
        dist.all_gather_object(gathered, counts)
        bench.barrier(ws)
        dist.destroy_process_group()
        q.put((rank, "ok", gathered))
    except BaseException as e:  # report to the parent instead of hanging it
        q.put((rank, "error", repr(e)))


@pytest.mark.timeout(300)
def test_two_gloo_ranks_shard_the_trace_by_sequence():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(ws):
        rank, status, payload = q.get(timeout=240)
        results[rank] = (status, payload)
    for p in procs:
        p.join(timeout=60)
    for rank in range(ws):
        assert results[rank][0] == "ok", results[rank][1]
    merged = {}
    for part in results[0][1]:
        assert not set(part) & set(merged), "a request finished on two ranks"
        merged.update(part)
    trace = _trace()
    assert sorted(merged) == sorted(r[1] for r in trace), "a request was lost"
    for _, rid, prompt, mt, eos in trace:
        assert merged[rid] == min(eos, mt, MML - prompt), rid
    # both ranks gathered the same picture
    assert results[0][1] == results[1][1]
