"""The native scheduler and pool (libpkv.so, host only) against the hand-worked
traces and, step by step, against the Python restatement in oracle/sched.py."""
import os

import numpy as np
import pytest

import sched_golden
from oracle.sched import Scheduler as PyScheduler
from paged_kv_cache_tables_gb300 import BlockPool, PkvError, Scheduler
from paged_kv_cache_tables_gb300._binding import PREEMPT_RECOMPUTE, PREEMPT_SWAP, SCHED_CONTINUOUS, SCHED_STATIC


class _Adapter:
    """Presents the native scheduler with the oracle's step()/stats() shape."""

    def __init__(self, **kw):
        self.s = Scheduler(**kw)

    def add(self, *a):
        self.s.add(*a)

    def step(self):
        m = self.s.step()
        if m is None:
            return None

        class M:
            pass
        out = M()
        for k, v in m.items():
            setattr(out, k, v)
        return out

    def stats(self):
        st = self.s.stats()
        st["finished"] = st["finished"]
        return st


@pytest.mark.parametrize("path", sched_golden.all_traces(), ids=os.path.basename)
def test_native_scheduler_reproduces_hand_worked_trace(path):
    from test_sched_oracle import replay
    c, _, _ = sched_golden.load(path)
    replay(_Adapter(num_blocks=c["num_blocks"], block_size=c["block_size"], max_batch=c["max_batch"],
                    max_num_batched_tokens=c["budget"], chunk=c["chunk"], max_model_len=c["max_model_len"]), path)


def run_both(seed, n=80, NB=96, max_batch=12, budget=160, chunk=48, mml=320, fail_every=0, policy="continuous",
             swap_blocks=0):
    rng = np.random.default_rng(seed)
    order = rng.permutation(NB)
    mode = "swap" if swap_blocks else "recompute"
    py = PyScheduler(NB, 16, max_batch, budget, chunk, mml, initial_order=order, policy=policy, preemption=mode,
                     swap_blocks=swap_blocks)
    nat = Scheduler(NB, 16, max_batch, budget, chunk, mml, initial_order=order,
                    policy={"continuous": SCHED_CONTINUOUS, "static": SCHED_STATIC}[policy],
                    preemption=PREEMPT_SWAP if swap_blocks else PREEMPT_RECOMPUTE, swap_blocks=swap_blocks)
    arrivals = sorted((int(rng.integers(0, 60)), rid, int(rng.integers(1, 200)), int(rng.integers(1, 120)),
                       int(rng.geometric(1 / 30))) for rid in range(n))
    i = 0
    for step in range(5000):
        while i < len(arrivals) and arrivals[i][0] <= step:
            _, rid, p, mt, eos = arrivals[i]
            py.add(rid, p, mt, eos)
            nat.add(rid, p, mt, eos)
            i += 1
        if fail_every and step % fail_every == 3:
            py.pool.fail_at = py.pool.alloc_calls + 1
            nat.inject_alloc_failure(1)
        a = py.step()
        b = nat.step()
        assert (a is None) == (b is None), "step %d" % step
        if a is not None:
            for k in ["seq_rids", "q_lens", "context_lens", "cu_seqlens", "block_tables", "slot_mapping",
                      "token_rids", "token_pos"]:
                assert np.array_equal(getattr(a, k), b[k]), "step %d field %s" % (step, k)
            assert a.num_prefill == b["num_prefill"]
            assert np.array_equal(a.finished_rids, b["finished_rids"]), "step %d finished" % step
            assert np.array_equal(a.swap_out, b["swap_out"]) and np.array_equal(a.swap_in, b["swap_in"]), step
        sa, sb = py.stats(), nat.stats()
        for k in ["free_blocks", "running", "waiting", "finished", "preemptions", "sum_running",
                  "swapped_out_blocks", "swapped_in_blocks", "free_swap_slots"]:
            assert sa[k] == sb[k], "step %d stat %s" % (step, k)
        if i == len(arrivals) and py.idle():
            break
    assert py.idle() and nat.stats()["free_blocks"] == NB
    return py


@pytest.mark.parametrize("seed", range(5))
def test_native_matches_python_restatement_step_by_step(seed):
    run_both(seed)


@pytest.mark.parametrize("seed", range(3))
def test_native_matches_python_under_memory_pressure_and_injected_failures(seed):
    py = run_both(100 + seed, NB=40, fail_every=7)
    assert py.n_preemptions > 0


def run_both_prefix(seed, NB=140, fail_every=0, policy="continuous", swap_blocks=0):
    """Native vs Python with prefix caching on a trace of requests from a few
    groups sharing page-aligned prompt heads (some prompts are a head alone)."""
    from test_sched_oracle import shared_prefix_trace
    rng = np.random.default_rng(seed)
    trace = shared_prefix_trace(rng, 70)
    order = rng.permutation(NB)
    py = PyScheduler(NB, 16, 10, 160, 48, 320, initial_order=order, policy=policy, prefix_caching=True,
                     preemption="swap" if swap_blocks else "recompute", swap_blocks=swap_blocks)
    nat = Scheduler(NB, 16, 10, 160, 48, 320, initial_order=order, prefix_caching=True,
                    policy={"continuous": SCHED_CONTINUOUS, "static": SCHED_STATIC}[policy],
                    preemption=PREEMPT_SWAP if swap_blocks else PREEMPT_RECOMPUTE, swap_blocks=swap_blocks)
    i = 0
    for step in range(5000):
        while i < len(trace) and trace[i][0] <= step:
            _, rid, toks, mt, eos = trace[i]
            py.add(rid, len(toks), mt, eos, tokens=toks)
            nat.add(rid, len(toks), mt, eos, tokens=toks)
            i += 1
        if fail_every and step % fail_every == 3:
            py.pool.fail_at = py.pool.alloc_calls + 1
            nat.inject_alloc_failure(1)
        a = py.step()
        b = nat.step()
        assert (a is None) == (b is None), "step %d" % step
        if a is not None:
            for k in ["seq_rids", "q_lens", "context_lens", "cu_seqlens", "block_tables", "slot_mapping",
                      "token_rids", "token_pos"]:
                assert np.array_equal(getattr(a, k), b[k]), "step %d field %s" % (step, k)
            assert np.array_equal(a.finished_rids, b["finished_rids"]), "step %d finished" % step
            assert np.array_equal(a.swap_out, b["swap_out"]) and np.array_equal(a.swap_in, b["swap_in"]), step
        sa, sb = py.stats(), nat.stats()
        for k in ["free_blocks", "running", "waiting", "finished", "preemptions", "prefix_hit_blocks",
                  "cached_blocks", "swapped_out_blocks", "swapped_in_blocks", "free_swap_slots"]:
            assert sa[k] == sb[k], "step %d stat %s: %s vs %s" % (step, k, sa[k], sb[k])
        if i == len(trace) and py.idle():
            break
    assert py.idle() and nat.stats()["free_blocks"] == NB and nat.stats()["cached_blocks"] == 0
    return py


@pytest.mark.parametrize("seed", range(4))
def test_native_prefix_cache_matches_python(seed):
    py = run_both_prefix(400 + seed)
    assert py.prefix_hit_blocks > 0


@pytest.mark.parametrize("seed", range(3))
def test_native_prefix_cache_matches_python_under_pressure(seed):
    py = run_both_prefix(500 + seed, NB=50, fail_every=7)
    assert py.n_preemptions > 0 and py.prefix_hit_blocks > 0
    run_both_prefix(600 + seed, NB=60, policy="static")


@pytest.mark.parametrize("seed", range(3))
def test_native_swap_preemption_matches_python(seed):
    py = run_both(700 + seed, NB=40, swap_blocks=30)
    assert py.swapped_out_blocks > 0
    py = run_both(710 + seed, NB=40, fail_every=7, swap_blocks=12)    # slots run out: some recompute
    assert py.swapped_out_blocks > 0
    py = run_both_prefix(720 + seed, NB=50, fail_every=5, swap_blocks=20)
    assert py.n_preemptions > 0


def test_native_add_tokens_checks_length():
    s = Scheduler(16, prefix_caching=True)
    with pytest.raises(ValueError):
        s.add(1, 5, 4, 4, tokens=[1, 2, 3])


@pytest.mark.parametrize("seed", range(3))
def test_native_matches_python_static_policy(seed):
    run_both(200 + seed, policy="static")
    py = run_both(300 + seed, NB=40, fail_every=7, policy="static")
    assert py.n_preemptions > 0


def test_native_rejects_unknown_policy():
    with pytest.raises(ValueError):
        Scheduler(16, policy=7)


def test_pool_stack_order_and_all_or_nothing():
    p = BlockPool(4)
    assert p.alloc(2) == [3, 2]
    with pytest.raises(PkvError):
        p.alloc(3)
    assert p.free_count() == 2          # failed alloc changed nothing
    p.free([2])
    assert p.free_list() == [0, 1, 2]
    with pytest.raises(PkvError):
        p.free([2])                     # double free rejected
    with pytest.raises(PkvError):
        p.free([9])                     # out of range rejected
    p.inject_failure(1)
    with pytest.raises(PkvError):
        p.alloc(1)
    assert p.alloc(1) == [2]


def test_pool_rejects_bad_initial_order():
    with pytest.raises(ValueError):
        BlockPool(3, [0, 0, 1])


def test_scheduler_rejects_bad_requests():
    s = Scheduler(16, max_model_len=64)
    with pytest.raises(PkvError):
        s.add(1, 0, 4, 4)
    with pytest.raises(PkvError):
        s.add(1, 64, 4, 4)
    s.add(1, 10, 4, 4)
    with pytest.raises(PkvError):
        s.add(1, 10, 4, 4)              # duplicate rid


def test_request_state_and_host_time():
    s = Scheduler(64, max_model_len=256)
    s.add(5, 20, 3, 100)
    assert s.request_state(5) == (0, 0)
    s.step()
    assert s.request_state(5) == (1, 1)
    while s.step() is not None:
        pass
    assert s.request_state(5) == (2, 3)
    assert s.request_state(99)[0] == -1
    assert s.stats()["host_ms"] >= 0.0


def test_forget_releases_finished_requests_and_reuses_their_slots():
    """A finished request can be forgotten (then unknown, its rid free again);
    a waiting or running one cannot; a long run that forgets every finished
    request emits the same steps as one that keeps them all."""
    s = Scheduler(64, max_model_len=256)
    s.add(5, 20, 3, 100)
    s.add(6, 40, 2, 100)
    with pytest.raises(PkvError):
        s.forget(5)                      # waiting
    s.step()
    with pytest.raises(PkvError):
        s.forget(5)                      # running
    while s.step() is not None:
        pass
    s.forget(5)
    assert s.request_state(5)[0] == -1 and s.request_state(6) == (2, 2)
    with pytest.raises(PkvError):
        s.forget(5)                      # already forgotten
    s.add(5, 16, 1, 100)                 # the rid is free again
    assert s.step()["seq_rids"].tolist() == [5]

    rng = np.random.default_rng(4)
    arrivals = [(int(rng.integers(0, 60)), rid, int(rng.integers(1, 90)), int(rng.integers(1, 40)))
                for rid in range(120)]
    arrivals.sort()
    traces = []
    for forget in (False, True):
        sc = Scheduler(48, max_batch=8, max_num_batched_tokens=128, chunk=48, max_model_len=256)
        i, steps = 0, []
        for step in range(4000):
            while i < len(arrivals) and arrivals[i][0] <= step:
                _, rid, p, eos = arrivals[i]
                sc.add(rid, p, 64, eos)
                i += 1
            m = sc.step()
            if m is not None:
                steps.append((m["seq_rids"].tolist(), m["slot_mapping"].tolist()))
                if forget:
                    for rid in m["finished_rids"]:
                        sc.forget(int(rid))
            if i == len(arrivals) and sc.stats()["running"] == 0 and sc.stats()["waiting"] == 0:
                break
        traces.append(steps)
    assert traces[0] == traces[1]
