"""The Python scheduler restatement against hand-worked traces and invariants."""
import os

import numpy as np
import pytest

from oracle.sched import Scheduler
import sched_golden


def replay(sched, path):
    config, requests, steps = sched_golden.load(path)
    for r in requests:
        sched.add(r["rid"], r["prompt"], r["max_tokens"], r["eos_after"])
    for n in sorted(steps):
        exp = steps[n]
        meta = sched.step()
        if exp["none"]:
            assert meta is None, "step %d: expected nothing scheduled" % n
        else:
            assert meta is not None, "step %d: nothing scheduled" % n
            assert len(meta.seq_rids) == len(exp["seqs"]), "step %d" % n
            for s, e in enumerate(exp["seqs"]):
                assert meta.seq_rids[s] == e["rid"], "step %d seq %d rid" % (n, s)
                assert meta.q_lens[s] == e["q"], "step %d seq %d q" % (n, s)
                assert meta.context_lens[s] == e["ctx"], "step %d seq %d ctx" % (n, s)
                row = meta.block_tables[s]
                assert row[: len(e["table"])].tolist() == e["table"], "step %d seq %d table" % (n, s)
                assert np.all(row[len(e["table"]):] == -1)
                got = meta.slot_mapping[meta.cu_seqlens[s]: meta.cu_seqlens[s + 1]].tolist()
                assert got == e["slots"], "step %d seq %d slots" % (n, s)
        st = sched.stats()
        for k, v in exp["after"].items():
            key = {"free": "free_blocks"}.get(k, k)
            assert st[key] == v, "step %d after: %s = %d, expected %d" % (n, k, st[key], v)


@pytest.mark.parametrize("path", sched_golden.all_traces(), ids=os.path.basename)
def test_python_scheduler_reproduces_hand_worked_trace(path):
    config, _, _ = sched_golden.load(path)
    sched = Scheduler(config["num_blocks"], config["block_size"], config["max_batch"], config["budget"],
                      config["chunk"], config["max_model_len"])
    replay(sched, path)


def random_trace(seed, n=60, NB=64, max_batch=8, budget=96, chunk=32, mml=256):
    rng = np.random.default_rng(seed)
    sched = Scheduler(NB, 16, max_batch, budget, chunk, mml, initial_order=rng.permutation(NB))
    arrivals = []
    for rid in range(n):
        arrivals.append((int(rng.integers(0, 40)), rid, int(rng.integers(1, 120)),
                         int(rng.integers(1, 80)), int(rng.geometric(1 / 20))))
    arrivals.sort()
    return sched, arrivals


@pytest.mark.parametrize("seed", range(6))
def test_invariants_hold_on_random_traces(seed):
    """free + owned == pool; no block owned twice; a scheduled sequence owns
    ceil(ctx/16) or more blocks and at most ceil(known_tokens/16); waste in the
    last block <= 15 tokens; the pool is whole again when idle."""
    sched, arrivals = random_trace(seed)
    NB = sched.pool.num_blocks
    i = 0
    for step in range(3000):
        while i < len(arrivals) and arrivals[i][0] <= step:
            _, rid, p, mt, eos = arrivals[i]
            sched.add(rid, p, mt, eos)
            i += 1
        meta = sched.step()
        owned = [b for r in sched.running for b in r.blocks]
        assert len(owned) == len(set(owned))
        assert len(owned) + sched.pool.free_count() == NB
        assert not set(owned) & set(sched.pool.free_list)
        for r in sched.running:
            known = r.num_computed
            assert len(r.blocks) * 16 - known <= 15 + 16 * (-(-(r.length - known) // 16)) + 15
        if meta is not None:
            for s in range(len(meta.seq_rids)):
                ctx = int(meta.context_lens[s])
                nb = int((meta.block_tables[s] >= 0).sum())
                assert nb >= -(-ctx // 16)
                assert meta.q_lens[s] >= 1
        if i == len(arrivals) and sched.idle():
            break
    assert sched.idle()
    assert sched.pool.free_count() == NB
    assert len(sched.finished) == len(arrivals)
    for r in sched.finished:
        assert r.generated == min(r.eos_after, r.max_tokens, sched.max_model_len - r.prompt_len)


def test_waste_per_decoding_sequence_is_at_most_block_size_minus_one():
    """"Project 17" states at most 12 tokens of waste per sequence with 16-token
    pages; the bound that holds is block_size - 1 = 15."""
    sched = Scheduler(256, 16, 16, 4096, 4096, 1024)
    for rid in range(16):
        sched.add(rid, 1 + 7 * rid, 500, 10 + 13 * rid)
    worst = 0
    while not sched.idle():
        sched.step()
        for r in sched.running:
            if r.num_computed == r.length - 1:      # decode phase: cache holds all but the newest token
                waste = len(r.blocks) * 16 - r.num_computed
                assert 0 <= waste <= 15
                worst = max(worst, waste)
    assert worst == 15


def test_generates_exactly_max_tokens():
    """Basic generation (cf. "Build a pure-Python ... engine", Running and Testing)."""
    sched = Scheduler(64, 16, 2, 8192, 512, 8192)
    sched.add(7, 11, 16, 10**6)
    while not sched.idle():
        sched.step()
    assert sched.finished[0].generated == 16


def test_tiny_pool_keeps_requests_pending():
    """A 2-block pool cannot admit 3-block prompts: they stay pending, and the
    pool is untouched (no leak)."""
    sched = Scheduler(2, 16, 4, 8192, 512, 8192)
    for rid in range(10):
        sched.add(rid, 40, 128, 128)
    for _ in range(5):
        assert sched.step() is None
    st = sched.stats()
    assert st["waiting"] == 10 and st["running"] == 0 and st["free_blocks"] == 2


def test_short_requests_complete_beside_a_long_one():
    """With a 4-block pool, a long request and several short ones: the short
    ones complete (preemption by recompute lets them through)."""
    sched = Scheduler(4, 16, 4, 8192, 512, 64)
    sched.add(0, 20, 1000, 1000)
    for rid in range(1, 6):
        sched.add(rid, 5, 4, 4)
    for _ in range(400):
        sched.step()
        if sched.idle():
            break
    done = {r.rid for r in sched.finished}
    assert {1, 2, 3, 4, 5} <= done
    assert sched.idle() and sched.pool.free_count() == 4


def test_injected_alloc_failure_preempts_lifo_and_recompute_reaches_same_state():
    sched = Scheduler(64, 16, 4, 8192, 512, 8192)
    for rid in range(3):
        sched.add(rid, 16, 40, 40)
    sched.step()                     # all three admitted (3 alloc calls)
    sched.pool.fail_at = sched.pool.alloc_calls + 1    # the next growth alloc fails
    meta = sched.step()
    assert sched.n_preemptions == 1
    # the newest request (rid 2) was the victim; blocks were free again for its
    # re-admission in the same step, as a recompute prefill of prompt + 1 token
    victim = [r for r in sched.running if r.rid == 2][0]
    assert victim.preemptions == 1
    assert meta.seq_rids.tolist() == [2, 0, 1]
    assert meta.q_lens.tolist() == [17, 1, 1]
    while not sched.idle():
        sched.step()
    assert [r.generated for r in sorted(sched.finished, key=lambda r: r.rid)] == [40, 40, 40]
    assert sched.pool.free_count() == 64


def _finish_steps(policy):
    """A (prompt 3, EOS after 2), B (prompt 2, EOS after 4), C (prompt 1, EOS
    after 1), all waiting at step 0, max_batch 2, no chunking.  Worked by hand:
    both policies admit A and B at step 0; A retires after step 1 and B after
    step 3.  Continuous admission puts C into A's freed slot at step 2 (it
    retires there); static batching holds C until the batch has drained and
    admits it at step 4."""
    s = Scheduler(64, 16, max_batch=2, max_num_batched_tokens=100, chunk=100, max_model_len=64, policy=policy)
    for rid, prompt, eos in ((0, 3, 2), (1, 2, 4), (2, 1, 1)):
        s.add(rid, prompt, 10, eos)
    done = {}
    for step in range(20):
        m = s.step()
        if m is not None:
            for rid in m.finished_rids:
                done[int(rid)] = step
        if s.idle():
            break
    return done


def test_static_batching_holds_new_requests_until_the_batch_drains():
    assert _finish_steps("continuous") == {0: 1, 1: 3, 2: 2}
    assert _finish_steps("static") == {0: 1, 1: 3, 2: 4}


def test_static_batching_admits_only_when_idle():
    """Static policy: a step that starts with anything running admits
    nobody; a step that starts idle admits min(max_batch, waiting)."""
    rng = np.random.default_rng(11)
    s = Scheduler(400, 16, max_batch=6, max_num_batched_tokens=64, chunk=32, max_model_len=256, policy="static")
    arrivals = sorted((int(rng.integers(0, 30)), rid, int(rng.integers(1, 100)), int(rng.geometric(1 / 20)))
                      for rid in range(40))
    i, batches = 0, 0
    for step in range(3000):
        while i < len(arrivals) and arrivals[i][0] <= step:
            _, rid, p, eos = arrivals[i]
            s.add(rid, p, 50, eos)
            i += 1
        running_before = len(s.running)
        waiting_before = {r.rid for r in s.waiting}
        s.step()
        admitted = waiting_before - {r.rid for r in s.waiting}
        if running_before:
            assert not admitted, "step %d admitted into a running batch" % step
        elif waiting_before:
            assert len(admitted) == min(6, len(waiting_before)), step
            batches += 1
        if i == len(arrivals) and s.idle():
            break
    assert s.idle() and len(s.finished) == 40 and batches >= 40 // 6


def test_prefix_cache_hand_worked_trace():
    """Block size 4, pool [0..19] popped from the end, no chunking.
    A: prompt 1..10, EOS after 3.  B: prompt 1..8, 50, 51, 52 (its first two
    pages equal A's), EOS after 2, arriving at step 2.  Worked by hand:
    step 0: A admitted with blocks 19, 18, 17, prefills 10 tokens; its two
            full pages are registered: (-1, 1-4) -> 19, (19, 5-8) -> 18.
    step 1: A decodes (position 10, block 17).
    step 2: B matches both pages (2 pages <= (11 - 1) // 4): blocks 19, 18 shared,
            one new block 16, computed length 8, prefill of 3 tokens at slots
            64, 65, 66; A decodes position 11 (slot 17 * 4 + 3 = 71), emits its
            third token and retires: 19 and 18 are still held by B, 17 is freed.
    step 3: B decodes and retires: 19, 18, 16 freed in table order; the cache
            empties."""
    s = Scheduler(20, 4, max_batch=4, max_num_batched_tokens=100, chunk=100, max_model_len=64, prefix_caching=True)
    s.add(0, 10, 10, 3, tokens=list(range(1, 11)))
    m0 = s.step()
    assert m0.block_tables[0, :3].tolist() == [19, 18, 17] and int(m0.q_lens[0]) == 10
    assert s.stats()["cached_blocks"] == 2
    s.step()
    s.add(1, 11, 10, 2, tokens=list(range(1, 9)) + [50, 51, 52])
    m2 = s.step()
    assert m2.seq_rids.tolist() == [1, 0]                    # B's prefill chunk first
    assert m2.q_lens.tolist() == [3, 1] and m2.context_lens.tolist() == [11, 12]
    assert m2.block_tables[0, :3].tolist() == [19, 18, 16]
    assert m2.slot_mapping.tolist() == [64, 65, 66, 71]
    assert m2.finished_rids.tolist() == [0]
    assert s.stats()["prefix_hit_blocks"] == 2
    m3 = s.step()
    assert m3.finished_rids.tolist() == [1]
    assert s.idle() and s.stats()["cached_blocks"] == 0
    assert s.pool.free_list == list(range(16)) + [17, 19, 18, 16]
    # C's prompt is exactly A's two registered pages: only one page may be
    # taken, so that the last prompt page is computed (in a block of its own)
    c = Scheduler(20, 4, max_batch=4, max_num_batched_tokens=100, chunk=100, max_model_len=64, prefix_caching=True)
    c.add(0, 10, 10, 9, tokens=list(range(1, 11)))
    c.step()
    c.add(2, 8, 10, 2, tokens=list(range(1, 9)))
    mc = c.step()
    assert mc.seq_rids.tolist() == [2, 0] and mc.q_lens.tolist() == [4, 1] and mc.context_lens.tolist() == [8, 11]
    assert mc.block_tables[0, :2].tolist() == [19, 16]
    # without the cache B recomputes everything in three fresh blocks
    n = Scheduler(20, 4, max_batch=4, max_num_batched_tokens=100, chunk=100, max_model_len=64)
    n.add(0, 10, 10, 3, tokens=list(range(1, 11)))
    n.step()
    n.step()
    n.add(1, 11, 10, 2, tokens=list(range(1, 9)) + [50, 51, 52])
    m = n.step()
    assert m.q_lens.tolist() == [11, 1] and m.block_tables[0, :3].tolist() == [16, 15, 14]


def shared_prefix_trace(rng, n, groups=4, prefix_pages=(1, 6), bs=16, tail=(0, 60), eos_mean=20):
    """Requests from a few groups: each group's prompts start with the same
    tokens (a whole number of pages), then a request's own tokens."""
    heads = [list(rng.integers(1000, 2000, size=int(rng.integers(*prefix_pages)) * bs)) for _ in range(groups)]
    out = []
    for rid in range(n):
        g = int(rng.integers(0, groups))
        toks = heads[g] + list(rng.integers(3000, 4000, size=int(rng.integers(*tail))))
        out.append((int(rng.integers(0, 50)), rid, toks, int(rng.integers(1, 60)), int(rng.geometric(1 / eos_mean))))
    return sorted(out, key=lambda x: (x[0], x[1]))


@pytest.mark.parametrize("seed", range(4))
def test_prefix_cache_invariants(seed):
    """With sharing: no emitted slot lands in a block two requests hold; each
    block's count equals its holders; free + held = pool; every request emits
    the same tokens as without sharing; the pool and cache are empty at the end."""
    rng = np.random.default_rng(seed)
    trace = shared_prefix_trace(rng, 60)
    runs = {}
    for caching in (False, True):
        s = Scheduler(120, 16, max_batch=10, max_num_batched_tokens=160, chunk=48, max_model_len=256,
                      prefix_caching=caching)
        i, prefill, computed = 0, 0, {}
        for step in range(5000):
            while i < len(trace) and trace[i][0] <= step:
                _, rid, toks, mt, eos = trace[i]
                s.add(rid, len(toks), mt, eos, tokens=toks)
                i += 1
            m = s.step()
            if m is not None:
                # holders when the step was emitted: the scheduled sequences'
                # tables, and the running requests that were not scheduled
                held = {}
                scheduled = set(int(x) for x in m.seq_rids)
                rows = [row[row >= 0] for row in m.block_tables]
                rows += [np.array(r.blocks) for r in s.running if r.rid not in scheduled]
                for row in rows:
                    for b in row:
                        held[int(b)] = held.get(int(b), 0) + 1
                prefill += int(m.q_lens[m.q_lens > 1].sum())
                for slot in m.slot_mapping:
                    assert held[int(slot) // 16] == 1, "step %d writes a shared block" % step
                for rid, q in zip(m.seq_rids, m.q_lens):
                    computed[int(rid)] = computed.get(int(rid), 0) + int(q)
            for r in s.running:
                for b in r.blocks:
                    assert s.refcount[b] == sum(b in x.blocks for x in s.running)
            held_now = set(b for r in s.running for b in r.blocks)
            assert len(held_now) + s.pool.free_count() == 120
            if i == len(trace) and s.idle():
                break
        assert s.idle() and s.pool.free_count() == 120 and not s.cache
        # every emitted token needs at least one token computed in its step
        for r in s.finished:
            assert computed[r.rid] >= r.generated, r.rid
        runs[caching] = ({r.rid: r.generated for r in s.finished}, prefill, s.prefix_hit_blocks)
    assert runs[True][0] == runs[False][0]
    assert runs[True][2] > 0 and runs[True][1] < runs[False][1]


def _swap_trace(preemption):
    s = Scheduler(6, 4, max_batch=4, max_num_batched_tokens=100, chunk=100, max_model_len=64,
                  preemption=preemption, swap_blocks=10)
    s.add(0, 7, 20, 10)
    s.add(1, 8, 20, 10)
    return s, [s.step() for _ in range(11)]


def test_swap_preemption_hand_worked_trace():
    """Block size 4, pool [0..5] popped from the end, host slots 0..9 (slot 0
    first).  A (prompt 7, EOS after 10) gets blocks 5, 4; B (prompt 8) gets 3, 2;
    B grows into 1 at step 1, A into 0 at step 2.  At step 5 B (context 12)
    needs a fourth block, none is free: B is the newest, so it preempts itself
    and is swapped out -- its three computed blocks 3, 2, 1 to slots 0, 1, 2 --
    keeping its 12 computed tokens; A takes block 1 at step 6 and retires after
    step 9.  At step 10 B comes back into blocks 1, 0, 4, 5: slots 0, 1, 2 are
    copied into 1, 0, 4 and it decodes position 12 (slot 5 * 4 + 0 = 20), where
    recompute would re-prefill all 13 tokens."""
    s, m = _swap_trace("swap")
    assert m[5].seq_rids.tolist() == [0]
    assert m[5].swap_out.tolist() == [[3, 0], [2, 1], [1, 2]] and len(m[5].swap_in) == 0
    assert m[6].block_tables[0, :4].tolist() == [5, 4, 0, 1]
    assert m[9].finished_rids.tolist() == [0]
    assert m[10].swap_in.tolist() == [[0, 1], [1, 0], [2, 4]]
    assert m[10].seq_rids.tolist() == [1] and m[10].q_lens.tolist() == [1]
    assert m[10].context_lens.tolist() == [13] and m[10].slot_mapping.tolist() == [20]
    assert m[10].block_tables[0, :4].tolist() == [1, 0, 4, 5]
    st = s.stats()
    assert st["swapped_out_blocks"] == 3 and st["swapped_in_blocks"] == 3 and st["free_swap_slots"] == 10
    _, r = _swap_trace("recompute")
    assert len(r[5].swap_out) == 0
    assert r[10].q_lens.tolist() == [13] and r[10].context_lens.tolist() == [13]


@pytest.mark.parametrize("seed", range(4))
def test_swap_preemption_invariants(seed):
    """Under memory pressure with swapping: host slots and device blocks are
    never lost (free + held = pool, free slots + slots held = capacity), no
    slot is swapped in and out in one step, a swapped request resumes with the length it had (its only prefill chunk
    after a swap-in starts where it stopped), every request emits the tokens it
    would emit with recompute, and less is recomputed."""
    rng = np.random.default_rng(seed)
    arrivals = sorted((int(rng.integers(0, 40)), rid, int(rng.integers(1, 120)), int(rng.integers(1, 80)),
                       int(rng.geometric(1 / 30))) for rid in range(50))
    runs = {}
    for mode in ("recompute", "swap"):
        s = Scheduler(40, 16, max_batch=12, max_num_batched_tokens=160, chunk=48, max_model_len=256,
                      preemption=mode, swap_blocks=24)
        i, prefill = 0, 0
        for step in range(5000):
            while i < len(arrivals) and arrivals[i][0] <= step:
                _, rid, p, mt, eos = arrivals[i]
                s.add(rid, p, mt, eos)
                i += 1
            before = {r.rid: r.num_computed for r in s.waiting if r.slots}
            m = s.step()
            if m is not None:
                prefill += int(m.q_lens[m.q_lens > 1].sum())
                for row, slot in m.swap_in:
                    assert 0 <= row < 24
                # a slot read by a swap-in is never the target of a swap-out
                # of the same step (the outs run first)
                assert not set(m.swap_in[:, 0].tolist()) & set(m.swap_out[:, 1].tolist())
                for rid, q, c in zip(m.seq_rids, m.q_lens, m.context_lens):
                    if int(rid) in before and not any(r.rid == rid and r.slots for r in s.waiting):
                        assert int(c) - int(q) == before[int(rid)], "resumed at the wrong length"
            held_slots = sum(len(r.slots) for r in s.waiting)
            assert held_slots + s.stats()["free_swap_slots"] == 24
            held = set(b for r in s.running for b in r.blocks)
            assert len(held) + s.pool.free_count() == 40
            if i == len(arrivals) and s.idle():
                break
        assert s.idle() and s.pool.free_count() == 40 and s.stats()["free_swap_slots"] == 24
        runs[mode] = ({r.rid: r.generated for r in s.finished}, prefill, s.stats())
    assert runs["swap"][0] == runs["recompute"][0]
    assert runs["swap"][2]["swapped_out_blocks"] > 0
    assert runs["swap"][1] < runs["recompute"][1]
