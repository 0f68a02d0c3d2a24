"""GPU parity of pkv_paged_decode_attention (K2 + K3) against the FP64 oracle.

Every workload is compared element by element in full, including the
Llama-3-8B-shaped step (256 sequences, lognormal contexts) at full size in the
launch configuration the benchmark uses.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (SPLIT_ATOL, SPLIT_RTOL, DeviceStep, assert_close, dev, dev_bits, host_bits,
                         oracle_decode_all, out_to_f64, split_excess)
from paged_kv_cache_tables_gb300 import decode_workspace_size, kv_append, paged_decode_attention
from synth import NAN_BITS, build_step, make_step, rne_bits

pytestmark = pytest.mark.gpu


def run_decode(ds, q, block_tables, context_lens, out_dtype, scale=None):
    st = ds.st
    S = q.shape[0]
    odt = torch.float32 if out_dtype == "fp32" else q.dtype
    out = torch.full((S, st.Hq, st.d), float("nan"), dtype=odt, device="cuda")
    paged_decode_attention(out, q, ds.k_cache, ds.v_cache, block_tables, context_lens, scale=scale,
                           dev_status=ds.status)
    torch.cuda.synchronize()
    return out


def append_then_decode(st, out_dtype, append=True):
    ds = DeviceStep(st)
    if append:
        kv_append(ds.k_new, ds.v_new, ds.slot_mapping, ds.k_cache, ds.v_cache, dev_status=ds.status)
    q_d, bt_d, cl_d = st.decode_part()
    p = st.n_prefill
    t0 = int(st.cu_seqlens[p])
    out = run_decode(ds, ds.q[t0:], ds.block_tables[p:], ds.context_lens[p:], out_dtype)
    kc, vc = st.k_cache, st.v_cache
    if append:
        kc, vc = kc.copy(), vc.copy()
        oracle.append(st.k_new, st.v_new, st.slot_mapping, kc, vc, st.bs)
    return ds, out, (q_d, kc, vc, bt_d, cl_d)


@pytest.mark.parametrize("out_dtype", ["fp32", "same"])
@pytest.mark.parametrize("name,kw", [("tiny", {}), ("llama1b", {"S": 64})])
def test_decode_small_workloads_full_compare(cuda_lib, name, kw, out_dtype):
    st = make_step(name, **kw)
    od = "fp32" if out_dtype == "fp32" else st.dtype
    ds, out, (q, kc, vc, bt, cl) = append_then_decode(st, od)
    ref = oracle.decode(q, kc, vc, bt, cl, st.dtype)
    err = assert_close(out_to_f64(out), ref, od, what=name)
    assert int(ds.status.item()) == 0
    print("%s %s max-abs %.3g" % (name, od, err))


def test_decode_llama8b_full_size_every_sequence(cuda_lib):
    """The Llama-3-8B-shaped step at full size, in the launch configuration
    the benchmark times (work stealing on), fp32 and bf16 outputs, compared
    with the oracle on all 256 sequences."""
    st = make_step("llama8b")
    ds, out32, (q, kc, vc, bt, cl) = append_then_decode(st, "fp32")
    out16 = run_decode(ds, ds.q, ds.block_tables, ds.context_lens, "bf16")
    ref = oracle_decode_all(q, kc, vc, bt, cl, st.dtype)
    e32 = assert_close(out_to_f64(out32), ref, "fp32", what="llama8b fp32")
    e16 = assert_close(out_to_f64(out16), ref, "bf16", what="llama8b bf16")
    assert int(ds.status.item()) == 0
    print("llama8b all 256 sequences max-abs fp32 %.3g bf16 %.3g" % (e32, e16))


def test_decode_part_of_mixed_step_with_nan_tails(cuda_lib):
    st = make_step("mixed", n_chunks=2, chunk=64, n_decode=40, NB=8192)
    ds, out, (q, kc, vc, bt, cl) = append_then_decode(st, "fp32")
    ref = oracle.decode(q, kc, vc, bt, cl, st.dtype)
    assert_close(out_to_f64(out), ref, "fp32", what="mixed decode")


def custom_step(ctx, Hq, Hkv, d, dtype, seed=0, NB=None):
    ctx = np.asarray(ctx, np.int64)
    rng = np.random.default_rng(seed)
    nb = int(((ctx + 15) // 16).sum())
    NB = NB or nb + 7
    # q_lens = 0: every position below the context is already stored; one
    # query row per sequence is drawn separately
    st = build_step("custom", rng, ctx=ctx, q_lens=np.zeros_like(ctx), Hq=Hq, Hkv=Hkv, d=d, NB=NB, dtype=dtype,
                    pool_order=rng.permutation(NB))
    st.q = rne_bits(rng.standard_normal((len(ctx), Hq, d), dtype=np.float32), dtype)
    return st


@pytest.mark.parametrize("Hq,Hkv,d,dtype", [
    (4, 4, 64, "fp16"), (32, 8, 64, "bf16"), (32, 8, 128, "bf16"), (32, 8, 128, "fp16"),
    (64, 8, 128, "bf16"), (32, 2, 128, "bf16"), (16, 1, 64, "fp16"), (12, 4, 128, "bf16"),
])
def test_decode_edge_contexts_and_group_sizes(cuda_lib, Hq, Hkv, d, dtype):
    ctx = [1, 15, 16, 17, 32, 33, 0, 250, 1000]
    st = custom_step(ctx, Hq, Hkv, d, dtype, seed=Hq * d)
    ds = DeviceStep(st)
    out = run_decode(ds, ds.q, ds.block_tables, ds.context_lens, "fp32")
    ref = oracle.decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, dtype)
    assert_close(out_to_f64(out), ref, "fp32", what="edges %d/%d d%d %s" % (Hq, Hkv, d, dtype))
    # context 0 gives exact zeros
    assert torch.all(out[6] == 0)
    assert int(ds.status.item()) == 0


def test_decode_one_long_sequence_split_across_many_warps(cuda_lib):
    st = custom_step([8192], 32, 8, 128, "bf16", seed=5)
    ds = DeviceStep(st)
    out = run_decode(ds, ds.q, ds.block_tables, ds.context_lens, "fp32")
    ref = oracle.decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, "bf16")
    assert_close(out_to_f64(out), ref, "fp32", what="8192 split")


def test_decode_many_sequences_plan_spans_several_scan_tiles(cuda_lib):
    rng = np.random.default_rng(2)
    ctx = rng.integers(0, 70, size=1100)
    st = custom_step(ctx, 8, 2, 64, "bf16", seed=3)
    ds = DeviceStep(st)
    out = run_decode(ds, ds.q, ds.block_tables, ds.context_lens, "fp32")
    ref = oracle.decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, "bf16")
    assert_close(out_to_f64(out), ref, "fp32", what="S=1100")


def test_decode_explicit_scale(cuda_lib):
    st = custom_step([40, 300], 8, 8, 64, "fp16", seed=9)
    ds = DeviceStep(st)
    out = run_decode(ds, ds.q, ds.block_tables, ds.context_lens, "fp32", scale=0.05)
    ref = oracle.decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, "fp16", scale=0.05)
    assert_close(out_to_f64(out), ref, "fp32", what="scale")


@pytest.fixture
def deterministic(monkeypatch):
    monkeypatch.setenv("PKV_DETERMINISTIC", "1")


def test_decode_block_permutation_gives_identical_bits(cuda_lib, deterministic):
    """With work stealing off, only the physical placement changes: the split
    of every range, and so every bit of the output, stays the same."""
    st = make_step("llama1b", S=16)
    ds = DeviceStep(st)
    out_a = run_decode(ds, ds.q, ds.block_tables, ds.context_lens - 1, "fp32")
    perm = np.random.default_rng(4).permutation(st.NB)
    kc = np.empty_like(st.k_cache)
    vc = np.empty_like(st.v_cache)
    kc[perm] = st.k_cache
    vc[perm] = st.v_cache
    tables = np.where(st.block_tables >= 0, perm[np.maximum(st.block_tables, 0)], -1).astype(np.int32)
    ds.k_cache = dev_bits(kc, st.dtype)
    ds.v_cache = dev_bits(vc, st.dtype)
    out_b = run_decode(ds, ds.q, dev(tables), ds.context_lens - 1, "fp32")
    assert torch.equal(out_a, out_b)


def test_decode_work_stealing_changes_only_rounding(cuda_lib, monkeypatch):
    """The 8B-shaped step with and without stealing, 50 stealing calls in a
    row: each the same attention as the fixed split up to the rounding of
    how the ranges were split (SPLIT_ATOL + SPLIT_RTOL |o|), on every
    sequence, with a clean status word (no self-check of the split
    bookkeeping failed)."""
    st = make_step("llama8b")
    ds = DeviceStep(st)
    cl = ds.context_lens - 1
    monkeypatch.setenv("PKV_DETERMINISTIC", "1")
    fixed = run_decode(ds, ds.q, ds.block_tables, cl, "fp32")
    again = run_decode(ds, ds.q, ds.block_tables, cl, "fp32")
    assert torch.equal(fixed, again)
    monkeypatch.delenv("PKV_DETERMINISTIC")
    worst = 0.0
    for k in range(50):
        stolen = run_decode(ds, ds.q, ds.block_tables, cl, "fp32")
        assert int(ds.status.item()) == 0, "call %d: status %d" % (k, int(ds.status.item()))
        diff = (stolen - fixed).abs()
        bad = ~(diff <= SPLIT_ATOL + SPLIT_RTOL * fixed.abs())       # NaN counts as bad
        if bool(bad.any()):
            s_, h_, _ = [int(x) for x in torch.nonzero(bad)[0]]
            raise AssertionError("call %d: %d elements differ, first at sequence %d head %d (max %g)"
                                 % (k, int(bad.sum()), s_, h_, float(diff.nan_to_num(1e9).max())))
        worst = max(worst, float(diff.max()))
    print("50 stealing calls: max |stolen - fixed| %.3g" % worst)


@pytest.mark.parametrize("fill", ["ones", "small_ints", "random", "other_layout"])
def test_decode_ignores_workspace_contents(cuda_lib, monkeypatch, fill):
    """Whatever the workspace holds on entry -- all-ones bytes, every 32-bit
    word a small integer (what old counters, block ids and record links look
    like), random bytes, or what a call with a different shape left there --
    the result is the same as on a fresh workspace."""
    st = make_step("llama8b")
    ds = DeviceStep(st)
    cl = ds.context_lens - 1
    size = decode_workspace_size(st.S, st.Hq, st.Hkv, st.d)
    monkeypatch.setenv("PKV_DETERMINISTIC", "1")
    clean = torch.zeros(size, dtype=torch.uint8, device="cuda")
    ref = torch.empty((st.S, st.Hq, st.d), dtype=torch.float32, device="cuda")
    paged_decode_attention(ref, ds.q, ds.k_cache, ds.v_cache, ds.block_tables, cl, workspace=clean)
    monkeypatch.delenv("PKV_DETERMINISTIC")
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    for k in range(8):
        if fill == "ones":
            ws.fill_(0xFF)
        elif fill == "small_ints":
            ws.view(torch.int32)[:] = torch.arange(ws.numel() // 4, device="cuda", dtype=torch.int32) % (k + 40)
        elif fill == "random":
            ws.copy_(torch.randint(0, 256, (size,), dtype=torch.uint8, device="cuda", generator=g))
        else:
            # a smaller step on the same workspace, then this one
            small = make_step("llama1b", S=48 + k) if k == 0 else None
            if small is not None:
                dsm = DeviceStep(small)
            o = torch.empty((dsm.st.S, dsm.st.Hq, dsm.st.d), dtype=torch.float32, device="cuda")
            paged_decode_attention(o, dsm.q, dsm.k_cache, dsm.v_cache, dsm.block_tables, dsm.context_lens,
                                   workspace=ws, dev_status=ds.status)
        out = torch.full_like(ref, float("nan"))
        paged_decode_attention(out, ds.q, ds.k_cache, ds.v_cache, ds.block_tables, cl, workspace=ws,
                               dev_status=ds.status)
        torch.cuda.synchronize()
        assert int(ds.status.item()) == 0
        assert split_excess(out, ref) <= 0, "fill %s, call %d: differs by %g" % (
            fill, k, float((out - ref).abs().nan_to_num(1e9).max()))


def test_decode_sequence_alone_equals_sequence_in_batch(cuda_lib):
    st = make_step("llama1b", S=64)
    ds = DeviceStep(st)
    full = run_decode(ds, ds.q, ds.block_tables, ds.context_lens - 1, "fp32")
    for s in [0, 17, 63]:
        alone = run_decode(ds, ds.q[s:s + 1], ds.block_tables[s:s + 1], ds.context_lens[s:s + 1] - 1, "fp32")
        # a sequence alone and in a batch is split differently: fp32 rounding
        # plus the rounding of P against each split's running maxima
        np.testing.assert_allclose(out_to_f64(alone[0]), out_to_f64(full[s]), rtol=SPLIT_RTOL, atol=1e-5)


def test_decode_flags_bad_block_ids_and_contexts_without_faulting(cuda_lib):
    st = custom_step([40, 40], 8, 8, 64, "bf16", seed=1)
    ds = DeviceStep(st)
    bt = st.block_tables.copy()
    bt[0, 1] = st.NB + 1000          # past the pool: reads zeros, flags
    cl = st.context_lens.copy()
    cl[1] = 10_000                   # beyond the table: clamped, flags
    run_decode(ds, ds.q, dev(bt), dev(cl), "fp32")
    flags = int(ds.status.item())
    assert flags & 1 and flags & 2


def test_decode_one_hot_closed_form_is_exact(cuda_lib):
    """q = 256 e_r, a single K row with 256 in dim r: the output is exactly the
    selected V row (fp32 output), whatever the split."""
    rng = np.random.default_rng(8)
    Hq, Hkv, d, dtype = 32, 8, 128, "bf16"
    G = Hq // Hkv
    ctx = np.array([3000, 17, 700], np.int64)
    st = custom_step(ctx, Hq, Hkv, d, dtype, seed=8)
    one = rne_bits(np.float32([256.0]), dtype)[0]
    kc = st.k_cache.copy()
    for s in range(len(ctx)):
        for t in range(int(ctx[s])):
            kc[st.block_tables[s, t // 16], :, t % 16, :] = 0
    q = np.zeros_like(st.q)
    expect = np.zeros((len(ctx), Hq, d))
    for s in range(len(ctx)):
        for h in range(Hq):
            g, r = h // G, h % G
            q[s, h, r] = one
            t = int(rng.integers(0, ctx[s]))
            while np.any(kc[st.block_tables[s, t // 16], g, t % 16, :G] != 0):
                t = int(rng.integers(0, ctx[s]))
            kc[st.block_tables[s, t // 16], g, t % 16, r] = one
            expect[s, h] = oracle.to_double(st.v_cache[st.block_tables[s, t // 16], g, t % 16], dtype)
    ds = DeviceStep(st)
    ds.k_cache = dev_bits(kc, dtype)
    ds.q = dev_bits(q, dtype)
    out = run_decode(ds, ds.q, ds.block_tables, ds.context_lens, "fp32")
    assert np.array_equal(out_to_f64(out), expect)


def test_workspace_size_is_independent_of_contexts(cuda_lib):
    a = decode_workspace_size(256, 32, 8, 128)
    assert a > 0 and a == decode_workspace_size(256, 32, 8, 128)
    # partial records hold exactly the G heads of a group
    assert decode_workspace_size(256, 8, 8, 128) < a < decode_workspace_size(256, 64, 8, 128) < \
        decode_workspace_size(256, 128, 8, 128)
    # head_dim 64: records of the 2G heads of a KV-head pair while G <= 4
    assert 0 < decode_workspace_size(256, 8, 8, 64) < decode_workspace_size(256, 32, 8, 64) < \
        decode_workspace_size(256, 128, 8, 64)


def test_decode_with_the_smallest_accepted_workspace(cuda_lib):
    """The call accepts a workspace down to two partial records per warp and
    four slots per range; a warp then steals only when its own share left no
    piece.  The smallest accepted size is found by bisection (a smaller
    workspace is rejected before anything is enqueued); it is eight records
    per warp (and, in a step of few ranges, 28 slots per range) short of the
    recommended size.  The 8B-shaped step run on it still matches the oracle
    on every sequence."""
    from paged_kv_cache_tables_gb300 import PkvError
    st = make_step("llama8b")
    ds = DeviceStep(st)
    cl = ds.context_lens - 1
    out = torch.empty((st.S, st.Hq, st.d), dtype=torch.float32, device="cuda")
    big = decode_workspace_size(st.S, st.Hq, st.Hkv, st.d)
    pool = torch.empty(big, dtype=torch.uint8, device="cuda")

    def accepted(n):
        try:
            paged_decode_attention(out, ds.q, ds.k_cache, ds.v_cache, ds.block_tables, cl, workspace=pool[:n],
                                   dev_status=ds.status)
            return True
        except PkvError as e:
            assert e.status == -3      # PKV_ERR_WORKSPACE, nothing enqueued
            return False

    lo, hi = 16, big                   # accepted(hi), not accepted(lo)
    assert accepted(hi) and not accepted(lo)
    while hi - lo > 16:
        mid = (lo + hi) // 2 // 16 * 16
        if accepted(mid):
            hi = mid
        else:
            lo = mid
    assert not accepted(hi - 1)
    G = st.Hq // st.Hkv
    rec_bytes = 4 * (((2 * G + G * st.d + 3) & ~3) + 4)
    n_warps = 8 * torch.cuda.get_device_properties(0).multi_processor_count
    a256 = lambda x: (x + 255) // 256 * 256
    # the recommended size adds eight records per warp, and 28 more slots per
    # range in a step of at most 1024 ranges
    slots = 32 if st.S * st.Hkv <= 1024 else 4
    assert big - hi == 8 * n_warps * rec_bytes + a256(st.S * st.Hkv * slots * 8) - a256(st.S * st.Hkv * 4 * 8)
    out.fill_(float("nan"))
    paged_decode_attention(out, ds.q, ds.k_cache, ds.v_cache, ds.block_tables, cl, workspace=pool[:hi],
                           dev_status=ds.status)
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0
    ref = oracle_decode_all(st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens - 1, st.dtype)
    err = assert_close(out_to_f64(out), ref, "fp32", what="smallest workspace (%d bytes)" % hi)
    print("smallest accepted workspace %d bytes (recommended %d), max-abs %.3g" % (hi, big, err))


def test_decode_back_to_back_calls_of_different_shapes_share_a_workspace(cuda_lib):
    """Decode calls of two different steps (the 1B shape with 64 sequences,
    the 8B shape with 96) alternate on one workspace and one stream, twelve
    times each, with no synchronisation between them.  Each call may start
    and plan while the previous one (another shape, same workspace) still
    runs.  Every call's context lengths are computed by the kernel just
    before it.  Every output matches its oracle on every sequence, and the
    status word stays clean."""
    sa = make_step("llama1b", S=64)
    sb = make_step("llama8b", seed=7, S=96, NB=16384)
    da, db = DeviceStep(sa), DeviceStep(sb)
    size = max(decode_workspace_size(s.S, s.Hq, s.Hkv, s.d) for s in (sa, sb))
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for k in range(12):
        for st, ds in ((sa, da), (sb, db)):
            out = torch.full((st.S, st.Hq, st.d), float("nan"), dtype=torch.float32, device="cuda")
            cl = ds.context_lens - 1          # written by the kernel right before the call
            paged_decode_attention(out, ds.q, ds.k_cache, ds.v_cache, ds.block_tables, cl, workspace=ws,
                                   dev_status=status)
            outs.append((st, out))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    refs = {id(st): oracle_decode_all(st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens - 1, st.dtype)
            for st in (sa, sb)}
    worst = 0.0
    for k, (st, out) in enumerate(outs):
        worst = max(worst, assert_close(out_to_f64(out), refs[id(st)], "fp32", what="call %d (%s)" % (k, st.name)))
    print("24 alternating calls on one workspace: max-abs %.3g" % worst)


@pytest.mark.parametrize("Hq,Hkv,dtype,S,ctx_hi", [
    (8, 8, "fp16", 256, 2048),     # G = 1: units of 2 query heads
    (16, 8, "bf16", 256, 2048),    # G = 2
    (32, 8, "bf16", 128, 8192),    # G = 4, wide tables: paired from 512 ranges on
    (32, 4, "fp16", 160, 2048),    # two KV-head pairs
])
def test_decode_head_dim_64_in_kv_head_pairs(cuda_lib, Hq, Hkv, dtype, S, ctx_hi):
    """Steps large enough for head_dim 64 to run two adjacent KV heads as
    one unit, against the oracle on every sequence (fp32 and 16-bit
    outputs); then the same step with a workspace too small for the paired
    layout but large enough for single heads, which must fall back and give
    the same attention."""
    rng = np.random.default_rng(Hq * 7 + Hkv)
    ctx = rng.integers(1, ctx_hi, size=S, endpoint=True)
    st = custom_step(ctx, Hq, Hkv, 64, dtype, seed=Hq + S)
    ds = DeviceStep(st)
    ref = oracle_decode_all(st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, st.dtype)
    out32 = run_decode(ds, ds.q, ds.block_tables, ds.context_lens, "fp32")
    out16 = run_decode(ds, ds.q, ds.block_tables, ds.context_lens, dtype)
    assert int(ds.status.item()) == 0
    e32 = assert_close(out_to_f64(out32), ref, "fp32", what="paired fp32")
    e16 = assert_close(out_to_f64(out16), ref, dtype, what="paired %s" % dtype)
    # the smallest accepted workspace: the single-head layout (smaller here)
    big = decode_workspace_size(st.S, st.Hq, st.Hkv, st.d)
    pool = torch.empty(big, dtype=torch.uint8, device="cuda")
    from paged_kv_cache_tables_gb300 import PkvError
    lo, hi = 16, big
    while hi - lo > 16:
        mid = (lo + hi) // 2 // 16 * 16
        try:
            paged_decode_attention(out32, ds.q, ds.k_cache, ds.v_cache, ds.block_tables, ds.context_lens,
                                   workspace=pool[:mid], dev_status=ds.status)
            hi = mid
        except PkvError as e:
            assert e.status == -3
            lo = mid
    out32.fill_(float("nan"))
    paged_decode_attention(out32, ds.q, ds.k_cache, ds.v_cache, ds.block_tables, ds.context_lens,
                           workspace=pool[:hi], dev_status=ds.status)
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0
    e_small = assert_close(out_to_f64(out32), ref, "fp32", what="fallback fp32")
    print("Hq %d Hkv %d %s S %d: fp32 %.3g, 16-bit %.3g; smallest workspace %d of %d: %.3g"
          % (Hq, Hkv, dtype, S, e32, e16, hi, big, e_small))
