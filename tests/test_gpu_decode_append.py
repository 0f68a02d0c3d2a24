"""GPU parity of pkv_paged_decode_append_attention: the decode step's append
fused into the attention launch.  Against the oracle: the caches after the
call equal oracle.append's bit for bit, the outputs equal the oracle's
attention over them within tolerance; with work stealing off, the fused
output is bit-identical to kv_append followed by decode."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (DeviceStep, assert_close, dev, dev_bits, host_bits, oracle_decode_all, out_to_f64,
                         split_excess)
from paged_kv_cache_tables_gb300 import kv_append, paged_decode_append_attention, paged_decode_attention
from synth import build_step, make_step, rne_bits

pytestmark = pytest.mark.gpu


def table_slots(block_tables, context_lens):
    """Slot of position ctx-1 of each sequence through its table (-1: none)."""
    out = np.full(len(context_lens), -1, np.int64)
    for s, c in enumerate(context_lens):
        if c > 0:
            out[s] = int(block_tables[s, (c - 1) // 16]) * 16 + (c - 1) % 16
    return out


def fused(ds, q, k_new, v_new, block_tables, context_lens, out_dtype):
    S = q.shape[0]
    odt = torch.float32 if out_dtype == "fp32" else q.dtype
    out = torch.full((S, ds.st.Hq, ds.st.d), float("nan"), dtype=odt, device="cuda")
    paged_decode_append_attention(out, q, k_new, v_new, ds.k_cache, ds.v_cache, block_tables, context_lens,
                                  dev_status=ds.status)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("out_dtype", ["fp32", "same"])
@pytest.mark.parametrize("name,kw", [("tiny", {}), ("llama1b", {"S": 64}), ("llama8b", {})])
def test_fused_append_matches_oracle(cuda_lib, name, kw, out_dtype):
    st = make_step(name, **kw)
    assert np.array_equal(st.slot_mapping, table_slots(st.block_tables, st.context_lens))
    od = "fp32" if out_dtype == "fp32" else st.dtype
    ds = DeviceStep(st)
    out = fused(ds, ds.q, ds.k_new, ds.v_new, ds.block_tables, ds.context_lens, od)
    kc, vc = st.k_cache.copy(), st.v_cache.copy()
    oracle.append(st.k_new, st.v_new, st.slot_mapping, kc, vc, st.bs)
    assert np.array_equal(host_bits(ds.k_cache), kc)
    assert np.array_equal(host_bits(ds.v_cache), vc)
    ref = oracle_decode_all(st.q, kc, vc, st.block_tables, st.context_lens, st.dtype)
    err = assert_close(out_to_f64(out), ref, od, what="fused %s" % name)
    assert int(ds.status.item()) == 0
    print("fused %s %s: all %d sequences, max-abs %.3g" % (name, od, st.S, err))


def test_fused_work_stealing_changes_only_rounding(cuda_lib, monkeypatch):
    """The fused append + decode on the 8B-shaped step, 50 stealing calls in
    a row (each rewrites the same new rows): every output within rounding of
    the fixed-split result, the caches unchanged after the first call, the
    status word clean."""
    st = make_step("llama8b")
    ds = DeviceStep(st)
    monkeypatch.setenv("PKV_DETERMINISTIC", "1")
    fixed = fused(ds, ds.q, ds.k_new, ds.v_new, ds.block_tables, ds.context_lens, "fp32")
    k_after = ds.k_cache.view(torch.int16).clone()
    v_after = ds.v_cache.view(torch.int16).clone()
    monkeypatch.delenv("PKV_DETERMINISTIC")
    for k in range(50):
        out = fused(ds, ds.q, ds.k_new, ds.v_new, ds.block_tables, ds.context_lens, "fp32")
        assert int(ds.status.item()) == 0, "call %d: status %d" % (k, int(ds.status.item()))
        assert split_excess(out, fixed) <= 0, "call %d differs from the fixed split by %g" % (
            k, float((out - fixed).abs().nan_to_num(1e9).max()))
    assert torch.equal(ds.k_cache.view(torch.int16), k_after)
    assert torch.equal(ds.v_cache.view(torch.int16), v_after)


def test_fused_equals_append_then_decode_bit_for_bit(cuda_lib, monkeypatch):
    monkeypatch.setenv("PKV_DETERMINISTIC", "1")
    st = make_step("llama8b")
    a = DeviceStep(st)
    kv_append(a.k_new, a.v_new, a.slot_mapping, a.k_cache, a.v_cache, dev_status=a.status)
    out_a = torch.empty((st.S, st.Hq, st.d), dtype=torch.float32, device="cuda")
    paged_decode_attention(out_a, a.q, a.k_cache, a.v_cache, a.block_tables, a.context_lens, dev_status=a.status)
    b = DeviceStep(st)
    out_b = fused(b, b.q, b.k_new, b.v_new, b.block_tables, b.context_lens, "fp32")
    assert torch.equal(out_a, out_b)
    # compare bit patterns: the pool's untouched rows hold NaN
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))


def new_rows_step(ctx, Hq, Hkv, d, dtype, seed):
    ctx = np.asarray(ctx, np.int64)
    rng = np.random.default_rng(seed)
    NB = int(((ctx + 15) // 16).sum()) + 7
    st = build_step("custom", rng, ctx=ctx, q_lens=np.zeros_like(ctx), Hq=Hq, Hkv=Hkv, d=d, NB=NB, dtype=dtype,
                    pool_order=rng.permutation(NB))
    S = len(ctx)
    st.q = rne_bits(rng.standard_normal((S, Hq, d), dtype=np.float32), dtype)
    k_new = rne_bits(rng.standard_normal((S, Hkv, d), dtype=np.float32), dtype)
    v_new = rne_bits(rng.standard_normal((S, Hkv, d), dtype=np.float32), dtype)
    return st, k_new, v_new


@pytest.mark.parametrize("Hq,Hkv,d,dtype", [
    (4, 4, 64, "fp16"), (32, 8, 128, "bf16"), (64, 4, 128, "bf16"), (16, 1, 64, "fp16"), (12, 4, 128, "fp16"),
])
def test_fused_append_edge_contexts(cuda_lib, Hq, Hkv, d, dtype):
    """New tokens that open a block (ctx 1, 17, 33), fill one (16, 32) or sit
    inside one; a sequence with context 0 appends nothing."""
    ctx = [1, 15, 16, 17, 32, 33, 0, 250, 1000]
    st, k_new, v_new = new_rows_step(ctx, Hq, Hkv, d, dtype, seed=Hq + d)
    ds = DeviceStep(st)
    out = fused(ds, ds.q, dev_bits(k_new, dtype), dev_bits(v_new, dtype), ds.block_tables, ds.context_lens, "fp32")
    slots = table_slots(st.block_tables, st.context_lens)
    keep = slots >= 0
    kc, vc = st.k_cache.copy(), st.v_cache.copy()
    oracle.append(k_new[keep], v_new[keep], slots[keep], kc, vc, 16)
    assert np.array_equal(host_bits(ds.k_cache), kc)
    assert np.array_equal(host_bits(ds.v_cache), vc)
    ref = oracle.decode(st.q, kc, vc, st.block_tables, st.context_lens, dtype)
    assert_close(out_to_f64(out), ref, "fp32", what="fused edges %d/%d d%d" % (Hq, Hkv, d))
    assert torch.all(out[6] == 0)
    assert int(ds.status.item()) == 0


def test_fused_append_skips_and_flags_a_bad_last_block(cuda_lib):
    st, k_new, v_new = new_rows_step([40, 40], 8, 8, 64, "bf16", seed=3)
    bt = st.block_tables.copy()
    bt[0, 2] = st.NB + 5          # the block of sequence 0's new token: past the pool
    ds = DeviceStep(st)
    fused(ds, ds.q, dev_bits(k_new, "bf16"), dev_bits(v_new, "bf16"), dev(bt), ds.context_lens, "fp32")
    assert int(ds.status.item()) & 1
    kc, vc = st.k_cache.copy(), st.v_cache.copy()
    oracle.append(k_new[1:], v_new[1:], table_slots(bt, st.context_lens)[1:], kc, vc, 16)
    assert np.array_equal(host_bits(ds.k_cache), kc)
    assert np.array_equal(host_bits(ds.v_cache), vc)
