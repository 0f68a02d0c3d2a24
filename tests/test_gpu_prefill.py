"""GPU parity of pkv_paged_prefill_attention (K4) against the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (DeviceStep, assert_close, dev, dev_bits, oracle_decode_all, oracle_prefill_all,
                         out_to_f64)
from paged_kv_cache_tables_gb300 import kv_append, paged_decode_attention, paged_prefill_attention
from synth import build_step, make_step, rne_bits

pytestmark = pytest.mark.gpu


def chunk_step(priors, q_lens, Hq, Hkv, d, dtype, seed=0):
    priors = np.asarray(priors, np.int64)
    q_lens = np.asarray(q_lens, np.int64)
    rng = np.random.default_rng(seed)
    ctx = priors + q_lens
    nb = int(((ctx + 15) // 16).sum())
    NB = nb + 9
    st = build_step("chunks", rng, ctx=ctx, q_lens=q_lens, Hq=Hq, Hkv=Hkv, d=d, NB=NB, dtype=dtype,
                    pool_order=rng.permutation(NB), n_prefill=len(ctx))
    return st


def run_prefill(ds, out_dtype, q=None, cu=None, bt=None, cl=None, max_q_len=None):
    st = ds.st
    q = ds.q if q is None else q
    cu = ds.cu_seqlens if cu is None else cu
    bt = ds.block_tables if bt is None else bt
    cl = ds.context_lens if cl is None else cl
    odt = torch.float32 if out_dtype == "fp32" else q.dtype
    out = torch.full((q.shape[0], st.Hq, st.d), float("nan"), dtype=odt, device="cuda")
    mq = int(st.q_lens.max()) if max_q_len is None else max_q_len
    paged_prefill_attention(out, q, cu, mq, ds.k_cache, ds.v_cache, bt, cl, dev_status=ds.status)
    torch.cuda.synchronize()
    return out


def oracle_after_append(st):
    kc, vc = st.k_cache.copy(), st.v_cache.copy()
    oracle.append(st.k_new, st.v_new, st.slot_mapping, kc, vc, st.bs)
    return kc, vc


@pytest.mark.parametrize("Hq,Hkv,d,dtype", [
    (4, 4, 64, "fp16"), (32, 8, 128, "bf16"), (32, 8, 64, "bf16"), (16, 2, 128, "fp16"), (12, 4, 128, "bf16"),
    (16, 1, 64, "bf16"),
])
def test_prefill_small_chunks_full_compare(cuda_lib, Hq, Hkv, d, dtype):
    priors = [0, 0, 5, 16, 100, 37]
    q_lens = [1, 40, 17, 33, 70, 129]
    st = chunk_step(priors, q_lens, Hq, Hkv, d, dtype, seed=Hq + d)
    ds = DeviceStep(st)
    kv_append(ds.k_new, ds.v_new, ds.slot_mapping, ds.k_cache, ds.v_cache, dev_status=ds.status)
    out = run_prefill(ds, "fp32")
    kc, vc = oracle_after_append(st)
    ref = oracle.prefill(st.q, st.cu_seqlens, kc, vc, st.block_tables, st.context_lens, dtype)
    assert_close(out_to_f64(out), ref, "fp32", what="prefill %d/%d d%d %s" % (Hq, Hkv, d, dtype))
    out16 = run_prefill(ds, dtype)
    assert_close(out_to_f64(out16), ref, dtype, what="prefill 16-bit out")
    assert int(ds.status.item()) == 0


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (16, 16, 64)])
def test_prefill_long_chunks_sampled_rows(cuda_lib, Hq, Hkv, d):
    """Chunks far longer than one tile pair (many pairs, ragged last pair),
    one behind an 8,000-token context: sampled rows against the oracle, each
    row being the decode of its own position (keys 0..pos) over the cache
    after the append."""
    priors, q_lens = [6500, 0, 77], [1500, 1100, 301]
    st = chunk_step(priors, q_lens, Hq, Hkv, d, "bf16", seed=d + 1)
    ds = DeviceStep(st)
    kv_append(ds.k_new, ds.v_new, ds.slot_mapping, ds.k_cache, ds.v_cache, dev_status=ds.status)
    out = run_prefill(ds, "fp32")
    kc, vc = oracle_after_append(st)
    rng = np.random.default_rng(3)
    got, ref = [], []
    for c, (pr, ql) in enumerate(zip(priors, q_lens)):
        rows = sorted(set([0, ql - 1, ql // 2] + list(rng.integers(0, ql, size=8))))
        for i in rows:
            row = int(st.cu_seqlens[c]) + i
            ref.append(oracle.decode(st.q[row:row + 1], kc, vc, st.block_tables[c:c + 1],
                                     np.array([pr + i + 1], np.int32), "bf16")[0])
            got.append(out_to_f64(out[row:row + 1])[0])
    assert_close(np.array(got), np.array(ref), "fp32", what="long chunks %d/%d d%d" % (Hq, Hkv, d))
    assert int(ds.status.item()) == 0


def test_prefill_with_one_query_row_equals_decode(cuda_lib):
    st = make_step("llama1b", S=24)
    ds = DeviceStep(st)
    kv_append(ds.k_new, ds.v_new, ds.slot_mapping, ds.k_cache, ds.v_cache)
    cu = torch.arange(st.S + 1, dtype=torch.int32, device="cuda")
    pre = torch.empty((st.S, st.Hq, st.d), dtype=torch.float32, device="cuda")
    paged_prefill_attention(pre, ds.q, cu, 1, ds.k_cache, ds.v_cache, ds.block_tables, ds.context_lens)
    dec = torch.empty_like(pre)
    paged_decode_attention(dec, ds.q, ds.k_cache, ds.v_cache, ds.block_tables, ds.context_lens)
    torch.cuda.synchronize()
    np.testing.assert_allclose(pre.cpu().numpy(), dec.cpu().numpy(), rtol=0, atol=2e-5)


@pytest.fixture(scope="module")
def mixed_reference():
    """The mixed step after its append, with the oracle's output for every
    prefill row and every decode row (computed once for the module)."""
    st = make_step("mixed")
    kc, vc = oracle_after_append(st)
    q_p, cu_p, bt_p, cl_p = st.prefill_part()
    ref_pre = oracle_prefill_all(q_p, cu_p, kc, vc, bt_p, cl_p, st.dtype)
    q_d, bt_d, cl_d = st.decode_part()
    ref_dec = oracle_decode_all(q_d, kc, vc, bt_d, cl_d, st.dtype)
    return st, ref_pre, ref_dec


def test_mixed_step_full_size_every_row(cuda_lib, mixed_reference):
    """The mixed step: append 4344 tokens, prefill 8 chunks of 512, decode 248
    sequences -- in the launch configuration of the benchmark -- every row of
    both parts against the oracle."""
    st, ref_pre, ref_dec = mixed_reference
    ds = DeviceStep(st)
    kv_append(ds.k_new, ds.v_new, ds.slot_mapping, ds.k_cache, ds.v_cache, dev_status=ds.status)
    p = st.n_prefill
    t1 = int(st.cu_seqlens[p])
    pre = torch.empty((t1, st.Hq, st.d), dtype=torch.float32, device="cuda")
    paged_prefill_attention(pre, ds.q[:t1], ds.cu_seqlens[:p + 1], 512, ds.k_cache, ds.v_cache,
                            ds.block_tables[:p], ds.context_lens[:p], dev_status=ds.status)
    pre16 = torch.empty((t1, st.Hq, st.d), dtype=ds.q.dtype, device="cuda")
    paged_prefill_attention(pre16, ds.q[:t1], ds.cu_seqlens[:p + 1], 512, ds.k_cache, ds.v_cache,
                            ds.block_tables[:p], ds.context_lens[:p], dev_status=ds.status)
    dec = torch.empty((st.S - p, st.Hq, st.d), dtype=torch.float32, device="cuda")
    paged_decode_attention(dec, ds.q[t1:], ds.k_cache, ds.v_cache, ds.block_tables[p:], ds.context_lens[p:],
                           dev_status=ds.status)
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0
    e1 = assert_close(out_to_f64(pre), ref_pre, "fp32", what="mixed prefill, fp32 out")
    e16 = assert_close(out_to_f64(pre16), ref_pre, st.dtype, what="mixed prefill, bf16 out")
    e2 = assert_close(out_to_f64(dec), ref_dec, "fp32", what="mixed decode")
    print("mixed step, every row: max-abs prefill fp32 %.3g bf16 %.3g, decode fp32 %.3g" % (e1, e16, e2))


def test_prefill_flags_a_chunk_longer_than_its_context(cuda_lib):
    st = chunk_step([10, 20], [5, 6], 8, 8, 64, "bf16", seed=4)
    ds = DeviceStep(st)
    cl = st.context_lens.copy()
    cl[0] = 3                         # q_len 5 > ctx 3: skipped and flagged
    out = torch.zeros((st.T, st.Hq, st.d), dtype=torch.float32, device="cuda")
    paged_prefill_attention(out, ds.q, ds.cu_seqlens, 6, ds.k_cache, ds.v_cache, ds.block_tables, dev(cl),
                            dev_status=ds.status)
    torch.cuda.synchronize()
    assert int(ds.status.item()) & 16
    assert torch.all(out[:5] == 0)    # the bad chunk's rows were not written


@pytest.mark.parametrize("decode_sms", [0, 24, 130])
def test_mixed_entry_side_by_side_matches_oracle(cuda_lib, mixed_reference, decode_sms):
    """pkv_paged_mixed_attention on the mixed step (prefill and decode kernels
    on split SMs, the split picked from host metadata or forced): the prefill
    rows are the bits of the plain prefill call, and every row of both parts
    matches the oracle."""
    from paged_kv_cache_tables_gb300 import paged_mixed_attention
    st, ref_pre, ref_dec = mixed_reference
    ds = DeviceStep(st)
    kv_append(ds.k_new, ds.v_new, ds.slot_mapping, ds.k_cache, ds.v_cache, dev_status=ds.status)
    p = st.n_prefill
    t1 = int(st.cu_seqlens[p])
    out = torch.full((st.T, st.Hq, st.d), float("nan"), dtype=torch.float32, device="cuda")
    paged_mixed_attention(out, ds.q, ds.cu_seqlens[:p + 1], p, 512, ds.k_cache, ds.v_cache, ds.block_tables,
                          ds.context_lens, cu_seqlens_host=st.cu_seqlens[:p + 1], context_lens_host=st.context_lens,
                          decode_sms=decode_sms, dev_status=ds.status)
    pre = torch.empty((t1, st.Hq, st.d), dtype=torch.float32, device="cuda")
    paged_prefill_attention(pre, ds.q[:t1], ds.cu_seqlens[:p + 1], 512, ds.k_cache, ds.v_cache,
                            ds.block_tables[:p], ds.context_lens[:p], dev_status=ds.status)
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0
    assert torch.equal(out[:t1], pre)
    assert np.all(np.isfinite(out.cpu().numpy()))
    assert_close(out_to_f64(out[:t1]), ref_pre, "fp32", what="mixed entry prefill rows")
    assert_close(out_to_f64(out[t1:]), ref_dec, "fp32", what="mixed entry decode rows")
