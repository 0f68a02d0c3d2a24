"""Seeded random steps against the oracle: many small shapes, each a mixed
step (prefill chunks first, then one-token decodes) with random head counts,
head sizes, 16-bit types and context lengths (including empty and
block-boundary ones), run through the plain entry points, the side-by-side
one, the fused decode + append one and the one-call mixed step with its
append.  Append must be bit-exact and attention within the tolerance; every
call must leave the status word clear."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceStep, assert_close, out_to_f64, host_bits
from paged_kv_cache_tables_gb300 import (kv_append, paged_decode_append_attention, paged_decode_attention,
                                         paged_mixed_append_attention, paged_mixed_attention,
                                         paged_prefill_attention)
from synth import build_step

pytestmark = pytest.mark.gpu

HEADS = [(4, 4), (8, 2), (12, 4), (32, 8), (16, 1), (64, 8), (32, 2)]


def random_step(seed):
    rng = np.random.default_rng(seed)
    Hq, Hkv = HEADS[int(rng.integers(0, len(HEADS)))]
    d = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["fp16", "bf16"]))
    n_pre = int(rng.integers(0, 4))
    n_dec = int(rng.integers(0 if n_pre else 1, 24))
    q_pre = rng.integers(1, 300, size=n_pre)
    prior = rng.choice([0, 1, 15, 16, 17, 100, 700, 2500], size=n_pre)
    ctx_dec = rng.choice([1, 2, 15, 16, 17, 33, 200, 1000, 3000], size=n_dec)
    ctx = np.concatenate([prior + q_pre, ctx_dec]).astype(np.int64)
    q_lens = np.concatenate([q_pre, np.ones(n_dec, np.int64)]).astype(np.int64)
    NB = int(((ctx + 15) // 16).sum()) + 11
    st = build_step("fuzz%d" % seed, rng, ctx=ctx, q_lens=q_lens, Hq=Hq, Hkv=Hkv, d=d, NB=NB, dtype=dtype,
                    pool_order=rng.permutation(NB), n_prefill=n_pre)
    return st


def oracle_step(st):
    kc, vc = st.k_cache.copy(), st.v_cache.copy()
    oracle.append(st.k_new, st.v_new, st.slot_mapping, kc, vc, st.bs)
    p = st.n_prefill
    t1 = int(st.cu_seqlens[p])
    pre = (oracle.prefill(st.q[:t1], st.cu_seqlens[:p + 1], kc, vc, st.block_tables[:p], st.context_lens[:p],
                          st.dtype) if p else np.zeros((0, st.Hq, st.d)))
    dec = oracle.decode(st.q[t1:], kc, vc, st.block_tables[p:], st.context_lens[p:], st.dtype)
    return kc, vc, np.concatenate([pre, dec]) if p else dec


@pytest.mark.parametrize("seed", range(12))
def test_random_mixed_steps_match_oracle(cuda_lib, seed):
    st = random_step(seed)
    p = st.n_prefill
    t1 = int(st.cu_seqlens[p])
    kc, vc, ref = oracle_step(st)
    max_q = int(st.q_lens[:p].max()) if p else 0

    # 1) append, then the plain prefill and decode entry points
    ds = DeviceStep(st)
    kv_append(ds.k_new, ds.v_new, ds.slot_mapping, ds.k_cache, ds.v_cache, dev_status=ds.status)
    assert np.array_equal(host_bits(ds.k_cache), kc) and np.array_equal(host_bits(ds.v_cache), vc)
    out = torch.full((st.T, st.Hq, st.d), float("nan"), dtype=torch.float32, device="cuda")
    if p:
        paged_prefill_attention(out[:t1], ds.q[:t1], ds.cu_seqlens[:p + 1], max_q, ds.k_cache, ds.v_cache,
                                ds.block_tables[:p], ds.context_lens[:p], dev_status=ds.status)
    if st.S > p:
        paged_decode_attention(out[t1:], ds.q[t1:], ds.k_cache, ds.v_cache, ds.block_tables[p:],
                               ds.context_lens[p:], dev_status=ds.status)
    torch.cuda.synchronize()
    assert_close(out_to_f64(out), ref, "fp32", what="fuzz %d plain" % seed)

    # 2) the side-by-side entry point on the same caches
    if p and st.S > p:
        out2 = torch.full_like(out, float("nan"))
        paged_mixed_attention(out2, ds.q, ds.cu_seqlens[:p + 1], p, max_q, ds.k_cache, ds.v_cache,
                              ds.block_tables, ds.context_lens, dev_status=ds.status,
                              cu_seqlens_host=st.cu_seqlens[:p + 1].astype(np.int32),
                              context_lens_host=st.context_lens.astype(np.int32))
        torch.cuda.synchronize()
        assert_close(out_to_f64(out2), ref, "fp32", what="fuzz %d mixed" % seed)
    assert int(ds.status.item()) == 0

    # 3) decodes with the append fused, on fresh caches (prefill rows appended first)
    if st.S > p:
        ds3 = DeviceStep(st)
        if p:
            kv_append(ds3.k_new[:t1], ds3.v_new[:t1], ds3.slot_mapping[:t1], ds3.k_cache, ds3.v_cache,
                      dev_status=ds3.status)
        out3 = torch.full((st.S - p, st.Hq, st.d), float("nan"), dtype=torch.bfloat16 if st.dtype == "bf16"
                          else torch.float16, device="cuda")
        paged_decode_append_attention(out3, ds3.q[t1:], ds3.k_new[t1:], ds3.v_new[t1:], ds3.k_cache, ds3.v_cache,
                                      ds3.block_tables[p:], ds3.context_lens[p:], dev_status=ds3.status)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(ds3.k_cache), kc) and np.array_equal(host_bits(ds3.v_cache), vc)
        assert_close(out_to_f64(out3), ref[t1:], st.dtype, what="fuzz %d fused" % seed)
        assert int(ds3.status.item()) == 0

    # 4) the whole step (append included) in one call, on fresh caches
    ds4 = DeviceStep(st)
    out4 = torch.full((st.T, st.Hq, st.d), float("nan"), dtype=torch.float32, device="cuda")
    paged_mixed_append_attention(out4, ds4.q, ds4.k_new, ds4.v_new, ds4.slot_mapping[:t1],
                                 ds4.cu_seqlens[:p + 1], p, max_q, ds4.k_cache, ds4.v_cache, ds4.block_tables, ds4.context_lens,
                                 dev_status=ds4.status, cu_seqlens_host=st.cu_seqlens[:p + 1].astype(np.int32),
                                 context_lens_host=st.context_lens.astype(np.int32))
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(ds4.k_cache), kc) and np.array_equal(host_bits(ds4.v_cache), vc)
    assert_close(out_to_f64(out4), ref, "fp32", what="fuzz %d one call" % seed)
    assert int(ds4.status.item()) == 0
