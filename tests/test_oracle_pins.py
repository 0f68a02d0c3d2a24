"""Pins of the FP64 oracle to facts outside itself (CPU only).

Each test ties an oracle function to something it cannot agree with by
construction: a library routine (numpy's/torch's 16-bit decoders, torch's
scaled-dot-product attention in float64 with its own lower-right causal mask),
a closed form (one-hot selection, uniform weights, the two-token logistic
weight), brute force on tiny inputs, or an invariance that a wrong index would
break (block permutation, identity tables, split-and-merge).  The cases are
chosen so a dropped term, a wrong head mapping, an off-by-one in the context
length or block offset, or a wrong scale fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import oracle
from synth import NAN_BITS, make_step, rne_bits

BS = 16


def rand_bits(rng, shape, dtype):
    return rne_bits(rng.standard_normal(shape, dtype=np.float32), dtype)


def place(k_seq, v_seq, table, NB, nan):
    """Scatter contiguous per-token rows [ctx, Hkv, d] into a [NB, Hkv, BS, d]
    pool through a block-table row (layout of the cache interface)."""
    ctx, Hkv, d = k_seq.shape
    kc = np.full((NB, Hkv, BS, d), nan, np.uint16)
    vc = np.full((NB, Hkv, BS, d), nan, np.uint16)
    for t in range(ctx):
        kc[table[t // BS], :, t % BS, :] = k_seq[t]
        vc[table[t // BS], :, t % BS, :] = v_seq[t]
    return kc, vc


def sdpa64(q, k, v, scale, mask=None):
    """torch SDPA in float64; q [Hq, Lq, d], k/v [Hkv, Lk, d]; KV heads are
    shared by contiguous groups of query heads."""
    G = q.shape[0] // k.shape[0]
    k = k.repeat_interleave(G, dim=0)
    v = v.repeat_interleave(G, dim=0)
    return F.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=mask, scale=scale)[0]


# ---------------------------------------------------------------- 16-bit decode

def test_fp16_decode_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.to_double(bits, "fp16")
    ref = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(mine[fin], ref[fin])
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(np.isinf(mine), np.isinf(ref))


def test_bf16_decode_matches_torch_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.to_double(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(mine[fin], ref[fin])
    assert np.array_equal(np.isnan(mine), np.isnan(ref))


# ------------------------------------------------- dense attention vs a library

@pytest.mark.parametrize("dtype,Hq,Hkv,d,ctx", [
    ("fp16", 4, 4, 64, 18), ("bf16", 32, 8, 64, 40), ("bf16", 8, 1, 128, 33), ("fp16", 16, 2, 128, 1),
])
def test_dense_matches_torch_sdpa(dtype, Hq, Hkv, d, ctx):
    rng = np.random.default_rng(7)
    q = rand_bits(rng, (Hq, d), dtype)
    k = rand_bits(rng, (ctx, Hkv, d), dtype)
    v = rand_bits(rng, (ctx, Hkv, d), dtype)
    mine = oracle.dense(q, k, v, dtype)
    tq = torch.from_numpy(oracle.to_double(q, dtype))[:, None, :]
    tk = torch.from_numpy(oracle.to_double(k, dtype)).permute(1, 0, 2)
    tv = torch.from_numpy(oracle.to_double(v, dtype)).permute(1, 0, 2)
    ref = sdpa64(tq, tk, tv, 1.0 / math.sqrt(d))[:, 0, :].numpy()
    np.testing.assert_allclose(mine, ref, rtol=0, atol=1e-12)


# ------------------------------------------------------- paged == brute force

@pytest.mark.parametrize("ctx", [1, 15, 16, 17, 32, 33, 100])
def test_paged_decode_equals_dense_on_random_tables(ctx):
    rng = np.random.default_rng(ctx)
    dtype, Hq, Hkv, d, NB = "bf16", 8, 2, 64, 24
    nblk = -(-ctx // BS)
    table = rng.permutation(NB)[:nblk].astype(np.int32)
    q = rand_bits(rng, (1, Hq, d), dtype)
    k = rand_bits(rng, (ctx, Hkv, d), dtype)
    v = rand_bits(rng, (ctx, Hkv, d), dtype)
    kc, vc = place(k, v, table, NB, NAN_BITS[dtype])
    paged = oracle.decode(q, kc, vc, table[None, :], np.array([ctx], np.int32), dtype)
    dense = oracle.dense(q[0], k, v, dtype)
    assert np.array_equal(paged[0], dense)          # same arithmetic order: bit-equal
    assert np.all(np.isfinite(paged))                # NaN tail never read


def test_identity_table_on_contiguous_pool_equals_dense():
    rng = np.random.default_rng(3)
    dtype, Hq, Hkv, d, ctx = "fp16", 4, 4, 64, 64
    table = np.arange(ctx // BS, dtype=np.int32)
    k = rand_bits(rng, (ctx, Hkv, d), dtype)
    v = rand_bits(rng, (ctx, Hkv, d), dtype)
    q = rand_bits(rng, (1, Hq, d), dtype)
    # contiguous pool: block b holds tokens 16b..16b+15 in [NB, Hkv, BS, d]
    kc = k.reshape(ctx // BS, BS, Hkv, d).transpose(0, 2, 1, 3).copy()
    vc = v.reshape(ctx // BS, BS, Hkv, d).transpose(0, 2, 1, 3).copy()
    out = oracle.decode(q, kc, vc, table[None], np.array([ctx], np.int32), dtype)
    assert np.array_equal(out[0], oracle.dense(q[0], k, v, dtype))


def test_block_permutation_invariance():
    st = make_step("llama1b", S=6)
    # attend only the prior context (append not applied): use ctx - 1
    ctx = st.context_lens - 1
    ref = oracle.decode(st.q, st.k_cache, st.v_cache, st.block_tables, ctx, st.dtype)
    rng = np.random.default_rng(11)
    perm = rng.permutation(st.NB)               # new id of old block b is perm[b]
    kc = np.empty_like(st.k_cache)
    vc = np.empty_like(st.v_cache)
    kc[perm] = st.k_cache
    vc[perm] = st.v_cache
    tables = np.where(st.block_tables >= 0, perm[np.maximum(st.block_tables, 0)], -1).astype(np.int32)
    out = oracle.decode(st.q, kc, vc, tables, ctx, st.dtype)
    assert np.array_equal(out, ref)


def test_copy_blocks_hand_worked_and_swap_round_trip_keeps_attention():
    # hand-worked: three 1-element blocks, pairs applied in order
    src = np.array([[10], [11], [12]], np.uint16)
    dst = np.zeros((4, 1), np.uint16)
    oracle.copy_blocks(src, dst, [[2, 0], [0, 3], [2, 1]])
    assert dst[:, 0].tolist() == [12, 12, 0, 10]
    # swap every sequence's blocks out to a host pool, back into fresh ids:
    # attention through the rewritten tables is unchanged
    st = make_step("llama1b", S=6)
    ctx = st.context_lens - 1
    ref = oracle.decode(st.q, st.k_cache, st.v_cache, st.block_tables, ctx, st.dtype)
    used = np.unique(st.block_tables[st.block_tables >= 0])
    host_k = np.zeros((len(used),) + st.k_cache.shape[1:], np.uint16)
    host_v = np.zeros_like(host_k)
    out_pairs = np.stack([used, np.arange(len(used))], 1)
    oracle.copy_blocks(st.k_cache, host_k, out_pairs)
    oracle.copy_blocks(st.v_cache, host_v, out_pairs)
    fresh = np.random.default_rng(2).permutation(st.NB)[:len(used)]
    kc = np.full_like(st.k_cache, NAN_BITS[st.dtype])
    vc = kc.copy()
    in_pairs = np.stack([np.arange(len(used)), fresh], 1)
    oracle.copy_blocks(host_k, kc, in_pairs)
    oracle.copy_blocks(host_v, vc, in_pairs)
    new_id = dict(zip(used.tolist(), fresh.tolist()))
    tables = np.vectorize(lambda b: new_id.get(int(b), -1))(st.block_tables).astype(np.int32)
    assert np.array_equal(oracle.decode(st.q, kc, vc, tables, ctx, st.dtype), ref)


# ------------------------------------------------------------- closed forms

@pytest.mark.parametrize("dtype,Hq,Hkv,d", [("fp16", 4, 4, 64), ("bf16", 32, 8, 128), ("bf16", 16, 2, 64)])
def test_one_hot_selects_exactly_one_value_row(dtype, Hq, Hkv, d):
    """q_h = 256 e_r (r = h mod G); K[t, g, r] = 256 only at the selected token
    of (g, r), zero elsewhere; every other score is 0, the gap >= 8192 makes
    exp underflow to 0 in double, so the output IS the selected V row.  The
    tail of the last block holds decoys with an even larger score."""
    rng = np.random.default_rng(5)
    G = Hq // Hkv
    S, NB = 3, 40
    ctxs = np.array([17, 33, 5], np.int32)
    one = rne_bits(np.float32([256.0]), dtype)[0]
    big = rne_bits(np.float32([1024.0]), dtype)[0]
    zero = np.uint16(0)
    perm = rng.permutation(NB)
    max_blocks = 4
    tables = np.full((S, max_blocks), -1, np.int32)
    kc = np.full((NB, Hkv, BS, d), zero, np.uint16)
    vc = rand_bits(rng, (NB, Hkv, BS, d), dtype)
    q = np.zeros((S, Hq, d), np.uint16)
    expect = np.zeros((S, Hq, d))
    used = 0
    for s in range(S):
        nb = -(-ctxs[s] // BS)
        tables[s, :nb] = perm[used:used + nb]
        used += nb
        # decoys past the context in the last block: huge score for every head
        for t in range(ctxs[s], nb * BS):
            for g in range(Hkv):
                kc[tables[s, t // BS], g, t % BS, :G] = big
        for h in range(Hq):
            g, r = h // G, h % G
            q[s, h, r] = one
            t_sel = int(rng.integers(0, ctxs[s]))
            # other heads of the group may select other tokens in other dims
            kc[tables[s, t_sel // BS], g, t_sel % BS, r] = one
    # expected: recompute which token each head selected from the K pattern
    for s in range(S):
        for h in range(Hq):
            g, r = h // G, h % G
            hits = [t for t in range(ctxs[s]) if kc[tables[s, t // BS], g, t % BS, r] == one]
            assert len(hits) == 1          # one selected token per (KV head, dim)
            t_sel = hits[0]
            expect[s, h] = oracle.to_double(vc[tables[s, t_sel // BS], g, t_sel % BS], dtype)
    out = oracle.decode(q, kc, vc, tables, ctxs, dtype)
    assert np.array_equal(out, expect)


@pytest.mark.parametrize("ctx", [1, 16, 17, 8192])
def test_uniform_weights_give_the_mean_of_values(ctx):
    rng = np.random.default_rng(ctx)
    dtype, Hq, Hkv, d = "bf16", 2, 1, 64
    nb = -(-ctx // BS)
    NB = nb + 3
    table = rng.permutation(NB)[:nb].astype(np.int32)
    k = rand_bits(rng, (ctx, Hkv, d), dtype)
    v = rand_bits(rng, (ctx, Hkv, d), dtype)
    kc, vc = place(k, v, table, NB, NAN_BITS[dtype])
    q = np.zeros((1, Hq, d), np.uint16)
    out = oracle.decode(q, kc, vc, table[None], np.array([ctx], np.int32), dtype)
    mean = oracle.to_double(v, dtype).mean(axis=0)[0]
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], mean, rtol=0, atol=1e-13)


@pytest.mark.parametrize("d", [64, 128])
def test_two_token_logistic_weight_pins_the_scale(d):
    """Two keys with q.k1 = a and q.k2 = b: weight of token 1 is
    1 / (1 + exp(-(a - b) / sqrt(d)))."""
    dtype = "fp16"
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = 2.0
    k = np.zeros((2, 1, d), np.float32)
    k[0, 0, 0] = 3.0      # a = 6
    k[1, 0, 0] = -1.5     # b = -3
    v = np.zeros((2, 1, d), np.float32)
    v[0, 0, :] = 1.0
    v[1, 0, :] = -2.0
    qb, kb, vb = (rne_bits(x, dtype) for x in (q, k, v))
    kc, vc = place(kb, vb, np.array([5], np.int32), 8, NAN_BITS[dtype])
    out = oracle.decode(qb, kc, vc, np.array([[5]], np.int32), np.array([2], np.int32), dtype)
    w = 1.0 / (1.0 + math.exp(-(6.0 - (-3.0)) / math.sqrt(d)))
    np.testing.assert_allclose(out[0, 0], w * 1.0 + (1 - w) * -2.0, rtol=0, atol=1e-14)
    # an explicit scale overrides 1/sqrt(d)
    out2 = oracle.decode(qb, kc, vc, np.array([[5]], np.int32), np.array([2], np.int32), dtype, scale=0.5)
    w2 = 1.0 / (1.0 + math.exp(-0.5 * 9.0))
    np.testing.assert_allclose(out2[0, 0], w2 - 2 * (1 - w2), rtol=0, atol=1e-14)


def test_zero_context_gives_zeros():
    rng = np.random.default_rng(0)
    q = rand_bits(rng, (2, 4, 64), "fp16")
    kc = np.full((4, 4, BS, 64), NAN_BITS["fp16"], np.uint16)
    out = oracle.decode(q, kc, kc, np.full((2, 1), -1, np.int32), np.array([0, 0], np.int32), "fp16")
    assert np.array_equal(out, np.zeros_like(out))


# ---------------------------------------------------------- split and merge

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_split_ranges_merged_by_lse_equal_unsplit(seed):
    st = make_step("llama1b", S=3)
    rng = np.random.default_rng(seed)
    ctx = st.context_lens - 1
    full = oracle.decode(st.q, st.k_cache, st.v_cache, st.block_tables, ctx, st.dtype)
    for s in range(st.S):
        n = int(ctx[s])
        cuts = np.sort(rng.choice(np.arange(1, n), size=min(5, n - 1), replace=False))
        edges = [0] + cuts.tolist() + [n]
        parts = [oracle.decode_range(st.q[s], st.k_cache, st.v_cache, st.block_tables[s], a, b, st.dtype)
                 for a, b in zip(edges[:-1], edges[1:])]
        # an empty range must be neutral
        parts.append(oracle.decode_range(st.q[s], st.k_cache, st.v_cache, st.block_tables[s], 3, 3, st.dtype))
        for h in range(st.Hq):
            m = np.array([p[0][h] for p in parts])
            l = np.array([p[1][h] for p in parts])
            acc = np.stack([p[2][h] for p in parts])
            merged = oracle.merge(m, l, acc)
            np.testing.assert_allclose(merged, full[s, h], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- prefill

def test_prefill_with_one_query_equals_decode():
    st = make_step("llama1b", S=5)
    cu = np.arange(st.S + 1, dtype=np.int32)
    pre = oracle.prefill(st.q, cu, st.k_cache, st.v_cache, st.block_tables, st.context_lens - 1,
                         st.dtype)
    dec = oracle.decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens - 1, st.dtype)
    assert np.array_equal(pre, dec)


@pytest.mark.parametrize("prior,q_len", [(0, 40), (0, 1), (23, 17), (64, 32), (5, 1)])
def test_prefill_matches_sdpa_lower_right_causal(prior, q_len):
    rng = np.random.default_rng(prior * 100 + q_len)
    dtype, Hq, Hkv, d = "bf16", 8, 2, 64
    ctx = prior + q_len
    nb = -(-ctx // BS)
    NB = nb + 5
    table = rng.permutation(NB)[:nb].astype(np.int32)
    k = rand_bits(rng, (ctx, Hkv, d), dtype)
    v = rand_bits(rng, (ctx, Hkv, d), dtype)
    q = rand_bits(rng, (q_len, Hq, d), dtype)
    kc, vc = place(k, v, table, NB, NAN_BITS[dtype])
    out = oracle.prefill(q, np.array([0, q_len], np.int32), kc, vc, table[None],
                         np.array([ctx], np.int32), dtype)
    tq = torch.from_numpy(oracle.to_double(q, dtype)).permute(1, 0, 2)
    tk = torch.from_numpy(oracle.to_double(k, dtype)).permute(1, 0, 2)
    tv = torch.from_numpy(oracle.to_double(v, dtype)).permute(1, 0, 2)
    ref = sdpa64(tq, tk, tv, 1.0 / math.sqrt(d), mask=causal_lower_right(q_len, ctx))
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_prefill_rejects_chunk_longer_than_context():
    q = np.zeros((4, 1, 64), np.uint16)
    kc = np.zeros((2, 1, BS, 64), np.uint16)
    with pytest.raises(ValueError):
        oracle.prefill(q, np.array([0, 4], np.int32), kc, kc, np.zeros((1, 1), np.int32),
                       np.array([3], np.int32), "fp16")


# ----------------------------------------------------------------- append

def test_append_then_read_back_through_the_table():
    """Append writes where decode reads: after appending a one-hot key at the
    new position and a known value, a one-hot query returns that value."""
    rng = np.random.default_rng(9)
    dtype, Hkv, d, NB = "fp16", 2, 64, 8
    prior = np.array([17, 14, 0], np.int32)
    tables = np.array([[6, 1, -1], [3, -1, -1], [0, -1, -1]], np.int32)
    kc = np.zeros((NB, Hkv, BS, d), np.uint16)
    vc = rand_bits(rng, (NB, Hkv, BS, d), dtype)
    before_k, before_v = kc.copy(), vc.copy()
    k_new = np.zeros((4, Hkv, d), np.uint16)
    k_new[:, :, 0] = rne_bits(np.float32([256.0]), dtype)[0]
    v_new = rand_bits(rng, (4, Hkv, d), dtype)
    # slots for positions 17 (seq 0), 14 (seq 1), 0 (seq 2), plus one padding row
    slots = np.array([tables[0, 1] * BS + 1, tables[1, 0] * BS + 14, tables[2, 0] * BS + 0, -1], np.int64)
    n = oracle.append(k_new, v_new, slots, kc, vc, BS)
    assert n == 3 * Hkv
    q = np.zeros((3, Hkv, d), np.uint16)
    q[:, :, 0] = rne_bits(np.float32([256.0]), dtype)[0]
    out = oracle.decode(q, kc, vc, tables, prior + 1, dtype)
    for s in range(3):
        assert np.array_equal(out[s], oracle.to_double(v_new[s], dtype))
    # exactly 3 tokens x Hkv rows changed, nothing else
    changed_k = np.any(kc != before_k, axis=-1).sum()
    changed_v = np.any(vc != before_v, axis=-1).sum()
    assert changed_k == 3 * Hkv and changed_v == 3 * Hkv


def test_append_rejects_slot_outside_pool():
    kc = np.zeros((2, 1, BS, 64), np.uint16)
    with pytest.raises(ValueError):
        oracle.append(np.zeros((1, 1, 64), np.uint16), np.zeros((1, 1, 64), np.uint16),
                      np.array([2 * BS], np.int64), kc, kc.copy(), BS)
