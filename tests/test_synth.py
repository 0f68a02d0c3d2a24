"""The seeded workloads have the shapes and structure their descriptions give."""
import os

import numpy as np

import oracle
from synth import NAN_BITS, make_step, rne_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_fixture(name):
    out = {}
    for raw in open(os.path.join(GOLDEN, name)):
        line = raw.split("#", 1)[0].split()
        if line:
            out[line[0]] = [int(x) for x in line[1:]]
    return out


def test_tiny_step_metadata_matches_fixture():
    fx = read_fixture("tiny_step.txt")
    st = make_step("tiny")
    assert st.context_lens.tolist() == fx["context_lens"]
    assert ((st.context_lens + 15) // 16).tolist() == fx["blocks_needed"]
    for s in range(st.S):
        slot = int(st.slot_mapping[s])
        assert slot % 16 == fx["new_token_offset"][s]
        assert slot // 16 == st.block_tables[s, fx["new_token_block_index"][s]]
    assert st.q.shape == (2, 4, 64) and st.k_cache.shape == (64, 4, 16, 64)


def test_rne_bits_agrees_with_torch_rounding():
    import torch
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * 3).astype(np.float32)
    x[:4] = [1.00390625, 1.01171875, -1.00390625, 0.0]     # exact bf16 ties
    mine = rne_bits(x, "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    mine16 = rne_bits(x, "fp16")
    ref16 = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine16, ref16)


def test_pool_slots_without_tokens_hold_nan():
    st = make_step("llama1b", S=4)
    prior = st.context_lens - st.q_lens
    vals = oracle.to_double(st.k_cache, st.dtype)
    for s in range(st.S):
        for t in range(int(st.context_lens[s]) + 3):
            b = t // 16
            if b >= st.block_tables.shape[1] or st.block_tables[s, b] < 0:
                break
            row = vals[st.block_tables[s, b], :, t % 16, :]
            assert np.all(np.isfinite(row)) == (t < prior[s])
    used = set(st.block_tables[st.block_tables >= 0].tolist())
    unused = [b for b in range(st.NB) if b not in used][:10]
    assert np.all(st.k_cache[unused] == NAN_BITS["bf16"])


def test_llama8b_context_distribution():
    from synth import llama8b_context_lens
    ctx = llama8b_context_lens(np.random.Generator(np.random.PCG64(1002)), 256)
    assert ctx.min() >= 32 and ctx.max() <= 8192
    assert 900 < np.median(ctx) < 1150


def test_mixed_step_layout():
    st = make_step("mixed", n_chunks=2, chunk=64, n_decode=5, NB=4096)
    assert st.n_prefill == 2 and st.T == 2 * 64 + 5
    q_p, cu_p, bt_p, cl_p = st.prefill_part()
    q_d, bt_d, cl_d = st.decode_part()
    assert q_p.shape[0] == 128 and q_d.shape[0] == 5 and cu_p.tolist() == [0, 64, 128]
    assert np.all(cl_p >= 64) and np.all(cl_d >= 256)
    # every slot is unique and inside its sequence's blocks
    assert len(set(st.slot_mapping.tolist())) == st.T
