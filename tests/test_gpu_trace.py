"""End-to-end engine loop on the GPU: the native scheduler drives append,
chunked prefill and decode over several layers for a request trace; sampled
layer-0 attention rows are checked against the FP64 oracle on K/V rebuilt from
the counter-based generator (so the check covers the scheduler's tables and
slots, every append, preemption by recompute or by swap and both attention
kernels)."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close
from oracle.trace_check import layer0_row
from paged_kv_cache_tables_gb300.engine import PagedEngine, run_trace
from synth import build as synth_build
from synth.trace import fill_rows_gpu, make_fill, make_requests, pick_rows, token_rows, kv_tag, q_tag

pytestmark = pytest.mark.gpu

HQ, HKV, D = 32, 8, 128


@pytest.fixture(scope="module")
def synth_gpu():
    synth_build.build()


def test_gpu_generator_matches_numpy(cuda_lib, synth_gpu):
    rids = torch.tensor([0, 7, 123456789012, 3], dtype=torch.int64, device="cuda")
    pos = torch.tensor([0, 15, 4095, 77], dtype=torch.int32, device="cuda")
    out = torch.empty((4, HKV, D), dtype=torch.bfloat16, device="cuda")
    for tag in (kv_tag(0, "k"), kv_tag(3, "v"), q_tag(31)):
        fill_rows_gpu(out, rids, pos, tag)
        torch.cuda.synchronize()
        got = out.cpu().view(torch.int16).numpy().view(np.uint16).reshape(4, -1)
        ref = token_rows(rids.cpu().numpy(), pos.cpu().numpy(), tag, HKV * D, "bf16")
        assert np.array_equal(got, ref)


def test_gpu_qkv_generator_matches_numpy(cuda_lib, synth_gpu):
    from synth.trace import fill_qkv_gpu
    rids = torch.tensor([5, 0, 99999999999, 7, 3], dtype=torch.int64, device="cuda")
    pos = torch.tensor([3, 0, 4095, 16, 17], dtype=torch.int32, device="cuda")
    q = torch.empty((5, HQ, D), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((5, HKV, D), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    tags = (q_tag(3), kv_tag(1, "k"), kv_tag(1, "v"))
    fill_qkv_gpu(q, k, v, rids, pos, *tags)
    torch.cuda.synchronize()
    for t, tag in zip((q, k, v), tags):
        got = t.cpu().view(torch.int16).numpy().view(np.uint16).reshape(5, -1)
        assert np.array_equal(got, token_rows(rids.cpu().numpy(), pos.cpu().numpy(), tag, got.shape[1], "bf16"))


def run(n, rate, prompt_mean, out_mean, NB, layers, caches, max_batch, budget, chunk, mml, seed, **kw):
    arrival, prompt, eos = make_requests(seed, n=n, rate=rate, prompt_mean=prompt_mean, out_mean=out_mean,
                                         pmax=mml // 2)
    eng = PagedEngine(NB, num_layers=layers, num_caches=caches, Hq=HQ, Hkv=HKV, d=D, max_batch=max_batch,
                      max_num_batched_tokens=budget, chunk=chunk, max_model_len=mml,
                      initial_order=np.random.default_rng(seed).permutation(NB), **kw)
    rng = np.random.default_rng(seed + 1)
    res = run_trace(eng, arrival, prompt, eos, max_tokens=mml, fill=make_fill(), sample_every=4,
                    pick=lambda info: pick_rows(info, rng))
    return eng, res, (arrival, prompt, eos)


def check_samples(res):
    checked = 0
    for rows, vals in res["samples"]:
        for (row, rid, pos), got in zip(rows, vals.numpy()):
            ref = layer0_row(rid, pos, HQ, HKV, D)
            assert_close(got, ref, "bf16", what="rid %d pos %d" % (rid, pos))
            checked += 1
    return checked


def test_trace_runs_to_completion_and_matches_oracle(cuda_lib, synth_gpu):
    eng, res, (arrival, prompt, eos) = run(n=48, rate=6, prompt_mean=120, out_mean=10, NB=4096, layers=3, caches=2,
                                           max_batch=16, budget=256, chunk=64, mml=1024, seed=5)
    assert len(res["finish_step"]) == 48
    assert int(eng.status.item()) == 0
    st = eng.sched.stats()
    assert st["free_blocks"] == 4096 and st["running"] == 0 and st["waiting"] == 0
    assert any(s["P"] > 0 for s in res["steps"]) and any(s["S"] > s["P"] for s in res["steps"])
    assert check_samples(res) >= 20


def test_trace_under_memory_pressure_preempts_and_recomputes_exactly(cuda_lib, synth_gpu):
    eng, res, _ = run(n=40, rate=8, prompt_mean=150, out_mean=40, NB=96, layers=2, caches=2, max_batch=16,
                      budget=512, chunk=128, mml=512, seed=9)
    assert len(res["finish_step"]) == 40
    st = eng.sched.stats()
    assert st["preemptions"] > 0
    assert st["free_blocks"] == 96
    assert int(eng.status.item()) == 0
    assert check_samples(res) >= 10


def test_trace_under_memory_pressure_swaps_blocks_out_and_back(cuda_lib, synth_gpu):
    """Preemption by swap: the victims' blocks go to pinned host memory and
    come back into other physical blocks on re-admission; every sampled row
    read through the restored blocks equals the oracle, and the prompts are
    prefilled fewer times than with recompute."""
    from paged_kv_cache_tables_gb300 import PREEMPT_SWAP
    cfg = dict(n=40, rate=8, prompt_mean=150, out_mean=40, NB=96, layers=2, caches=2, max_batch=16, budget=512,
               chunk=128, mml=512, seed=9)
    eng, res, _ = run(**cfg, preemption=PREEMPT_SWAP, swap_blocks=400)
    st = eng.sched.stats()
    assert len(res["finish_step"]) == 40 and int(eng.status.item()) == 0
    assert st["preemptions"] > 0 and st["swapped_out_blocks"] > 0
    assert st["swapped_in_blocks"] == st["swapped_out_blocks"]
    assert st["free_blocks"] == 96 and st["free_swap_slots"] == 400
    assert check_samples(res) >= 10
    rec, _, _ = run(**cfg)
    assert st["prefill_tokens"] < rec.sched.stats()["prefill_tokens"]


def test_trace_with_small_swap_space_mixes_swap_and_recompute(cuda_lib, synth_gpu):
    """With fewer host slots than the victims need, some preemptions fall back
    to recompute; the outputs stay exact either way."""
    from paged_kv_cache_tables_gb300 import PREEMPT_SWAP
    eng, res, _ = run(n=40, rate=8, prompt_mean=150, out_mean=40, NB=96, layers=2, caches=2, max_batch=16,
                      budget=512, chunk=128, mml=512, seed=11, preemption=PREEMPT_SWAP, swap_blocks=12)
    st = eng.sched.stats()
    assert len(res["finish_step"]) == 40 and int(eng.status.item()) == 0
    assert st["swapped_out_blocks"] > 0 and st["free_swap_slots"] == 12 and st["free_blocks"] == 96
    assert check_samples(res) >= 10


def run_shared(n, NB, caching, seed, layers=2, max_batch=16, budget=256, chunk=64, mml=1024):
    from synth.trace import content_keys, make_shared_requests
    arrival, prompt, eos, tokens, head_len, group = make_shared_requests(
        seed, n=n, rate=6, groups=3, head_mean=96, tail_mean=30, out_mean=10, pmax=mml // 2)
    eng = PagedEngine(NB, num_layers=layers, num_caches=2, Hq=HQ, Hkv=HKV, d=D, max_batch=max_batch,
                      max_num_batched_tokens=budget, chunk=chunk, max_model_len=mml,
                      initial_order=np.random.default_rng(seed).permutation(NB), prefix_caching=caching,
                      row_keys=lambda r, p: content_keys(r, p, head_len, group))
    rng = np.random.default_rng(seed + 1)
    res = run_trace(eng, arrival, prompt, eos, max_tokens=mml, fill=make_fill(), sample_every=3,
                    pick=lambda info: pick_rows(info, rng), tokens=tokens)
    checked = 0
    for rows, vals in res["samples"]:
        for (row, rid, pos), got in zip(rows, vals.numpy()):
            ref = layer0_row(rid, pos, HQ, HKV, D, keys=lambda ps, r=rid: content_keys(np.full(len(ps), r), ps,
                                                                                       head_len, group))
            assert_close(got, ref, "bf16", what="rid %d pos %d" % (rid, pos))
            checked += 1
    return eng, res, checked


def test_prefix_cached_trace_reads_shared_pages_correctly(cuda_lib, synth_gpu):
    """Requests sharing prompt heads: with prefix caching their block tables
    point at the same physical pages, written once; every sampled row still
    equals the oracle on the request's own (content-keyed) rows."""
    eng, res, checked = run_shared(48, 4096, True, seed=21)
    st = eng.sched.stats()
    assert len(res["finish_step"]) == 48 and int(eng.status.item()) == 0
    assert st["prefix_hit_blocks"] > 20 and st["cached_blocks"] == 0 and st["free_blocks"] == 4096
    assert checked >= 20
    # the same trace without sharing computes more prefill tokens
    eng2, _, _ = run_shared(48, 4096, False, seed=21)
    assert eng2.sched.stats()["prefill_tokens"] > st["prefill_tokens"]


def test_prefix_cached_trace_under_memory_pressure(cuda_lib, synth_gpu):
    eng, res, checked = run_shared(40, 60, True, seed=23, budget=512, chunk=128, mml=512)
    st = eng.sched.stats()
    assert len(res["finish_step"]) == 40 and int(eng.status.item()) == 0
    assert st["preemptions"] > 0 and st["prefix_hit_blocks"] > 0 and st["free_blocks"] == 60
    assert checked >= 10


@pytest.mark.parametrize("Hq,Hkv,d,dtype", [(8, 8, 64, "fp16"), (16, 2, 128, "fp16"), (12, 4, 64, "bf16")])
def test_trace_other_shapes_and_types(cuda_lib, synth_gpu, Hq, Hkv, d, dtype):
    """The engine loop on other head layouts, head sizes and 16-bit types, under
    memory pressure with swapping: every sampled row against the oracle."""
    from paged_kv_cache_tables_gb300 import PREEMPT_SWAP
    seed = Hq * 100 + d
    arrival, prompt, eos = make_requests(seed, n=30, rate=6, prompt_mean=150, out_mean=30, pmax=256)
    eng = PagedEngine(80, num_layers=2, num_caches=2, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype, max_batch=12,
                      max_num_batched_tokens=384, chunk=96, max_model_len=512,
                      initial_order=np.random.default_rng(seed).permutation(80), preemption=PREEMPT_SWAP,
                      swap_blocks=200)
    rng = np.random.default_rng(seed + 1)
    res = run_trace(eng, arrival, prompt, eos, max_tokens=512, fill=make_fill(), sample_every=3,
                    pick=lambda info: pick_rows(info, rng))
    st = eng.sched.stats()
    assert len(res["finish_step"]) == 30 and int(eng.status.item()) == 0
    assert st["free_blocks"] == 80 and st["free_swap_slots"] == 200
    assert st["preemptions"] > 0 and st["swapped_out_blocks"] > 0
    checked = 0
    for rows, vals in res["samples"]:
        for (row, rid, pos), got in zip(rows, vals.numpy()):
            ref = layer0_row(rid, pos, Hq, Hkv, d, dtype=dtype)
            assert_close(got, ref, dtype, what="%d/%d d%d %s rid %d pos %d" % (Hq, Hkv, d, dtype, rid, pos))
            checked += 1
    assert checked >= 10
