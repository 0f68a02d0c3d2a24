"""Helpers for the GPU parity tests: move synth arrays to the device, run the
C-ABI calls, and compare with the oracle under the stated tolerance.

Tolerance (from the 2e-3 max-abs target on fp32-accumulated outputs):
  * fp32 output: |gpu - oracle| <= 2e-3 everywhere;
  * 16-bit output: |gpu - oracle| <= max(2e-3, ulp(oracle)/2 + 1e-4), because a
    correctly rounded bf16 value near 1 is already 2^-8 = 3.9e-3 away at worst.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

ATOL = 2e-3
# Two splits of the same decode agree to fp32 rounding plus the rounding of
# the softmax weights P, which each split forms against its own running
# maximum as a 16-bit value and its 16-bit residual (about 16 significant
# bits): |a - b| <= SPLIT_ATOL + SPLIT_RTOL * |b|.  A range merged with a
# piece missing or doubled is off by 1e-3 or more.
SPLIT_ATOL = 2e-6
SPLIT_RTOL = 2.0 ** -15


def split_excess(a, b):
    """How far two decode outputs (torch tensors) of different splits exceed
    the split tolerance: max of |a - b| - (SPLIT_ATOL + SPLIT_RTOL |b|), NaN
    counted as a large excess.  <= 0 means they agree."""
    d = (a - b).abs() - (SPLIT_ATOL + SPLIT_RTOL * b.abs())
    return float(d.nan_to_num(1e9).max())
TORCH_DT = {"fp16": torch.float16, "bf16": torch.bfloat16}
MANT_BITS = {"fp16": 10, "bf16": 7}


def dev_bits(bits, dtype):
    """uint16 bit patterns -> CUDA tensor of the 16-bit dtype (same bits)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(TORCH_DT[dtype]).cuda()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def out_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def half_ulp(x, dtype):
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 1e-30)))
    if dtype == "fp16":
        e = np.maximum(e, -14)
    return np.exp2(e - MANT_BITS[dtype] - 1)


def assert_close(gpu, ref, out_dtype, dtype=None, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(gpu)), "%s: non-finite output" % what
    err = np.abs(gpu - ref)
    if out_dtype == "fp32":
        bound = np.full_like(ref, ATOL)
    else:
        bound = np.maximum(ATOL, half_ulp(ref, out_dtype) + 1e-4)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError("%s: %d elements over tolerance; worst at %s: gpu %.6g ref %.6g err %.3g bound %.3g"
                             % (what, bad.sum(), i, gpu[i], ref[i], err[i], bound[i]))
    return float(err.max())


class DeviceStep:
    """A synth.Step resident on the GPU."""

    def __init__(self, st):
        self.st = st
        dt = st.dtype
        self.q = dev_bits(st.q, dt)
        self.k_new = dev_bits(st.k_new, dt)
        self.v_new = dev_bits(st.v_new, dt)
        self.k_cache = dev_bits(st.k_cache, dt)
        self.v_cache = dev_bits(st.v_cache, dt)
        self.slot_mapping = dev(st.slot_mapping)
        self.block_tables = dev(st.block_tables)
        self.context_lens = dev(st.context_lens)
        self.cu_seqlens = dev(st.cu_seqlens)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")


def oracle_decode_all(q, k_cache, v_cache, block_tables, context_lens, dtype, scale=None):
    """oracle.decode over every sequence of a step, the sequences split into
    slices of about equal attended tokens run side by side on host threads
    (the oracle's C loops run outside the GIL).  The oracle itself is
    unchanged: each slice is one plain call."""
    S = q.shape[0]
    threads = max(1, min(len(os.sched_getaffinity(0)), 16, S))
    cum = np.concatenate([[0], np.cumsum(np.asarray(context_lens, np.int64))])
    cuts = sorted(set([0, S] + [int(np.searchsorted(cum, cum[-1] * k / threads)) for k in range(1, threads)]))
    out = np.empty((S,) + q.shape[1:], np.float64)

    def run(lo_hi):
        lo, hi = lo_hi
        out[lo:hi] = oracle.decode(q[lo:hi], k_cache, v_cache, block_tables[lo:hi], context_lens[lo:hi], dtype,
                                   scale=scale)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(run, [(cuts[i], cuts[i + 1]) for i in range(len(cuts) - 1) if cuts[i + 1] > cuts[i]]))
    return out


def oracle_prefill_all(q, cu_seqlens, k_cache, v_cache, block_tables, context_lens, dtype, scale=None):
    """oracle.prefill over every chunk of a step, one plain oracle call per
    chunk, run side by side on host threads (longest first)."""
    n = len(cu_seqlens) - 1
    out = np.empty((int(cu_seqlens[n]),) + q.shape[1:], np.float64)
    threads = max(1, min(len(os.sched_getaffinity(0)), 16, n))

    def run(c):
        lo, hi = int(cu_seqlens[c]), int(cu_seqlens[c + 1])
        out[lo:hi] = oracle.prefill(q[lo:hi], np.array([0, hi - lo], np.int32), k_cache, v_cache,
                                    block_tables[c:c + 1], context_lens[c:c + 1], dtype, scale=scale)

    work = sorted(range(n), key=lambda c: -int(context_lens[c]) * int(cu_seqlens[c + 1] - cu_seqlens[c]))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(run, work))
    return out
