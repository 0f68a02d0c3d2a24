"""pkv_paged_decode_attention_static: decode attention for callers that cannot
allocate device memory (their engine or host framework owns every device
allocation, or cudaMalloc's possible device synchronisation is not allowed on
their path).  It runs on a scratch array the library keeps in device global
memory instead of a caller workspace.

Called through the C ABI and compared with pkv_paged_decode_attention (which
takes a caller workspace): a Llama-3.2-1B-shaped step, then a Llama-3-8B-shaped
one, so the later calls run on scratch an earlier call of another shape left
behind.  With the split fixed the two entry points agree bit for bit; with
work stealing, within rounding, on two calls in a row that change neither
torch's allocation count nor the device's free memory.  Collected last on
purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from gpu_helpers import ATOL, DeviceStep
from paged_kv_cache_tables_gb300 import paged_decode_attention
from synth import make_step

pytestmark = pytest.mark.gpu


def call_static(L, out, q, ds, dev_status):
    st = ds.st
    S, Hq, d = q.shape
    return L.pkv_paged_decode_attention_static(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(ds.k_cache.data_ptr()),
        ctypes.c_void_p(ds.v_cache.data_ptr()), ctypes.c_void_p(ds.block_tables.data_ptr()), st.max_blocks,
        ctypes.c_void_p(ds.context_lens.data_ptr()), S, st.NB, Hq, st.Hkv, d, st.bs, 1.0 / math.sqrt(d),
        1, 2, ctypes.c_void_p(dev_status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("calls", [[("llama1b", {"S": 64}), ("llama8b", {"S": 128, "NB": 16384})]])
def test_static_scratch_decode_matches_workspace_decode(cuda_lib, calls, monkeypatch):
    L = cuda_lib
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for name, kw in calls:
        st = make_step(name, **kw)
        ds = DeviceStep(st)
        ds.context_lens -= 1          # attend the stored prior context
        # with the split fixed (no work stealing) both entry points split
        # every range the same way, so the bits must agree exactly
        monkeypatch.setenv("PKV_DETERMINISTIC", "1")
        ref = torch.empty((st.S, st.Hq, st.d), dtype=torch.float32, device="cuda")
        paged_decode_attention(ref, ds.q, ds.k_cache, ds.v_cache, ds.block_tables, ds.context_lens)
        out = torch.full_like(ref, float("nan"))
        rc = call_static(L, out, ds.q, ds, status)
        assert rc == 0, L.pkv_status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "%s: fixed-split static decode differs from the workspace decode" % name
        monkeypatch.delenv("PKV_DETERMINISTIC")
        # the default (work-stealing) launch on the same scratch: equal up to
        # the rounding of the split.  The first call also warms up torch's
        # own kernels used around it (their code loads on first use and takes
        # device memory); across the next two calls in a row nothing may be
        # allocated -- neither through torch's allocator nor on the device
        def stolen_call():
            out.fill_(float("nan"))
            rc = call_static(L, out, ds.q, ds, status)
            assert rc == 0, L.pkv_status_string(rc)
            torch.cuda.synchronize()
            diff = (out - ref).abs().nan_to_num(1e9).max().item()
            assert diff <= ATOL, "%s: static-scratch decode differs by %g" % (name, diff)

        stolen_call()
        torch.cuda.synchronize()
        alloc0 = torch.cuda.memory_allocated()
        free0, _ = torch.cuda.mem_get_info()
        for _ in range(2):
            stolen_call()
        free1, _ = torch.cuda.mem_get_info()
        assert torch.cuda.memory_allocated() == alloc0
        assert free1 == free0, "%s: device free memory changed by %d bytes" % (name, free0 - free1)
        assert int(status.item()) == 0


def test_static_scratch_rejects_too_many_sequences(cuda_lib):
    L = cuda_lib
    fake = ctypes.c_void_p(1 << 20)      # never dereferenced: the size check comes first
    rc = L.pkv_paged_decode_attention_static(fake, fake, fake, fake, fake, 4, fake, 16385, 64, 32, 8, 128, 16,
                                             0.088, 1, 1, None, None)
    assert rc == -3    # PKV_ERR_WORKSPACE
    assert b"PKV_STATIC_MAX_SEQS" in L.pkv_last_cuda_error()
