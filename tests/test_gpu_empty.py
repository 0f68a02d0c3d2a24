"""Empty steps through every entry point: no sequences, no chunks, nothing
to append.  Each call returns without error, writes nothing and flags
nothing."""
import numpy as np
import pytest
import torch

from paged_kv_cache_tables_gb300 import (kv_append, paged_decode_append_attention, paged_decode_attention,
                                         paged_mixed_attention, paged_prefill_attention)

pytestmark = pytest.mark.gpu

HQ, HKV, D, NB, MB = 32, 8, 128, 64, 8


@pytest.fixture
def pool():
    kc = torch.randn((NB, HKV, 16, D), device="cuda").to(torch.bfloat16)
    return kc, kc.clone()


def test_empty_decode_and_fused_append(cuda_lib, pool):
    kc, vc = pool
    k0, v0 = kc.clone(), vc.clone()
    q = torch.empty((0, HQ, D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    bt = torch.empty((0, MB), dtype=torch.int32, device="cuda")
    cl = torch.empty(0, dtype=torch.int32, device="cuda")
    new = torch.empty((0, HKV, D), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    paged_decode_attention(out, q, kc, vc, bt, cl, dev_status=status)
    paged_decode_append_attention(out, q, new, new, kc, vc, bt, cl, dev_status=status)
    kv_append(new, new, torch.empty(0, dtype=torch.int64, device="cuda"), kc, vc, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(kc, k0) and torch.equal(vc, v0)


def test_empty_prefill_and_mixed(cuda_lib, pool):
    kc, vc = pool
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = torch.empty((0, HQ, D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = torch.empty((0, MB), dtype=torch.int32, device="cuda")
    cl = torch.empty(0, dtype=torch.int32, device="cuda")
    paged_prefill_attention(out, q, cu, 0, kc, vc, bt, cl, dev_status=status)
    paged_mixed_attention(out, q, cu, 0, 0, kc, vc, bt, cl, dev_status=status,
                          cu_seqlens_host=np.zeros(1, np.int32), context_lens_host=np.zeros(0, np.int32))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
