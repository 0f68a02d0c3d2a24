"""GPU parity of pkv_copy_blocks, the block mover of preemption by swap:
bit-exact against the oracle's block copy, device -> pinned host and back."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_tables_gb300 import copy_blocks

pytestmark = pytest.mark.gpu


def bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("NB,Hkv,d,n", [(64, 4, 64, 1), (4096, 8, 128, 300), (1024, 8, 128, 1024)])
def test_swap_out_and_back_is_bit_exact(cuda_lib, NB, Hkv, d, n):
    rng = np.random.default_rng(NB + n)
    cache = torch.from_numpy(rng.integers(0, 1 << 16, size=(NB, Hkv, 16, d), dtype=np.uint16).view(np.int16))
    cache = cache.view(torch.bfloat16).cuda()
    host = torch.zeros((n + 7, Hkv, 16, d), dtype=torch.bfloat16).pin_memory()
    src = rng.choice(NB, size=n, replace=False).astype(np.int32)
    slots = rng.choice(n + 7, size=n, replace=False).astype(np.int32)
    out_pairs = torch.from_numpy(np.stack([src, slots], 1)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    copy_blocks(host, cache, out_pairs, dev_status=status)
    torch.cuda.synchronize()
    want_host = np.zeros((n + 7, Hkv, 16, d), np.uint16)
    oracle.copy_blocks(bits(cache), want_host, np.stack([src, slots], 1))
    assert np.array_equal(bits(host), want_host)
    # back into other device blocks; pairs in pinned memory this time
    dst = rng.choice(NB, size=n, replace=False).astype(np.int32)
    back = torch.zeros_like(cache)
    in_pairs = torch.from_numpy(np.stack([slots, dst], 1)).pin_memory()
    copy_blocks(back, host, in_pairs, dev_status=status)
    torch.cuda.synchronize()
    want = np.zeros(cache.shape, np.uint16)
    oracle.copy_blocks(want_host, want, np.stack([slots, dst], 1))
    assert np.array_equal(bits(back), want)
    assert int(status.item()) == 0


def test_out_of_range_pairs_are_skipped_and_flagged(cuda_lib):
    cache = torch.arange(8 * 2 * 16 * 64, dtype=torch.float32).to(torch.bfloat16).view(8, 2, 16, 64).cuda()
    host = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16).pin_memory()
    pairs = torch.tensor([[1, 0], [8, 1], [2, 4], [-1, 2], [3, 3]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    copy_blocks(host, cache, pairs, dev_status=status)
    torch.cuda.synchronize()
    want = np.zeros(host.shape, np.uint16)
    oracle.copy_blocks(bits(cache), want, [[1, 0], [3, 3]])
    assert np.array_equal(bits(host), want)
    assert int(status.item()) != 0


def test_empty_pair_list_launches_nothing(cuda_lib):
    cache = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    copy_blocks(cache, cache.clone(), torch.zeros((0, 2), dtype=torch.int32, device="cuda"))
