"""libpkv.so loads on a machine without a GPU and exports every symbol that
include/pkv.h declares; host-only entry points work there; device entry points
reject bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_tables_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["pkv_kv_append", "pkv_paged_decode_attention", "pkv_paged_prefill_attention",
                     "pkv_decode_workspace_size", "pkv_status_string", "pkv_sched_step", "pkv_pool_alloc"]:
        assert required in names


def test_every_declared_symbol_is_exported():
    L = _binding.lib()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings():
    L = _binding.lib()
    assert L.pkv_status_string(0) == b"PKV_OK"
    assert L.pkv_status_string(-3) == b"PKV_ERR_WORKSPACE"
    assert L.pkv_status_string(-7) == b"PKV_ERR_NO_MEMORY"
    assert L.pkv_status_string(12345) == b"PKV_ERR_UNKNOWN"
    assert b"sm_103a" in L.pkv_version()


def test_device_entry_points_validate_before_launch():
    L = _binding.lib()
    P = ctypes.c_void_p
    fake = P(1 << 20)       # never dereferenced: validation fails first
    # unsupported head_dim
    assert L.pkv_kv_append(fake, fake, fake, 4, fake, fake, 8, 16, 2, 96, 1, None, None) == -2
    # block_size other than 16
    assert L.pkv_kv_append(fake, fake, fake, 4, fake, fake, 8, 8, 2, 64, 1, None, None) == -2
    # zero tokens is a no-op
    assert L.pkv_kv_append(None, None, None, 0, None, None, 8, 16, 2, 64, 1, None, None) == 0
    # Hq not a multiple of Hkv
    assert L.pkv_paged_decode_attention(fake, fake, fake, fake, fake, 4, fake, 2, 8, 6, 4, 64, 16, 0.125, 1, 1,
                                        fake, 1 << 20, None, None) == -1
    # group of 32 query heads per KV head is not built
    assert L.pkv_paged_decode_attention(fake, fake, fake, fake, fake, 4, fake, 2, 8, 32, 1, 64, 16, 0.125, 1, 1,
                                        fake, 1 << 20, None, None) == -2
    # fp32 inputs are not a supported dtype
    assert L.pkv_paged_decode_attention(fake, fake, fake, fake, fake, 4, fake, 2, 8, 8, 8, 64, 16, 0.125, 2, 2,
                                        fake, 1 << 20, None, None) == -2
    # NaN scale
    assert L.pkv_paged_decode_attention(fake, fake, fake, fake, fake, 4, fake, 2, 8, 8, 8, 64, 16, float("nan"), 1, 1,
                                        fake, 1 << 20, None, None) == -1
    # zero sequences is a no-op
    assert L.pkv_paged_decode_attention(None, None, None, None, None, 4, None, 0, 8, 8, 8, 64, 16, 0.125, 1, 1,
                                        None, 0, None, None) == 0


def test_workspace_size_without_a_device_is_zero():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert _binding.decode_workspace_size(4, 32, 8, 128) == 0


def test_newer_entry_points_validate_before_launch():
    L = _binding.lib()
    P = ctypes.c_void_p
    fake = P(1 << 20)
    # fused decode + append: k_new without v_new, and zero sequences
    assert L.pkv_paged_decode_append_attention(fake, fake, fake, None, fake, fake, fake, 4, fake, 2, 8, 8, 8, 64, 16,
                                               0.125, 1, 1, fake, 1 << 20, None, None) == -1
    assert L.pkv_paged_decode_append_attention(None, None, None, None, None, None, None, 4, None, 0, 8, 8, 8, 64, 16,
                                               0.125, 1, 1, None, 0, None, None) == 0
    # one-call mixed step: no k_new, an empty step, negative counts
    args_tail = [fake, fake, fake, 4, fake, 8, 8, 8, 64, 16, 0.125, 1, 1, fake, 1 << 20, None, None, 0, None, None]
    assert L.pkv_paged_mixed_append_attention(fake, fake, None, fake, fake, fake, 1, 16, 16, 1, *args_tail) == -1
    assert L.pkv_paged_mixed_append_attention(fake, fake, fake, fake, fake, fake, 0, 0, 0, 0, *args_tail) == 0
    assert L.pkv_paged_mixed_append_attention(fake, fake, fake, fake, fake, fake, -1, 0, 0, 1, *args_tail) == -1
    # side-by-side entry: null output with work to do
    assert L.pkv_paged_mixed_attention(None, fake, fake, 1, 16, 16, 1, fake, fake, fake, 4, fake, 8, 8, 8, 64, 16,
                                       0.125, 1, 1, fake, 1 << 20, None, None, 0, None, None) == -1
    # block mover: a block size that is not a multiple of 16 bytes, and no pairs
    assert L.pkv_copy_blocks(fake, 4, fake, 4, fake, 2, 24, None, None) == -1
    assert L.pkv_copy_blocks(None, 4, None, 4, None, 0, 4096, None, None) == 0
    # prefill: unsupported block size
    assert L.pkv_paged_prefill_attention(fake, fake, fake, 1, 16, 16, fake, fake, fake, 4, fake, 8, 8, 8, 64, 8,
                                         0.125, 1, 1, None, None) == -2


def test_mixed_split_picks_all_sms_without_prefill_and_none_without_decode():
    L = _binding.lib()
    import numpy as np
    cu = np.array([0, 512], np.int32)
    ctx = np.array([1024, 500, 700], np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    assert L.pkv_mixed_split(152, p(cu), 0, p(ctx), 3, 32, 8, 128, 2) == 152
    assert L.pkv_mixed_split(152, p(cu), 1, p(ctx), 0, 32, 8, 128, 2) == 0
    d = L.pkv_mixed_split(152, p(cu), 1, p(ctx), 2, 32, 8, 128, 2)
    assert 1 <= d < 152
