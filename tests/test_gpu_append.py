"""GPU parity of pkv_kv_append (K1): bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceStep, dev, dev_bits, host_bits
from paged_kv_cache_tables_gb300 import kv_append
from synth import NAN_BITS, make_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("llama1b", {"S": 64}), ("mixed", {"NB": 65536})])
def test_append_is_bit_exact(cuda_lib, name, kw):
    st = make_step(name, **kw)
    ds = DeviceStep(st)
    kv_append(ds.k_new, ds.v_new, ds.slot_mapping, ds.k_cache, ds.v_cache, dev_status=ds.status)
    torch.cuda.synchronize()
    kc, vc = st.k_cache.copy(), st.v_cache.copy()
    n = oracle.append(st.k_new, st.v_new, st.slot_mapping, kc, vc, st.bs)
    assert n == st.T * st.Hkv
    assert np.array_equal(host_bits(ds.k_cache), kc)
    assert np.array_equal(host_bits(ds.v_cache), vc)
    assert int(ds.status.item()) == 0


def test_append_skips_padding_and_flags_out_of_pool_slots(cuda_lib):
    rng = np.random.default_rng(3)
    NB, Hkv, d = 8, 2, 128
    kc0 = np.full((NB, Hkv, 16, d), NAN_BITS["bf16"], np.uint16)
    k = rng.integers(0, 1 << 15, size=(5, Hkv, d), dtype=np.uint16)
    v = rng.integers(0, 1 << 15, size=(5, Hkv, d), dtype=np.uint16)
    slots = np.array([3, -1, 127, NB * 16, 40], np.int64)   # padding, last slot, one past the pool
    kc, vc = dev_bits(kc0, "bf16"), dev_bits(kc0, "bf16")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv_append(dev_bits(k, "bf16"), dev_bits(v, "bf16"), dev(slots), kc, vc, dev_status=status)
    torch.cuda.synchronize()
    ek, ev = kc0.copy(), kc0.copy()
    oracle.append(k[[0, 2, 4]], v[[0, 2, 4]], slots[[0, 2, 4]], ek, ev, 16)
    assert np.array_equal(host_bits(kc), ek)
    assert np.array_equal(host_bits(vc), ev)
    assert int(status.item()) & 8   # PKV_DEV_BAD_SLOT


def test_append_zero_tokens_is_a_no_op(cuda_lib):
    kc = torch.zeros((4, 1, 16, 64), dtype=torch.float16, device="cuda")
    e = torch.empty((0, 1, 64), dtype=torch.float16, device="cuda")
    kv_append(e, e, torch.empty(0, dtype=torch.int64, device="cuda"), kc, kc.clone())
    torch.cuda.synchronize()
    assert int(kc.abs().sum().item()) == 0
