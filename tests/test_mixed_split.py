"""pkv_mixed_split: the host-side choice of how many SMs the decode kernel
gets when a mixed step runs its prefill and decode kernels side by side (a
scheduling heuristic, not part of the attention arithmetic)."""
import numpy as np
import pytest

from paged_kv_cache_tables_gb300 import PkvError, mixed_split


def split(priors, q_lens, dec_ctx, sms=152):
    priors, q_lens = np.asarray(priors), np.asarray(q_lens)
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    ctx = np.concatenate([priors + q_lens, dec_ctx])
    return mixed_split(sms, cu, len(q_lens), ctx, 32, 8, 128)


def test_one_kind_of_work_takes_everything():
    assert split([], [], [1000] * 10) == 152
    assert split([100], [512], []) == 0


def test_split_follows_the_work():
    base = split([2000] * 8, [512] * 8, [2000] * 248)
    assert 1 <= base <= 151
    assert split([2000] * 8, [512] * 8, [4000] * 248) >= base      # more decode bytes
    assert split([4000] * 8, [512] * 8, [2000] * 248) <= base      # more prefill work
    assert split([2000] * 2, [512] * 2, [2000] * 248) >= base      # less prefill work


def test_split_stays_inside_the_gpu():
    for dec in ([1] * 2, [8000] * 4000):
        for pri in ([0], [8000] * 64):
            d = split(pri, [512] * len(pri), dec)
            assert 1 <= d <= 151


def test_bad_arguments():
    with pytest.raises(PkvError):
        mixed_split(1, np.zeros(2), 1, np.zeros(3), 32, 8, 128)
