"""The benchmark's own arithmetic, on the CPU: the algorithmic byte and FLOP
counts the reported rates divide by, the clock-record parsing that decides
whether a run is throttled, and the config both arms print."""
import numpy as np

import bench
from synth import make_step


def test_decode_bytes_by_hand():
    # two sequences of 17 and 32 tokens, 4 query / 2 KV heads, head_dim 64,
    # 16-bit: K+V once per KV head per token, Q in and O out, table entries
    # (2 + 2 blocks) and the two context lengths
    got = bench.decode_bytes([17, 32], Hq=4, Hkv=2, d=64)
    kv = (17 + 32) * 2 * 2 * 64 * 2
    qo = 2 * 4 * 64 * 2 * 2
    assert got == kv + qo + 4 * 4 + 4 * 2


def test_prefill_flops_by_hand():
    # a chunk of 3 queries behind 2 prior tokens attends 3, 4 and 5 keys;
    # each (query head, key) costs 2d for Q.K^T and 2d for P.V
    Hq, d = 2, 8
    assert bench.prefill_flops([5], [3], Hq, d) == 4 * Hq * d * (3 + 4 + 5)
    # no prior context: 1 + 2 + ... + q keys
    assert bench.prefill_flops([4], [4], 1, 1) == 4 * (1 + 2 + 3 + 4)


def test_clock_summary_flags_throttle_reasons():
    c = bench.ClockSampler(0)
    c.lines = ["2070, 2070, Not Active, Not Active, Not Active, Not Active",
               "1980, 2070, Not Active, Not Active, Not Active, Active",
               "garbage line",
               "2070, 2070, Active, Not Active, Not Active, Not Active"]
    s = c.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    empty = bench.ClockSampler(0)
    assert empty.summary()["reasons"] == ["unsampled"]


def test_traffic_is_reported_only_for_the_captured_source(monkeypatch):
    assert bench.decode_traffic(True) in (None, bench.DECODE_TRAFFIC_BYTES)
    assert bench.decode_traffic(False) is None          # another workload: never the captured bytes
    monkeypatch.setattr(bench, "DECODE_TRAFFIC_SHA1", "0" * 40)
    assert bench.decode_traffic(True) is None


def test_step_config_describes_the_workload():
    st = make_step("tiny")
    cfg = bench.step_config(st, 1)
    assert cfg["workload"] == bench.WORKLOAD and cfg["seqs_per_gpu"] == st.S
    assert cfg["q_heads"] == st.Hq and cfg["kv_heads"] == st.Hkv and cfg["head_dim"] == st.d
    assert cfg["parallelism"] == "dp1"
    assert abs(cfg["mean_context"] - float(np.mean(st.context_lens))) < 0.1
