"""The benchmark's CPU-oracle legs on the host: per-op, per-workload timing.

Runs the spawned per-core oracle processes on the tiny workload (2 processes
and 1, one pass) and checks the shape of what the benchmark reports: a GB/s
figure per op for all cores and for one core, the sample described, and the
sample sizing rule (the whole workload when it fits, else a token prefix).
"""
import pytest

import bench
from sequence_head_relayout_gb300 import workloads as W

pytestmark = pytest.mark.usefixtures("oracle_built")


def test_per_config_oracle_timing_tiny():
    r = bench.cpu_per_config(["tiny"], cores=2, passes=1)
    assert r["cores"] == 2 and r["kind"] == "oracle"
    assert r["sample"]["tiny"].startswith("64 of 64 tokens")
    row = r["table"]["tiny"]
    assert set(row) == set(bench.CPU_OPS)
    for op in bench.CPU_OPS:
        assert row[op]["cpu_gbs"] > 0 and row[op]["cpu_gbs_1core"] > 0


def test_sample_tokens_rule():
    tiny, large = W.CONFIGS["tiny"], W.CONFIGS["large"]
    assert bench.cpu_sample_tokens(tiny) == tiny.T
    n = bench.cpu_sample_tokens(large)
    assert 0 < n < large.T
    H, D, Hp = large.H, large.D, large.H // large.P
    per_token = 2 * (6 * H * D + 4 * H * D + 6 * Hp * D)
    assert n * per_token <= bench.CPU_SAMPLE_BYTES < (n + 1) * per_token
