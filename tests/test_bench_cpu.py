"""Host logic of bench.py that needs no GPU: the percentile helper and the
per-workload oracle baselines of the configs block."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_percentile_nearest_rank():
    vals = sorted([5.0, 1.0, 3.0, 2.0, 4.0])
    assert bench._pct(vals, 50) == 3.0
    assert bench._pct(vals, 95) == 5.0
    assert bench._pct(vals, 0) == 1.0
    assert bench._pct([7.0], 95) == 7.0


def test_oracle_rate_decode_covers_every_sequence():
    """The tiny decode: every sequence is sampled, the rate is in the decode
    unit, and one thread is reported as one core."""
    p = W.config(1)
    r = bench.oracle_config_rate(p, 0.05)
    assert r["unit"] == "GB/s" and r["kind"] == "oracle" and r["value"] > 0
    assert r["sample"].startswith(f"fp64 oracle on {p.num_seqs} of {p.num_seqs} requests")
    one = bench.oracle_config_rate(p, 0.05, threads=1)
    assert one["cores"] == 1 and one["value"] > 0


def test_oracle_rate_prefill_takes_at_least_one_request():
    """A budget smaller than one request still times one whole request, in
    TFLOP/s of the visible causal pairs."""
    r = bench.oracle_config_rate(W.config(3), 1e-6)
    assert r["unit"] == "TFLOP/s" and r["value"] > 0
    assert "1 request calls (512 query tokens)" in r["sample"]


@pytest.mark.parametrize("name", sorted(bench.CONFIG_CPU_CASES))
def test_config_cpu_cases_name_configs_block_entries(name):
    """Every CPU-baseline entry lands beside a configs-block entry of the
    same name."""
    assert name in bench.CONFIG_CASES
