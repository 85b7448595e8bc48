"""The benchmark's host-side pieces that need no GPU: every mode it accepts has
an oracle it is timed against for its `cpu_baseline` (also a run whose modes
are all consumers or allocation-free calls), the roofline rules, and the
launch counts it claims per call."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synthetic  # noqa: E402


@pytest.mark.parametrize("mode", sorted(bench.MODE_IDS))
def test_every_mode_has_a_timed_oracle(mode):
    w = synthetic.gaussian(32, 256, 0.02, 5)
    gbs, seconds, reps, rows = bench.oracle_time_mode(w, mode, 1, 0.01, batch=4)
    assert gbs > 0 and seconds >= 0.01 and reps >= 1 and 16 <= rows <= 32


def test_cpu_baseline_without_hot_path_modes():
    w = synthetic.gaussian(32, 256, 0.02, 6)
    step, per = bench.oracle_cpu_baseline(w, ["gemv", "swizzle", "max_noalloc"], 0, 0.01, batch=2)
    assert step["value"] > 0 and step["kind"] == "oracle" and set(per) == {"gemv", "swizzle", "max_noalloc"}
    assert "max oracle" in per["max_noalloc"]["sample"]


def test_rules_and_launch_counts():
    n, l2 = 1 << 24, 128 << 20
    # one HBM read of W when it fits in half of L2, else two
    assert bench.algorithmic(0, 5, 1 << 20, l2)[2] == bench.ONE_PASS * (1 << 20)
    assert bench.algorithmic(1, 5, n * 4, l2)[2] == bench.TWO_PASS * n * 4
    # CJSO(T): T + 2 reads of W plus the outputs; decoupled: 505 flop per element
    assert bench.algorithmic(2, 5, n * 4, l2)[2] == (7 * 2 + 0.5625) * n * 4
    assert bench.algorithmic(3, 5, n, l2)[0] == "alu"
    assert bench.algorithmic(3, 5, n, l2)[2] == 505 * n
    # kernels per call: amax + quantize; amax + T + 1 sweeps (+ search and deferred-block kernel)
    assert [bench.kernels_per_call(m, 5) for m in range(5)] == [2, 2, 7, 9, 1]
