"""Host-side pieces of bench.py that need no GPU: the per-chunk step statistics and the
bounded CPU-oracle samples (all threads and one thread)."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import bench  # noqa: E402
import workloads as WL  # noqa: E402


def test_step_stats_percentiles():
    # 11 chunks of 100 steps: 1..11 ms per chunk -> 10..110 us per step
    secs = [i * 1e-3 for i in range(1, 12)]
    st = bench.step_stats(secs, [100] * 11)
    assert st["chunks"] == 11
    assert abs(st["median"] - 60.0) < 1e-9
    assert abs(st["p10"] - 20.0) < 1e-9
    assert abs(st["p90"] - 100.0) < 1e-9
    # a short last chunk counts per step
    st = bench.step_stats([1e-3, 0.5e-3], [100, 50])
    assert abs(st["median"] - 10.0) < 1e-9 and st["chunks"] == 2
    assert bench.step_stats([], []) is None


def test_cpu_oracle_rate_all_and_one_thread():
    mats = WL.make_random_layer(128, 64, seed=7)
    X = WL.make_random_tokens(2, 128, seed=8)
    rate, n, dt, threads = bench.cpu_oracle_rate(mats, X, 0.5, 0.5, 0.05)
    assert n >= 1 and dt >= 0.05 and rate > 0 and threads >= 1
    rate1, n1, dt1, threads1 = bench.cpu_oracle_rate(mats, X, 0.5, 0.5, 0.05, threads=1)
    assert n1 >= 1 and rate1 > 0 and threads1 == 1
