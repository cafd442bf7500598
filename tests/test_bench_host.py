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


def test_plan_chunks_replays_exactly_k_steps():
    for K, cyc in ((20, 256), (1, 4), (1000, 256), (1025, 256), (7, 1)):
        plan = bench.plan_chunks(K, cyc)
        assert sum(plan) == K
        assert max(plan) <= 4 * cyc
    assert bench.plan_chunks(0, 10) == []


def test_resolve_workloads():
    a = bench.parse([])
    a.steps = 10
    c = bench.resolve(a)
    assert (c["d"], c["F"], c["batch"], c["sparsity"], c["input_sparsity"]) == \
        (4096, 14336, 1, 0.7, 0.5)
    assert c["layers"] * c["packed_bytes"] >= 3 * bench.L2_BYTES
    c1 = bench.resolve(bench.parse(["--workload", "1"]))
    assert (c1["d"], c1["F"], c1["sparsity"]) == (1024, 2816, 0.5)
    assert c1["layers"] * c1["packed_bytes"] >= 3 * bench.L2_BYTES
    c4 = bench.resolve(bench.parse(["--workload", "4"]))
    assert c4["chain"] and c4["depth"] == 32 and c4["layers"] == 32
    c5 = bench.resolve(bench.parse(["--workload", "5", "--batch", "8", "--sparsity", "0.9"]))
    assert (c5["d"], c5["F"], c5["batch"], c5["sparsity"]) == (8192, 28672, 8, 0.9)


def test_clock_summary():
    text = ("2032, 2032, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
            "1900, 2032, 1090.0, 0x4, Not Active, Not Active, Not Active, Active\n"
            "210, 2032, 90.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    c = bench.summarize_clocks(text)
    assert c["sm_max_mhz"] == 2032 and c["reasons"] == ["sw_power_cap"]
    assert c["sm_mhz"] == 1966.0   # the idle sample is left out of the median


def test_reference_arm_line(capsys):
    """The reference arm times exactly the requested steps and reports the GPU arm's config
    keys for the same workload."""
    import json
    a = bench.parse(["--impl", "reference", "--workload", "1", "--steps", "2", "--warmup", "1",
                     "--tokens", "4"])
    bench.run_reference(a)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    cfg = bench.resolve(a)
    want = bench.workload_config(cfg, 1, 4, 1408, 512)
    assert line["config"] == want
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
