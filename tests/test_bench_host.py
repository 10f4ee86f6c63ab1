"""bench.py's host-side arithmetic, without a GPU: the algorithmic bytes of
every operator, the whole-job rate, the nvidia-smi clock summary, and the rule
that a recorded DRAM traffic figure is reported only for the sources and plan
it was taken on."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("dtype,s", [("f32", 4), ("bf16", 2)])
def test_min_bytes(dtype, s):
    M, N = 37, 4104
    want = {
        "softmax": 2 * M * N * s,                              # x in, y out
        "rmsnorm": 2 * M * N * s + N * s + 4 * M,              # x, w in; y, rstd out
        "xent": M * N * s + 8 * M + 4 * M + 4 * M,             # logits, targets in; loss, lse out
        "layernorm": 2 * M * N * s + 2 * N * s + 4 * M + 4 * M,  # x, w, b in; y, mean, rstd out
        "softmax_bwd": 3 * M * N * s,                          # y, dy in; dx out
        "rmsnorm_bwd": 3 * M * N * s + N * s + 4 * M + 4 * N,  # x, dy, w, rstd in; dx, dw out
        "xent_bwd": 2 * M * N * s + 8 * M + 4 * M + 4 * M,     # logits, targets, lse, dloss in; dx out
    }
    for op, b in want.items():
        assert bench.min_bytes(op, dtype, M, N) == b, op
    with pytest.raises(ValueError):
        bench.min_bytes("nothing", dtype, M, N)


def test_whole_job_rate():
    # 2 ranks x 10 steps x 1e9 bytes in 4 ms: 5 TB/s
    assert bench.whole_job_tbs(10 ** 9, 2, 10, 4.0) == pytest.approx(5.0)


def test_clock_summary():
    cs = bench.ClockSampler(0)
    cs.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1900, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    s = cs.summary()
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    cs.lines = []
    assert cs.summary()["samples"] == 0


@pytest.mark.parametrize("workload", sorted(f[:-len(".traffic.json")] for f in os.listdir(os.path.join(ROOT, "profiles"))
                                            if f.endswith(".traffic.json")))
def test_recorded_traffic_follows_sources_and_plan(workload):
    rec = json.load(open(os.path.join(ROOT, "profiles", f"{workload}.traffic.json")))
    plan = dict(rec["plan"])
    assert rec["dram_bytes_per_launch"] > 0 and rec["algorithmic_bytes_per_launch"] > 0
    got = bench.recorded_traffic(workload, plan)
    if rec["kernel_source_hash"] == bench.kernel_source_hash():
        assert got == rec["dram_bytes_per_launch"]
    else:
        assert got is None  # taken on other sources: not reported
    other = dict(plan, slots=plan["slots"] + 1)
    assert bench.recorded_traffic(workload, other) is None  # another plan: not reported
    assert bench.recorded_traffic("no_such_workload", plan) is None


def test_peaks():
    peak, source = bench.measured_peak()
    assert peak > 1000 and isinstance(source, str)
    assert bench.NOMINAL_HBM_GBS == 7900.0
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
