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


def test_clock_windows_by_timestamp():
    """Samples carry nvidia-smi's timestamp; a window keeps only its own."""
    import datetime
    cs = bench.ClockSampler(0)
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)
    def line(dt_s, mhz, cap="Not Active"):
        ts = (base + datetime.timedelta(seconds=dt_s)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, 0, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    cs.lines = [line(0.0, 1500), line(0.1, 2070), line(0.2, 2070, "Active"), line(0.3, 1000)]
    t = base.timestamp()
    w = cs.summary(t + 0.05, t + 0.25)
    assert w["samples"] == 2 and w["sm_mhz"] == 2070 and w["reasons"] == ["sw_power_cap"]
    assert cs.summary()["samples"] == 4
    assert cs.summary(t + 5, t + 6)["samples"] == 0


def test_rotating_sets_and_kernel_counts():
    L2 = bench.L2_BYTES
    assert bench.n_sets(4 * L2) == 1 and bench.n_sets(10 * L2) == 1
    assert bench.n_sets(L2) == 4 and bench.n_sets(4 * L2 - 1) == 2
    for b in (1, 10 ** 6, L2 // 3, 2 * L2):  # together they pass 4x L2
        assert bench.n_sets(b) * b >= 4 * L2
    assert bench.kernels_per_step("rmsnorm_bwd") == 2
    assert all(bench.kernels_per_step(op) == 1 for op in ("softmax", "rmsnorm", "xent", "layernorm"))


def test_sweep_summary():
    cs = bench.ClockSampler(0)
    pts = []
    for N, f in ((1024, 0.4), (4096, 0.9), (16384, 0.8), (65536, 0.95)):
        pts.append({"op": "softmax", "dtype": "f32", "M": 8192, "N": N, "frac": f, "frac_stream": f - 0.1,
                    "TBps": f * 6.8, "clocks": {"sm_mhz": 2070}})
    s = bench.sweep_summary(pts, (0.0, 1.0), cs)
    k = s["per_kernel"]["softmax_f32"]
    assert k["points"] == 4 and k["points_N_ge_4096"] == 3
    assert k["min_frac_N_ge_4096"] == 0.8 and k["worst"]["N"] == 16384
    assert k["median_frac_N_ge_4096"] == 0.9
    assert s["points_N_ge_4096_at_or_above_0.85"] == 2 and s["points_N_ge_4096"] == 3
    assert len(s["points"]) == 4 and s["points"][0][:4] == ["softmax", "f32", 8192, 1024]
