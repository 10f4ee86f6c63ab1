"""LayerNorm forward: CUDA path against the fp64 oracle, through the C ABI.

Tolerances (derived from the fp32 arithmetic, fixed before the kernel ran):
  * y: |got - ref| <= 1e-5 * ((|x| + |mean|) * rstd * |w| + |b|), plus one
    bf16 ulp of the value for bf16 outputs.  x - mean rounds relative to the
    larger of |x| and |mean| (the two can cancel), and the rest is a product
    and one fused add, so the error is bounded by the magnitude of the terms.
  * mean: |got - ref| <= 1e-5 * (1/N) sum_j |x_j| (a rounded sum of N terms).
  * rstd: relative error <= 1e-5 * (1 + |mean| * rstd); the squared
    deviations are formed from x - mean, which rounds relative to |mean| too.
NaN-prefilled outputs catch any element the kernels do not write.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
from parity import check_scaled, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EPS = 1e-5
DTYPES = ("f32", "bf16")
DT_CODE = {"f32": qb.QK_F32, "bf16": qb.QK_BF16}
OP = qb.QK_OP_LAYERNORM


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    qb.load_library()
    torch.cuda.set_device(0)
    yield
    for dt in DT_CODE.values():
        qb.qk_set_plan_override(OP, dt, None)


def run_gpu(inp, dtype, eps=EPS, bias=True, stats=True, y=None):
    x = inp["x"]
    M, N = x.shape
    y = torch.full_like(x, float("nan")) if y is None else y
    mean = rstd = None
    if stats:
        mean = torch.full((M,), float("nan"), dtype=torch.float32, device=x.device)
        rstd = torch.full((M,), float("nan"), dtype=torch.float32, device=x.device)
    qb.qk_layernorm_fwd(x, inp["w"], inp["b"] if bias else None, y, mean, rstd, M, N, eps,
                        DT_CODE[dtype])
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    return {"y": y, "mean": mean, "rstd": rstd}


def check(inp_cpu, out, dtype, eps=EPS, bias=True, rows=None, what=""):
    sel = slice(None) if rows is None else rows
    x = to_f64(inp_cpu["x"][sel])
    w = to_f64(inp_cpu["w"])
    b = to_f64(inp_cpu["b"]) if bias else None
    ref_y, ref_m, ref_r = oracle.layernorm_fwd(x, w, b, eps)
    scale = ((np.abs(x) + np.abs(ref_m)[:, None]) * ref_r[:, None] * np.abs(w)[None, :]
             + (np.abs(b)[None, :] if bias else 0.0))
    check_scaled(to_f64(out["y"][sel]), ref_y, scale, dtype, f"layernorm y {what}")
    if out["mean"] is not None:
        check_scaled(to_f64(out["mean"][sel]), ref_m, np.abs(x).mean(axis=1), "f32",
                     f"layernorm mean {what}")
        check_scaled(to_f64(out["rstd"][sel]), ref_r, ref_r * (1 + np.abs(ref_m) * ref_r), "f32",
                     f"layernorm rstd {what}")


def full_check(dtype, M, N, seed, what="", **kw):
    inp = syn.make_inputs("layernorm", dtype, M, N, seed, "cpu")
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = run_gpu(dev, dtype, **kw)
    check(inp, out, dtype, bias=kw.get("bias", True), what=what or f"{dtype} {M}x{N}")
    return inp, out


def _rows_for(N):
    return max(3, min(37, (1 << 22) // N)) if N <= 65536 else 3


SMALL_N = [1, 2, 3, 8, 31, 64, 100, 256, 257, 1000, 1024, 2048, 4096, 4097, 8192, 16384,
           20000, 32768]


@pytest.mark.parametrize("N", SMALL_N)
@pytest.mark.parametrize("dtype", DTYPES)
def test_shapes(dtype, N):
    full_check(dtype, _rows_for(N), N, seed=1100 + N)


@pytest.mark.parametrize("stats", [True, False])
@pytest.mark.parametrize("bias", [True, False])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N", [24, 4096, 131072 + 8, 5000])
def test_optional_bias_and_stats(dtype, N, bias, stats):
    """No bias means b = 0; the statistics may be left out (NULL)."""
    full_check(dtype, 5, N, seed=1200 + N, bias=bias, stats=stats)


@pytest.mark.parametrize("N", [65536, 131072, 262144, 524288, 262148, 300001])
@pytest.mark.parametrize("dtype", DTYPES)
def test_long_rows(dtype, N):
    """Clustered rows up to 1 MiB, rows beyond it streamed twice, unaligned long
    rows on the shifted or the masked kernel."""
    if N > qb.qk_max_row_elements(OP, DT_CODE[dtype]):
        x = torch.empty((1, N), dtype=syn.DTYPES[dtype], device=DEV)
        w = torch.empty(N, dtype=syn.DTYPES[dtype], device=DEV)
        with pytest.raises(qb.QkError) as e:
            qb.qk_layernorm_fwd(x, w, None, x, None, None, 1, N, EPS, DT_CODE[dtype])
        assert e.value.status == qb.QK_ERR_UNSUPPORTED
        return
    full_check(dtype, 3, N, seed=1300 + N)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N", [64, 4096, 40000])
def test_unaligned_pointers(dtype, N):
    """x and y one element past a 16-byte boundary take the masked path."""
    M = 5
    inp = syn.make_inputs("layernorm", dtype, M, N, 1400 + N, "cpu")
    t = syn.DTYPES[dtype]
    xs = torch.empty(M * N + 1, dtype=t, device=DEV)
    x = xs[1:].view(M, N)
    x.copy_(inp["x"])
    ys = torch.full((M * N + 1,), float("nan"), dtype=t, device=DEV)
    dev = {"x": x, "w": inp["w"].to(DEV), "b": inp["b"].to(DEV)}
    out = run_gpu(dev, dtype, y=ys[1:].view(M, N))
    check(inp, out, dtype, what="unaligned")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N", [4096, 131072])
def test_in_place(dtype, N):
    M = 17 if N == 4096 else 3
    inp = syn.make_inputs("layernorm", dtype, M, N, 1500, "cpu")
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = run_gpu(dev, dtype, y=dev["x"])
    check(inp, out, dtype, what="in place")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N", [4096, 4100, 65536])
def test_degenerate_rows(dtype, N):
    """A constant row has variance 0: y = b and rstd = eps^-1/2 (its mean is
    exactly the constant when the constant is a power of two); a row with a
    large offset (mean 1000 times its deviation) checks the pairwise merge."""
    M = 4
    t = syn.DTYPES[dtype]
    x = syn.offset_rows(M, N, dtype, 1600, "cpu")
    x[0] = 0.0
    x[1] = -0.25
    x[2] = syn.normal_rows(1, N, dtype, 1601, "cpu")[0] * 1e-3 + 1.0
    inp = {"x": x, "w": syn.uniform_weight(N, dtype, 1602, "cpu"),
           "b": syn.uniform_weight(N, dtype, 1603, "cpu", lo=-0.5, hi=0.5)}
    out = run_gpu({k: v.to(DEV) for k, v in inp.items()}, dtype)
    check(inp, out, dtype, what="degenerate rows")
    for r, c in ((0, 0.0), (1, -0.25)):
        assert out["mean"][r].item() == c
        assert torch.equal(out["y"][r].cpu(), inp["b"].to(t))
        assert abs(out["rstd"][r].item() - EPS ** -0.5) <= 1e-6 * EPS ** -0.5


PLANS = [
    dict(threads=256, row_threads=32, vec_per_thread=1, cluster=1, slots=2, grid=3),
    dict(threads=256, row_threads=64, vec_per_thread=4, cluster=1, slots=2, grid=2),
    dict(threads=128, row_threads=128, vec_per_thread=4, cluster=1, slots=4, grid=7),
    dict(threads=256, row_threads=256, vec_per_thread=8, cluster=1, slots=2, grid=1),
    dict(threads=512, row_threads=512, vec_per_thread=4, cluster=1, slots=5, grid=4),
    dict(threads=256, row_threads=256, vec_per_thread=8, cluster=2, slots=2, grid=2),
    dict(threads=512, row_threads=512, vec_per_thread=4, cluster=4, slots=3, grid=8),
    dict(threads=512, row_threads=512, vec_per_thread=8, cluster=16, slots=2, grid=16),
    dict(threads=256, row_threads=8, vec_per_thread=4, cluster=1, slots=2, grid=3),
    dict(threads=256, row_threads=16, vec_per_thread=8, cluster=1, slots=1, grid=2),
    dict(threads=256, row_threads=32, vec_per_thread=16, cluster=1, slots=2, grid=2),
    dict(threads=256, row_threads=256, vec_per_thread=16, cluster=4, slots=1, grid=8),
]


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: "t{threads}r{row_threads}v{vec_per_thread}c{cluster}s{slots}g{grid}".format(**p))
@pytest.mark.parametrize("dtype", DTYPES)
def test_forced_plans(dtype, plan):
    """Tiny grids: every CTA walks many items and reuses each ring slot; the
    rows fill most of the plan and are ragged in vectors, so some warps and
    cluster ranks hold fewer elements than others."""
    E = 4 if dtype == "f32" else 8
    cap = plan["row_threads"] * plan["vec_per_thread"] * E * plan["cluster"]
    N = max(E, cap - 3 * E) if cap > 4 * E else cap
    rows_per_step = plan["threads"] // plan["row_threads"]
    M = max(61, 3 * rows_per_step * plan["grid"] + 5) if N <= 8192 else 9
    qb.qk_set_plan_override(OP, DT_CODE[dtype], plan)
    try:
        got = qb.qk_get_plan(OP, DT_CODE[dtype], M, N)
        assert got["threads"] == plan["threads"] and got["cluster"] == plan["cluster"]
        assert got["grid"] == plan["grid"]
        full_check(dtype, M, N, seed=1700 + N, what=f"plan {plan}")
    finally:
        qb.qk_set_plan_override(OP, DT_CODE[dtype], None)


def test_tensor_helper():
    inp = syn.make_inputs("layernorm", "bf16", 33, 1536, 1800, "cpu")
    dev = {k: v.to(DEV) for k, v in inp.items()}
    y, mean, rstd = qb.layernorm_fwd(dev["x"], dev["w"], dev["b"], eps=EPS)
    torch.cuda.synchronize()
    check(inp, {"y": y, "mean": mean, "rstd": rstd}, "bf16", what="tensor helper")
    y2, m2, r2 = qb.layernorm_fwd(dev["x"], dev["w"], None, eps=EPS, want_stats=False)
    torch.cuda.synchronize()
    assert m2 is None and r2 is None
    check(inp, {"y": y2, "mean": None, "rstd": None}, "bf16", bias=False, what="no bias")


def check_rows(inp, out, dtype, idx, what):
    inp_rows = {"x": inp["x"].index_select(0, idx).cpu(), "w": inp["w"].cpu(), "b": inp["b"].cpu()}
    out_rows = {k: v.index_select(0, idx) for k, v in out.items()}
    check(inp_rows, out_rows, dtype, what=what)


def test_benchmark_workload_every_row():
    """The benchmark's LayerNorm workload at full size (2^26 elements), default
    plan: every row against the oracle, in blocks of rows."""
    M, N = 16384, 4096
    inp = syn.make_inputs("layernorm", "bf16", M, N, 1900, DEV)
    out = run_gpu(inp, "bf16")
    for r0 in range(0, M, 1024):
        check_rows(inp, out, "bf16", torch.arange(r0, r0 + 1024, device=DEV), f"{M}x{N} rows {r0}+")


@pytest.mark.parametrize("dtype", DTYPES)
def test_largest_sweep_shape_sampled_rows(dtype):
    """32768 rows of 262144 (1 MiB fp32 rows on clusters of 16; 2^33 elements):
    256 seeded rows against the oracle, every row's statistics for sanity."""
    M, N = 32768, 262144
    inp = syn.make_inputs("layernorm", dtype, M, N, 1950, DEV)
    out = run_gpu(inp, dtype)
    rng = np.random.default_rng(1950)
    rows = torch.tensor(sorted(set(rng.choice(M, 254, replace=False).tolist()) | {0, M - 1}))
    check_rows(inp, out, dtype, rows.to(DEV), f"{M}x{N} sampled rows")
    for r0 in range(0, M, 1024):
        assert torch.isfinite(out["y"][r0:r0 + 1024]).all()
    assert (out["mean"].abs() <= 1.5).all()            # row offsets are in [-1, 1]
    assert ((out["rstd"] > 0.8) & (out["rstd"] < 1.25)).all()  # unit variance rows
    del inp, out
    torch.cuda.empty_cache()


# Rows longer than a cluster holds stream through shared memory twice; the
# forced plans give several chunks per slice, ring reuse, clusters splitting
# the row, a ragged last chunk and a short last slice.
TWO_PASS_PLANS = [
    dict(path=4, threads=256, row_threads=256, vec_per_thread=8, cluster=1, slots=2, grid=3),
    dict(path=4, threads=256, row_threads=256, vec_per_thread=8, cluster=4, slots=2, grid=8),
    dict(path=4, threads=256, row_threads=256, vec_per_thread=8, cluster=16, slots=3, grid=16),
]


@pytest.mark.parametrize("pi", range(len(TWO_PASS_PLANS)))
@pytest.mark.parametrize("dtype", DTYPES)
def test_forced_two_pass(dtype, pi):
    plan = TWO_PASS_PLANS[pi]
    E = 4 if dtype == "f32" else 8
    N = (5 * 2048 * plan["cluster"] + 37) * E  # about 5 chunks per slice, ragged
    qb.qk_set_plan_override(OP, DT_CODE[dtype], plan)
    try:
        got = qb.qk_get_plan(OP, DT_CODE[dtype], 7, N)
        assert got["path"] == 4 and got["cluster"] == plan["cluster"] and got["chunks"] >= 5
        full_check(dtype, 7, N, seed=2100 + pi, what=f"two-pass plan {plan}")
    finally:
        qb.qk_set_plan_override(OP, DT_CODE[dtype], None)


@pytest.mark.parametrize("M", [1, 5, 400])
def test_rows_beyond_a_cluster(M):
    """Default two-pass plans: split over a cluster when there are few rows,
    one CTA per row when there are many."""
    N = 3 * 2 ** 19 if M <= 5 else 2 ** 18 + 4096
    assert qb.qk_get_plan(OP, qb.QK_F32, M, N)["path"] == 4
    inp = syn.make_inputs("layernorm", "f32", M, N, 2200 + M, "cpu")
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = run_gpu(dev, "f32")
    rows = None if M <= 5 else torch.tensor([0, 1, 199, 398, 399])
    check(inp, out, "f32", rows=rows, what=f"two-pass {M}x{N}")
