"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Inputs come from the seeded generators in memory_bound_row_rmsnorm_gb300.synthetic,
are copied to the GPU, and the same bytes (widened exactly to float64) go to
the oracle.  Outputs are pre-filled with NaN so an element the kernels never
write fails the comparison.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
from parity import check_rows, check_scalars, loss_denominator, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EPS = 1e-6
OPS = ("softmax", "rmsnorm", "xent")
DTYPES = ("f32", "bf16")
OP_CODE = {"softmax": qb.QK_OP_SOFTMAX, "rmsnorm": qb.QK_OP_RMSNORM, "xent": qb.QK_OP_XENT}
DT_CODE = {"f32": qb.QK_F32, "bf16": qb.QK_BF16}


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    qb.load_library()
    torch.cuda.set_device(0)
    yield
    for op in OP_CODE.values():
        for dt in DT_CODE.values():
            qb.qk_set_plan_override(op, dt, None)


def nan_like(t, dtype=None):
    return torch.full_like(t, float("nan"), dtype=dtype)


def run_gpu(op, inp, dtype, eps=EPS, y=None):
    """One call through the C ABI on device tensors; returns the outputs."""
    x = inp["x"]
    M, N = x.shape
    code = DT_CODE[dtype]
    if op == "softmax":
        y = nan_like(x) if y is None else y
        qb.qk_softmax_fwd(x, y, M, N, code)
        out = {"y": y}
    elif op == "rmsnorm":
        y = nan_like(x) if y is None else y
        rstd = torch.full((M,), float("nan"), dtype=torch.float32, device=x.device)
        qb.qk_rmsnorm_fwd(x, inp["w"], y, rstd, M, N, eps, code)
        out = {"y": y, "rstd": rstd}
    else:
        loss = torch.full((M,), float("nan"), dtype=torch.float32, device=x.device)
        lse = torch.full((M,), float("nan"), dtype=torch.float32, device=x.device)
        qb.qk_xent_fwd(x, inp["targets"], loss, lse, M, N, code)
        out = {"loss": loss, "lse": lse}
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    return out


def check_against_oracle(op, dtype, inp_cpu, out, rows=None, eps=EPS, what=""):
    """Compare `out` (device tensors) with the oracle on `rows` (all if None)."""
    sel = slice(None) if rows is None else rows
    x64 = to_f64(inp_cpu["x"][sel])
    if op == "softmax":
        ref = oracle.softmax_fwd(x64)
        check_rows(to_f64(out["y"][sel]), ref, dtype, True, f"softmax {what}")
    elif op == "rmsnorm":
        ref_y, ref_r = oracle.rmsnorm_fwd(x64, to_f64(inp_cpu["w"]), eps)
        check_rows(to_f64(out["y"][sel]), ref_y, dtype, False, f"rmsnorm y {what}")
        check_scalars(to_f64(out["rstd"][sel]), ref_r, f"rmsnorm rstd {what}")
    else:
        t = inp_cpu["targets"][sel].numpy()
        ref_loss, ref_lse = oracle.xent_fwd(x64, t)
        check_scalars(to_f64(out["lse"][sel]), ref_lse, f"xent lse {what}")
        check_scalars(to_f64(out["loss"][sel]), ref_loss, f"xent loss {what}",
                      denom=loss_denominator(ref_loss, ref_lse))


def full_check(op, dtype, M, N, seed, sigma=1.0, what=""):
    inp = syn.make_inputs(op, dtype, M, N, seed, "cpu", sigma)
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = run_gpu(op, dev, dtype)
    check_against_oracle(op, dtype, inp, out, what=what or f"{dtype} {M}x{N}")
    return inp, out


def _rows_for(N):
    """Row counts: ragged against every rows-per-CTA choice, bounded work."""
    return max(3, min(37, (1 << 22) // N)) if N <= 65536 else 3


SMALL_N = [1, 2, 3, 8, 31, 64, 100, 256, 257, 1000, 1024, 2048, 4096, 4097, 8192, 16384,
           20000, 32768]


@pytest.mark.parametrize("N", SMALL_N)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
def test_shapes(op, dtype, N):
    full_check(op, dtype, _rows_for(N), N, seed=100 + N)


@pytest.mark.parametrize("N", [65536, 131072, 262144, 524288, 262148, 300001, 1048576])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
def test_long_rows(op, dtype, N):
    """Clustered rows up to 1 MiB, streamed-twice rows beyond it, masked long rows."""
    full_check(op, dtype, 3, N, seed=200 + N)


@pytest.mark.parametrize("M", [1, 5, 400])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm"])
def test_rows_beyond_a_cluster(op, M):
    """Rows beyond 1 MiB take two passes: split over a cluster when there are
    few rows, one CTA per row when there are many."""
    N = 3 * 2 ** 19 if M <= 5 else 2 ** 18 + 4096
    got = qb.qk_get_plan(OP_CODE[op], qb.QK_F32, M, N)
    assert got["path"] == 4
    inp = syn.make_inputs(op, "f32", M, N, 250 + M, "cpu")
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = run_gpu(op, dev, "f32")
    rows = None if M <= 5 else torch.tensor([0, 1, 199, 398, 399])
    check_against_oracle(op, "f32", inp, out, rows=rows, what=f"two-pass {M}x{N}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", ["softmax", "rmsnorm"])
def test_unaligned_rows_beyond_limit_are_refused(op, dtype):
    """The masked path (unaligned rows) holds rows of up to 524,288 elements."""
    N = 524288 + 3
    x = torch.empty((1, N), dtype=syn.DTYPES[dtype], device=DEV)
    with pytest.raises(qb.QkError) as e:
        if op == "softmax":
            qb.qk_softmax_fwd(x, x, 1, N, DT_CODE[dtype])
        else:
            w = torch.empty(N, dtype=syn.DTYPES[dtype], device=DEV)
            qb.qk_rmsnorm_fwd(x, w, x, None, 1, N, 1e-6, DT_CODE[dtype])
    assert e.value.status == qb.QK_ERR_UNSUPPORTED


# Forced two-pass plans on moderate rows: several chunks per slice, ring reuse,
# clusters splitting the row, ragged last chunk and a short last slice.
TWO_PASS_PLANS = [
    dict(path=4, threads=256, row_threads=256, vec_per_thread=8, cluster=1, slots=2, grid=3),
    dict(path=4, threads=256, row_threads=256, vec_per_thread=8, cluster=1, slots=3, grid=16),
    dict(path=4, threads=256, row_threads=256, vec_per_thread=8, cluster=4, slots=2, grid=8),
    dict(path=4, threads=256, row_threads=256, vec_per_thread=8, cluster=16, slots=3, grid=16),
]


@pytest.mark.parametrize("pi", range(len(TWO_PASS_PLANS)))
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", ["softmax", "rmsnorm"])
def test_forced_two_pass(op, dtype, pi):
    plan = TWO_PASS_PLANS[pi]
    E = 4 if dtype == "f32" else 8
    N = (5 * 2048 * plan["cluster"] + 37) * E  # about 5 chunks per slice, ragged
    M = 7
    qb.qk_set_plan_override(OP_CODE[op], DT_CODE[dtype], plan)
    try:
        got = qb.qk_get_plan(OP_CODE[op], DT_CODE[dtype], M, N)
        assert got["path"] == 4 and got["cluster"] == plan["cluster"] and got["chunks"] >= 5
        full_check(op, dtype, M, N, seed=260 + pi, what=f"two-pass plan {plan}")
    finally:
        qb.qk_set_plan_override(OP_CODE[op], DT_CODE[dtype], None)


# Forced plans: tiny grids make every CTA walk many items, so each ring slot is
# reused many times (both barrier parities) and the last item is ragged.
PLANS = [
    dict(threads=256, row_threads=32, vec_per_thread=1, cluster=1, slots=2, grid=3),
    dict(threads=256, row_threads=32, vec_per_thread=4, cluster=1, slots=3, grid=5),
    dict(threads=256, row_threads=64, vec_per_thread=4, cluster=1, slots=2, grid=2),
    dict(threads=128, row_threads=128, vec_per_thread=4, cluster=1, slots=4, grid=7),
    dict(threads=256, row_threads=256, vec_per_thread=8, cluster=1, slots=2, grid=1),
    dict(threads=512, row_threads=512, vec_per_thread=4, cluster=1, slots=5, grid=4),
    dict(threads=256, row_threads=256, vec_per_thread=8, cluster=2, slots=2, grid=2),
    dict(threads=512, row_threads=512, vec_per_thread=4, cluster=4, slots=3, grid=8),
    dict(threads=512, row_threads=512, vec_per_thread=8, cluster=8, slots=2, grid=8),
    dict(threads=512, row_threads=512, vec_per_thread=8, cluster=16, slots=2, grid=16),
    dict(threads=256, row_threads=8, vec_per_thread=4, cluster=1, slots=2, grid=3),
    dict(threads=256, row_threads=16, vec_per_thread=8, cluster=1, slots=1, grid=2),
    dict(threads=256, row_threads=32, vec_per_thread=16, cluster=1, slots=2, grid=2),
    dict(threads=256, row_threads=64, vec_per_thread=8, cluster=1, slots=1, grid=5),
    dict(threads=256, row_threads=256, vec_per_thread=16, cluster=4, slots=1, grid=8),
    dict(threads=256, row_threads=256, vec_per_thread=4, cluster=16, slots=3, grid=32),
]


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: "t{threads}r{row_threads}v{vec_per_thread}c{cluster}s{slots}g{grid}".format(**p))
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
def test_forced_plans(op, dtype, plan):
    if op == "xent" and plan["cluster"] > 1:
        pytest.skip("cross-entropy has no clustered kernel")
    E = 4 if dtype == "f32" else 8
    cap = plan["row_threads"] * plan["vec_per_thread"] * E * plan["cluster"]
    # a row that fills most of the plan's capacity and is ragged in vectors
    N = max(E, cap - 3 * E) if cap > 4 * E else cap
    rows_per_step = plan["threads"] // plan["row_threads"]
    # several steps per CTA, and a last step that is only partly filled
    M = max(61, 3 * rows_per_step * plan["grid"] + 5) if N <= 8192 else 9
    if op == "xent" and plan["row_threads"] == plan["threads"]:
        N = 5 * cap + 7 * E  # streamed through several chunks per row
    qb.qk_set_plan_override(OP_CODE[op], DT_CODE[dtype], plan)
    try:
        got = qb.qk_get_plan(OP_CODE[op], DT_CODE[dtype], M, N)
        assert got["threads"] == plan["threads"] and got["cluster"] == plan["cluster"]
        assert got["grid"] == plan["grid"]
        full_check(op, dtype, M, N, seed=300 + N, what=f"plan {plan}")
    finally:
        qb.qk_set_plan_override(OP_CODE[op], DT_CODE[dtype], None)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", ["softmax", "rmsnorm"])
@pytest.mark.parametrize("N", [4096, 131072])
def test_in_place(op, dtype, N):
    M = 17 if N == 4096 else 3
    inp = syn.make_inputs(op, dtype, M, N, 400, "cpu")
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = run_gpu(op, dev, dtype, y=dev["x"])  # y aliases x exactly
    check_against_oracle(op, dtype, inp, out, what="in place")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("N", [64, 4096, 40000])
def test_unaligned_pointers(op, dtype, N):
    """Inputs that start one element past a 16-byte boundary take the masked path."""
    M = 5
    inp = syn.make_inputs(op, dtype, M, N, 500 + N, "cpu")
    x_store = torch.empty(M * N + 1, dtype=syn.DTYPES[dtype], device=DEV)
    x = x_store[1:].view(M, N)
    x.copy_(inp["x"])
    dev = dict({k: v.to(DEV) for k, v in inp.items()}, x=x)
    y_store = torch.full((M * N + 1,), float("nan"), dtype=syn.DTYPES[dtype], device=DEV)
    out = run_gpu(op, dev, dtype, y=y_store[1:].view(M, N) if op != "xent" else None)
    check_against_oracle(op, dtype, inp, out, what="unaligned")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N", [7, 4096, 131072])
def test_softmax_extreme_rows(dtype, N):
    M = 4
    x = syn.normal_rows(M, N, dtype, 600, "cpu", sigma=100.0)
    x[1] = 3.25                        # constant row -> exactly 1/N
    x[2, :] = -1e4
    x[2, N // 2] = 50.0                # one dominant entry
    inp = {"x": x}
    out = run_gpu("softmax", {"x": x.to(DEV)}, dtype)
    check_against_oracle("softmax", dtype, inp, out, what="extreme rows")
    y1 = to_f64(out["y"][1])
    assert np.all(np.abs(y1 - 1.0 / N) <= (1e-5 if dtype == "f32" else 2 ** -7) / N)


@pytest.mark.parametrize("dtype", DTYPES)
def test_rmsnorm_zero_and_constant_rows(dtype):
    M, N = 3, 4096
    x = torch.zeros((M, N), dtype=syn.DTYPES[dtype])
    x[1] = -0.75
    x[2] = syn.normal_rows(1, N, dtype, 700, "cpu")[0] * 1e3
    inp = {"x": x, "w": syn.uniform_weight(N, dtype, 701, "cpu")}
    out = run_gpu("rmsnorm", {k: v.to(DEV) for k, v in inp.items()}, dtype)
    check_against_oracle("rmsnorm", dtype, inp, out, what="zero/constant rows")
    assert torch.all(out["y"][0] == 0)
    assert abs(out["rstd"][0].item() - EPS ** -0.5) <= 1e-5 * EPS ** -0.5


INT64_MIN, INT64_MAX = -(2 ** 63), 2 ** 63 - 1


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N", [10, 4096, 131072])
def test_xent_targets_out_of_range(dtype, N):
    """Every target outside [0, N) gives NaN, the extreme int64 values too
    (no target value stands for "no ignore index").  N = 10 takes the
    shifted kernel, 4096 the ring, 131072 the streamed ring."""
    M = 8
    inp = syn.make_inputs("xent", dtype, M, N, 800, "cpu")
    inp["targets"] = torch.tensor([-1, N, 0, N - 1, 2 ** 40, -(2 ** 40), INT64_MIN, INT64_MAX],
                                  dtype=torch.int64)
    out = run_gpu("xent", {k: v.to(DEV) for k, v in inp.items()}, dtype)
    check_against_oracle("xent", dtype, inp, out, what="targets out of range")
    loss = out["loss"].cpu()
    assert torch.isnan(loss[[0, 1, 4, 5, 6, 7]]).all() and torch.isfinite(loss[[2, 3]]).all()
    assert torch.isfinite(out["lse"]).all()


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N", [10, 4096, 131072, 4101])
def test_xent_extreme_targets_through_the_variants(dtype, N):
    """qk_xent_fwd_ex without an ignore index treats INT64_MIN / INT64_MAX
    as out of range (NaN); with INT64_MIN as the ignore index that row is
    ignored (loss 0, left out of the mean) and INT64_MAX is still NaN."""
    M = 8
    inp = syn.make_inputs("xent", dtype, M, N, 810, "cpu")
    t = torch.tensor([INT64_MIN, 3, INT64_MAX, 0, N - 1, 1, INT64_MIN, 2], dtype=torch.int64)
    inp["targets"] = t
    d = {k: v.to(DEV) for k, v in inp.items()}
    x64 = to_f64(inp["x"])
    for ignore in (None, INT64_MIN):
        loss = torch.full((M,), float("nan"), dtype=torch.float32, device=DEV)
        lse = torch.full((M,), float("nan"), dtype=torch.float32, device=DEV)
        qb.qk_xent_fwd_ex(d["x"], d["targets"], loss, lse, None, M, N, DT_CODE[dtype], ignore_index=ignore)
        torch.cuda.synchronize()
        ref_loss, ref_lse, _ = oracle.xent_fwd_ex(x64, t.numpy(), ignore_index=ignore)
        check_scalars(to_f64(lse), ref_lse, f"xent ex lse, ignore {ignore}")
        check_scalars(to_f64(loss), ref_loss, f"xent ex loss, ignore {ignore}",
                      denom=loss_denominator(ref_loss, ref_lse))
        got = loss.cpu()
        if ignore is None:
            assert torch.isnan(got[[0, 2, 6]]).all()
        else:
            assert (got[[0, 6]] == 0).all() and torch.isnan(got[2])


def test_xent_constant_row_is_log_n():
    for N in (1, 4096, 100000):
        x = torch.full((2, N), -4.25, dtype=torch.float32, device=DEV)
        t = torch.tensor([0, N - 1], dtype=torch.int64, device=DEV)
        out = run_gpu("xent", {"x": x, "targets": t}, "f32")
        assert np.allclose(to_f64(out["loss"]), math.log(N), rtol=1e-5, atol=1e-6)


def test_zero_rows_launch_nothing():
    x = torch.empty((0, 128), dtype=torch.float32, device=DEV)
    qb.qk_softmax_fwd(x, x, 0, 128, qb.QK_F32)
    assert qb.qk_get_device_status() == qb.QK_OK


def test_streams_are_honoured():
    s = torch.cuda.Stream()
    inp = syn.make_inputs("softmax", "f32", 64, 4096, 900, "cpu")
    x = inp["x"].to(DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        y = torch.full_like(x, float("nan"))
        qb.qk_softmax_fwd(x, y, 64, 4096, qb.QK_F32, s)
    s.synchronize()
    check_against_oracle("softmax", "f32", inp, {"y": y}, what="side stream")
