"""Parity at the benchmark workloads' full sizes, in the launch configuration
bench.py times (the library's default plan), and on the M x N sweep grid.

Matrices of at most 2^27 elements (softmax 1024 x 4096, RMSNorm 16384 x 4096)
are compared with the oracle element by element on every row, in blocks of
rows.  Larger ones are compared on 256 seeded rows (always including the
first and the last), and every row is checked against properties that hold
at any size:
  softmax   every entry finite and >= 0, each row sums to 1;
  RMSNorm   rstd finite, 0 < rstd <= eps^-1/2, mean_j (y_ij / w_j)^2 = ms_i/(ms_i+eps) ~ 1;
  x-entropy lse finite and in [max_j x_ij, max_j x_ij + ln N], loss = lse - x_t >= 0.
Outputs start as NaN, so a row the kernels never wrote fails.

The backward workloads bench.py times, and the backward passes at the
sweep's largest shape (2^33 elements), are checked the same way: dx on 256
seeded rows against the oracle (each row of dx depends on its own row only),
every row finite, and RMSNorm's dw, a sum over every row, against the same
sum taken in float64 by PyTorch in blocks of rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import test_backward as tb
from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
from parity import check_scaled, to_f64
from test_parity import DEV, DT_CODE, EPS, check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    qb.load_library()
    torch.cuda.set_device(0)
    yield
    torch.cuda.empty_cache()


WHOLE_MATRIX_ELEMENTS = 1 << 27  # up to this size every row goes to the oracle
SAMPLED_ROWS = 256
ORACLE_BLOCK_ELEMENTS = 1 << 22  # rows handed to the oracle at a time


def sample_rows(M, seed):
    """SAMPLED_ROWS seeded rows, the first and the last among them."""
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(M, size=min(M, SAMPLED_ROWS - 2), replace=False).tolist()) | {0, M - 1}
    extra = iter(rng.permutation(M).tolist())
    while len(rows) < min(M, SAMPLED_ROWS):
        rows.add(next(extra))
    return torch.tensor(sorted(rows), dtype=torch.int64)


def whole_matrix_properties(op, dtype, inp, out, N):
    if op == "softmax":
        y = out["y"]
        assert torch.isfinite(y).all() and (y >= 0).all()
        sums = torch.cat([y[i:i + 1024].double().sum(1) for i in range(0, y.shape[0], 1024)])
        tol = 1e-5 if dtype == "f32" else 2 ** -8
        assert (sums - 1).abs().max().item() <= tol
    elif op == "rmsnorm":
        r = out["rstd"]
        assert torch.isfinite(r).all() and (r > 0).all() and (r <= EPS ** -0.5 * (1 + 1e-6)).all()
        w = inp["w"].double()
        e = torch.cat([((out["y"][i:i + 1024].double() / w) ** 2).mean(1)
                       for i in range(0, out["y"].shape[0], 1024)])
        assert torch.isfinite(e).all() and (e - 1).abs().max().item() <= 2e-2
    else:
        lse, loss = out["lse"], out["loss"]
        assert torch.isfinite(lse).all() and torch.isfinite(loss).all()
        mx = torch.cat([inp["x"][i:i + 1024].float().amax(1) for i in range(0, inp["x"].shape[0], 1024)])
        assert (lse >= mx - 1e-5 * mx.abs()).all()
        assert (lse <= mx + math.log(N) + 1e-5 * (mx.abs() + math.log(N))).all()
        assert (loss >= -1e-6).all()


def check_rows_against_oracle(op, dtype, inp, out, idx, what):
    """The oracle on rows `idx` (a device index tensor) of the inputs."""
    inp_rows = {"x": inp["x"].index_select(0, idx).cpu()}
    if op == "rmsnorm":
        inp_rows["w"] = inp["w"].cpu()
    if op == "xent":
        inp_rows["targets"] = inp["targets"].index_select(0, idx).cpu()
    out_rows = {k: v.index_select(0, idx) for k, v in out.items()}
    check_against_oracle(op, dtype, inp_rows, out_rows, what=what)


def check_workload(op, dtype, M, N, sigma, seed):
    inp = syn.make_inputs(op, dtype, M, N, seed, DEV, sigma)
    out = run_gpu(op, inp, dtype)
    if M * N <= WHOLE_MATRIX_ELEMENTS:
        block = max(1, ORACLE_BLOCK_ELEMENTS // N)
        for r0 in range(0, M, block):
            idx = torch.arange(r0, min(M, r0 + block), device=DEV)
            check_rows_against_oracle(op, dtype, inp, out, idx, f"{op} {dtype} {M}x{N} rows {r0}+")
    else:
        idx = sample_rows(M, seed).to(DEV)
        check_rows_against_oracle(op, dtype, inp, out, idx, f"{op} {dtype} {M}x{N} sampled rows")
    whole_matrix_properties(op, dtype, inp, out, N)
    del inp, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", sorted(syn.WORKLOADS))
def test_benchmark_workload(name):
    op, dtype, M, N, sigma = syn.WORKLOADS[name]
    check_workload(op, dtype, M, N, sigma, seed=1000)


@pytest.mark.parametrize("N", syn.SWEEP_N)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "xent"])
def test_sweep_grid(op, dtype, N):
    check_workload(op, dtype, syn.SWEEP_M[0], N, 1.0, seed=2000 + N)


@pytest.mark.parametrize("M", syn.SWEEP_M[1:])
def test_sweep_largest_rows(M):
    """The largest M of the sweep at its longest row (up to 64 GiB moved)."""
    check_workload("softmax", "f32", M, syn.SWEEP_N[-1], 1.0, seed=3000 + M)


@pytest.mark.parametrize("op,dtype", [("rmsnorm", "f32"), ("rmsnorm", "bf16"), ("xent", "f32"), ("xent", "bf16"),
                                      ("softmax", "bf16")])
def test_sweep_largest_shape(op, dtype):
    """The sweep's largest shape, 32768 x 262144 (2^33 elements, element
    offsets past 2^32), for the other operators and dtypes."""
    check_workload(op, dtype, syn.SWEEP_M[-1], syn.SWEEP_N[-1], 1.0, seed=3100)


def check_backward_workload(op, dtype, M, N, sigma, seed):
    """One backward call at full size on the device (the saved forward
    quantities are the generators' stand-ins of the right range), checked on
    sampled rows against the oracle, every row for finiteness, and RMSNorm's
    dw over all rows against a float64 column sum."""
    base = op[:-len("_bwd")]
    case = syn.make_inputs(op, dtype, M, N, seed, DEV, sigma)
    out = tb.run_gpu(base, dtype, case)
    dx = out["dx"]
    for r0 in range(0, M, 1024):
        assert torch.isfinite(dx[r0:r0 + 1024]).all(), f"{op} {M}x{N}: non-finite dx near row {r0}"
    idx = sample_rows(M, seed).to(DEV)
    rows = {k: (v.index_select(0, idx) if v.dim() == 2 or k in ("rstd", "lse", "dloss", "targets") else v).cpu()
            for k, v in case.items()}
    what = f"{op} {dtype} {M}x{N} sampled rows"
    got = dx.index_select(0, idx)
    if base in ("softmax", "xent"):
        tb.check(base, dtype, rows, {"dx": got}, what)
    else:
        x, w, r, dy = (to_f64(rows[k]) for k in ("x", "w", "rstd", "dy"))
        ref_dx, _ = oracle.rmsnorm_bwd(x, w, r, dy)  # dx rows are row-local; the dw of these rows is not dw
        r2 = r[:, None]
        scale = r2 * np.abs(dy) * w + np.abs(x) * r2 ** 3 * np.sum(np.abs(dy * w * x), axis=1, keepdims=True) / N
        check_scaled(to_f64(got), ref_dx, scale, dtype, f"rmsnorm bwd dx {what}")
        dw = torch.zeros(N, dtype=torch.float64, device=DEV)
        dws = torch.zeros(N, dtype=torch.float64, device=DEV)
        for r0 in range(0, M, 1024):
            t = case["dy"][r0:r0 + 1024].double() * case["x"][r0:r0 + 1024].double()
            t *= case["rstd"][r0:r0 + 1024].double()[:, None]
            dw += t.sum(0)
            dws += t.abs().sum(0)
            del t
        check_scaled(to_f64(out["dw"]), dw.cpu().numpy(), dws.cpu().numpy(), "f32", f"rmsnorm bwd dw {op} {M}x{N}")
    del case, out, dx
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", sorted(syn.BWD_WORKLOADS))
def test_backward_workload(name):
    op, dtype, M, N, sigma = syn.BWD_WORKLOADS[name]
    check_backward_workload(op, dtype, M, N, sigma, seed=1100)


@pytest.mark.parametrize("op", ["softmax_bwd", "rmsnorm_bwd", "xent_bwd"])
def test_backward_largest_sweep_shape(op):
    """The sweep's largest backward shape, bf16 32768 x 262144: 2^33 elements
    (16 GiB a matrix), so element offsets pass 2^32."""
    check_backward_workload(op, "bf16", syn.SWEEP_M[-1], syn.SWEEP_N[-1], 1.0, seed=3300)
