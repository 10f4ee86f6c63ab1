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
"""
import math

import numpy as np
import pytest
import torch

from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
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
