"""RMSNorm backward without a caller-provided workspace.

qk_rmsnorm_bwd_noalloc serves callers that cannot allocate device memory: it
takes its scratch from a fixed array in the library's device memory.  This
checks, through the C ABI, two calls in a row (the second reuses the array
the first one left behind):
  * against the fp64 oracle's RMSNorm backward -- dx on 256 seeded rows
    (every row for the smaller case), dw over all rows -- within the
    tolerance the backward tests use;
  * against the ordinary entry point given a PyTorch-allocated workspace:
    both run the same plan and kernels, so dx and dw must agree bit for bit.
It needs nothing from the other tests and runs alone in a fresh process as
well."""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
from parity import check_scaled, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    qb.load_library()
    torch.cuda.set_device(0)


def inputs(M, N, dtype, seed):
    return {"x": syn.normal_rows(M, N, dtype, seed, DEV),
            "w": syn.uniform_weight(N, dtype, seed + 1, DEV),
            "rstd": syn.uniform_weight(M, "f32", seed + 2, DEV),
            "dy": syn.normal_rows(M, N, dtype, seed + 3, DEV)}


def with_workspace(d, M, N, code):
    nbytes = qb.qk_rmsnorm_bwd_workspace_size(M, N, code)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    dx = torch.empty_like(d["x"])
    dw = torch.empty(N, dtype=torch.float32, device=DEV)
    qb.qk_rmsnorm_bwd(d["x"], d["w"], d["rstd"], d["dy"], dx, dw, ws, nbytes, M, N, code)
    return dx, dw


def without_workspace(d, M, N, code):
    dx = torch.full_like(d["x"], float("nan"))
    dw = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    qb.qk_rmsnorm_bwd_noalloc(d["x"], d["w"], d["rstd"], d["dy"], dx, dw, M, N, code)
    return dx, dw


def check_against_oracle(d, dx, dw, dtype, seed, what):
    """dx on every row of a small case, else on 256 seeded rows (the first and
    the last among them); dw, a sum over every row, on all columns."""
    x, w, r, dy = (to_f64(d[k]) for k in ("x", "w", "rstd", "dy"))
    ref_dx, ref_dw = oracle.rmsnorm_bwd(x, w, r, dy)
    M, N = x.shape
    if M <= 1024:
        rows = np.arange(M)
    else:
        rows = np.sort(np.random.default_rng(seed).choice(M, size=256, replace=False))
        rows = np.union1d(rows, [0, M - 1])
    r2 = r[:, None]
    sdx = r2 * np.abs(dy) * w + np.abs(x) * r2 ** 3 * np.sum(np.abs(dy * w * x), axis=1, keepdims=True) / N
    sdw = np.sum(np.abs(dy * x) * r2, axis=0)
    check_scaled(to_f64(dx)[rows], ref_dx[rows], sdx[rows], dtype, f"noalloc dx {what}")
    check_scaled(to_f64(dw), ref_dw, sdw, "f32", f"noalloc dw {what}")


@pytest.mark.parametrize("dtype,M,N", [("bf16", 16384, 4096), ("f32", 777, 16384)])
def test_two_calls_match_the_oracle_and_the_workspace_entry_point(dtype, M, N):
    code = qb.QK_F32 if dtype == "f32" else qb.QK_BF16
    for call, seed in enumerate((31, 47)):  # two calls in a row, different data
        d = inputs(M, N, dtype, seed)
        dx, dw = without_workspace(d, M, N, code)
        torch.cuda.synchronize()
        assert qb.qk_get_device_status() == qb.QK_OK
        check_against_oracle(d, dx, dw, dtype, seed, f"call {call}")
        ref_dx, ref_dw = with_workspace(d, M, N, code)
        torch.cuda.synchronize()
        assert torch.equal(dx, ref_dx), f"noalloc dx differs from the workspace entry point, call {call}"
        assert torch.equal(dw, ref_dw), f"noalloc dw differs from the workspace entry point, call {call}"


def test_sizes_beyond_the_array_are_refused():
    """Find a shape whose workspace exceeds the fixed 16 MiB and check that it
    is refused before anything runs.  The workspace holds one fp32 row of N
    partial sums per CTA (or cluster) of the launch, so it grows with M until
    the persistent grid is full: the smallest such M is searched for each N.
    Rows of an odd length take the masked kernel (one row per CTA), whose
    grids are the largest."""
    limit = 16 << 20
    for dtype, code in (("f32", qb.QK_F32), ("bf16", qb.QK_BF16)):
        for N in (8191, 8193, 16383, 4095, 8192, 16384, 32768, 65536, 131072):
            if N > qb.qk_max_row_elements(qb.QK_OP_RMSNORM_BWD, code):
                continue
            M = 64
            while M <= (1 << 16) and qb.qk_rmsnorm_bwd_workspace_size(M, N, code) <= limit:
                M *= 2
            if M > (1 << 16) or M * N * 4 > (1 << 31):
                continue
            d = inputs(M, N, dtype, 5)
            dx = torch.full_like(d["x"], float("nan"))
            dw = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
            with pytest.raises(qb.QkError) as e:
                qb.qk_rmsnorm_bwd_noalloc(d["x"], d["w"], d["rstd"], d["dy"], dx, dw, M, N, code)
            assert e.value.status == qb.QK_ERR_UNSUPPORTED
            torch.cuda.synchronize()
            assert torch.isnan(dw).all() and torch.isnan(dx).all(), "a refused call wrote its outputs"
            return
    pytest.skip("no default plan on this device needs more than the fixed scratch")
