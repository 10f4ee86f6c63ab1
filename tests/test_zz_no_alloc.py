"""RMSNorm backward without a caller-provided workspace.

qk_rmsnorm_bwd_noalloc serves callers that cannot allocate device memory: it
takes its scratch from a fixed array in the library's device memory.  This
checks, through the C ABI, that two calls in a row agree with the ordinary
entry point (which is given a PyTorch-allocated workspace) within the
tolerance the backward tests use -- the second call reuses the array the
first one left behind.  It needs nothing from the other tests and runs alone
in a fresh process as well."""
import numpy as np
import pytest
import torch

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


def scales(d):
    x, w, r, dy = (to_f64(d[k]) for k in ("x", "w", "rstd", "dy"))
    r2 = r[:, None]
    sdx = r2 * np.abs(dy) * w + np.abs(x) * r2 ** 3 * np.sum(np.abs(dy * w * x), axis=1, keepdims=True) / x.shape[1]
    sdw = np.sum(np.abs(dy * x) * r2, axis=0)
    return sdx, sdw


@pytest.mark.parametrize("dtype,M,N", [("bf16", 16384, 4096), ("f32", 777, 16384)])
def test_two_calls_match_the_workspace_entry_point(dtype, M, N):
    code = qb.QK_F32 if dtype == "f32" else qb.QK_BF16
    for call, seed in enumerate((31, 47)):  # two calls in a row, different data
        d = inputs(M, N, dtype, seed)
        ref_dx, ref_dw = with_workspace(d, M, N, code)
        dx, dw = without_workspace(d, M, N, code)
        torch.cuda.synchronize()
        assert qb.qk_get_device_status() == qb.QK_OK
        sdx, sdw = scales(d)
        check_scaled(to_f64(dx), to_f64(ref_dx), sdx, dtype, f"noalloc dx, call {call}")
        check_scaled(to_f64(dw), to_f64(ref_dw), sdw, "f32", f"noalloc dw, call {call}")


def test_sizes_beyond_the_array_are_refused():
    """Find a shape whose workspace exceeds the fixed 16 MiB (if any plan on
    this device needs that much) and check it is refused, not run."""
    limit = 16 << 20
    for dtype, code in (("bf16", qb.QK_BF16), ("f32", qb.QK_F32)):
        for N in (4096, 8192, 12288, 16384, 32768, 65536, 131072):
            if N > qb.qk_max_row_elements(qb.QK_OP_RMSNORM_BWD, code):
                continue
            if qb.qk_rmsnorm_bwd_workspace_size(64, N, code) > limit:
                d = inputs(64, N, dtype, 5)
                dx = torch.empty_like(d["x"])
                dw = torch.empty(N, dtype=torch.float32, device=DEV)
                with pytest.raises(qb.QkError) as e:
                    qb.qk_rmsnorm_bwd_noalloc(d["x"], d["w"], d["rstd"], d["dy"], dx, dw, 64, N, code)
                assert e.value.status == qb.QK_ERR_UNSUPPORTED
                return
    pytest.skip("no default plan on this device needs more than the fixed scratch")
