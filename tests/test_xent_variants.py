"""Cross-entropy variants (ignore index, z-loss, mean over rows) through the
C ABI against the fp64 oracle, on the fast, masked and streamed paths."""
import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
from parity import REL_F32, check_scaled, check_scalars, loss_denominator, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DT = {"f32": qb.QK_F32, "bf16": qb.QK_BF16}


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    qb.load_library()
    torch.cuda.set_device(0)


def case(dtype, M, N, seed, ignore=-100, frac_ignored=0.25):
    x = syn.normal_rows(M, N, dtype, seed, "cpu", sigma=2 ** 0.5)
    t = syn.uniform_targets(M, N, seed + 1, "cpu")
    mask = torch.from_numpy(np.random.default_rng(seed).random(M) < frac_ignored)
    t[mask] = ignore
    return x, t


@pytest.mark.parametrize("z", [0.0, 1e-4, 0.5])
@pytest.mark.parametrize("N", [256, 1001, 4096, 131072])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forward_and_mean(dtype, N, z):
    M = 4 if N > 100000 else 37
    x, t = case(dtype, M, N, seed=10 + N)
    ref_loss, ref_lse, ref_mean = oracle.xent_fwd_ex(to_f64(x), t.numpy(), -100, z)
    xd, td = x.to(DEV), t.to(DEV)
    loss = torch.full((M,), float("nan"), device=DEV)
    lse = torch.full((M,), float("nan"), device=DEV)
    mean = torch.full((1,), float("nan"), device=DEV)
    qb.qk_xent_fwd_ex(xd, td, loss, lse, mean, M, N, DT[dtype], ignore_index=-100, z_loss=z)
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    check_scalars(to_f64(lse), ref_lse, "lse")
    check_scalars(to_f64(loss), ref_loss, "loss", denom=loss_denominator(ref_loss, ref_lse))
    assert torch.all(loss.cpu()[t == -100] == 0)
    assert abs(mean.item() - ref_mean) <= REL_F32 * abs(ref_mean)


def test_mean_of_no_rows_is_nan():
    x, t = case("f32", 8, 512, seed=3, ignore=-1, frac_ignored=1.0)
    loss = torch.empty(8, device=DEV)
    mean = torch.empty(1, device=DEV)
    qb.qk_xent_fwd_ex(x.to(DEV), t.to(DEV), loss, None, mean, 8, 512, qb.QK_F32, ignore_index=-1)
    torch.cuda.synchronize()
    assert math.isnan(mean.item()) and torch.all(loss == 0)


def test_plain_call_matches_options_defaults():
    x, t = case("bf16", 64, 4096, seed=4, frac_ignored=0.0)
    xd, td = x.to(DEV), t.to(DEV)
    a = torch.empty(64, device=DEV)
    b = torch.empty(64, device=DEV)
    qb.qk_xent_fwd(xd, td, a, None, 64, 4096, qb.QK_BF16)
    qb.qk_xent_fwd_ex(xd, td, b, None, None, 64, 4096, qb.QK_BF16)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("z", [0.0, 0.5])
@pytest.mark.parametrize("N", [256, 4096, 131072])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward(dtype, N, z):
    M = 4 if N > 100000 else 37
    x, t = case(dtype, M, N, seed=20 + N)
    _, lse, _ = oracle.xent_fwd_ex(to_f64(x), t.numpy(), -100, z)
    g = syn.uniform_weight(M, "f32", 7, "cpu", lo=0.25, hi=2.0)
    ref = oracle.xent_bwd_ex(to_f64(x), t.numpy(), lse, to_f64(g), -100, z)
    xd = x.to(DEV)
    dx = torch.full_like(xd, float("nan"))
    qb.qk_xent_bwd_ex(xd, t.to(DEV), torch.from_numpy(lse).float().to(DEV), g.to(DEV), dx, M, N,
                      DT[dtype], ignore_index=-100, z_loss=z)
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    lse32 = to_f64(torch.from_numpy(lse).float())
    tn = t.numpy()
    onehot = np.zeros((M, N))
    ok = (tn >= 0) & (tn < N)
    onehot[np.arange(M)[ok], tn[ok]] = 1.0
    p = np.exp(to_f64(x) - lse32[:, None])
    scale = np.abs(to_f64(g))[:, None] * (np.abs(1 + 2 * z * lse32)[:, None] * p + onehot)
    check_scaled(to_f64(dx), ref, scale, dtype, f"xent bwd ex z={z}")
    assert torch.all(dx.cpu()[t == -100] == 0)


@pytest.mark.parametrize("ignore", [None, -(2 ** 63)])
@pytest.mark.parametrize("N", [1024, 1001, 131072])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_extreme_targets_forward_mean_and_backward(dtype, N, ignore):
    """INT64_MIN and INT64_MAX targets: out of range (NaN loss, NaN gradient
    row) when no ignore index is given; with INT64_MIN as the ignore index,
    those rows give loss 0, a zero gradient and stay out of the mean, while
    INT64_MAX rows are still NaN.  Ring (1024), shifted (1001) and streamed
    (131072) rows."""
    M = 6
    x = syn.normal_rows(M, N, dtype, 40 + N, "cpu", sigma=2 ** 0.5)
    t = torch.tensor([-(2 ** 63), 5, 2 ** 63 - 1, 0, N - 1, -(2 ** 63)], dtype=torch.int64)
    ref_loss, ref_lse, ref_mean = oracle.xent_fwd_ex(to_f64(x), t.numpy(), ignore_index=ignore)
    xd, td = x.to(DEV), t.to(DEV)
    loss = torch.full((M,), float("nan"), device=DEV)
    lse = torch.full((M,), float("nan"), device=DEV)
    mean = torch.full((1,), 0.0, device=DEV)
    qb.qk_xent_fwd_ex(xd, td, loss, lse, mean, M, N, DT[dtype], ignore_index=ignore)
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    check_scalars(to_f64(lse), ref_lse, "lse")
    check_scalars(to_f64(loss), ref_loss, "loss", denom=loss_denominator(ref_loss, ref_lse))
    # INT64_MAX is never ignored, so the mean over the rows not ignored is NaN either way
    assert math.isnan(mean.item()) and math.isnan(ref_mean)
    g = syn.uniform_weight(M, "f32", 9, "cpu", lo=0.25, hi=2.0)
    ref = oracle.xent_bwd_ex(to_f64(x), t.numpy(), ref_lse, to_f64(g), ignore_index=ignore)
    dx = torch.full_like(xd, float("nan"))
    qb.qk_xent_bwd_ex(xd, td, torch.from_numpy(ref_lse).float().to(DEV), g.to(DEV), dx, M, N, DT[dtype],
                      ignore_index=ignore)
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    lse32 = to_f64(torch.from_numpy(ref_lse).float())
    tn = t.numpy()
    onehot = np.zeros((M, N))
    ok = (tn >= 0) & (tn < N)
    onehot[np.arange(M)[ok], tn[ok]] = 1.0
    scale = np.abs(to_f64(g))[:, None] * (np.exp(to_f64(x) - lse32[:, None]) + onehot)
    check_scaled(to_f64(dx), ref, scale, dtype, f"xent bwd ex, extreme targets, ignore {ignore}")
    got = dx.cpu()
    assert torch.isnan(got[2]).all()
    if ignore is None:
        assert torch.isnan(got[[0, 5]]).all() and torch.isnan(loss.cpu()[[0, 2, 5]]).all()
    else:
        assert (got[[0, 5]] == 0).all() and (loss.cpu()[[0, 5]] == 0).all()
