"""Rows with -inf entries (masked logits) through every forward path, against
the fp64 oracle.

A -inf entry has probability exactly 0: softmax writes 0 there and the rest of
the row is the softmax of the finite entries; cross-entropy's log-sum-exp
ignores it.  The oracle computes the same from the definition in float64
(exp(-inf - m) = 0), so partly masked rows are compared element by element
with the usual tolerances.  A row with no finite entry has no distribution:
softmax gives 0/0 = NaN in every entry, as the oracle does, so the whole
matrix is compared (NaN must meet NaN); cross-entropy gives that row
lse = -inf and loss = NaN (the library's documented answer, checked exactly:
the oracle's shifted form gives NaN for its lse).  A masked target gives
loss = +inf.  The backward passes are checked on the rows with a finite
entry: masked entries get a gradient of exactly 0.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
from parity import check_rows, check_scalars, check_scaled, loss_denominator, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DT = {"f32": qb.QK_F32, "bf16": qb.QK_BF16}
NEG_INF = float("-inf")
FULLY_MASKED = 2  # the row of each batch with no finite entry


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    qb.load_library()
    torch.cuda.set_device(0)


def masked_rows(M, N, dtype, seed):
    """M seeded N(0, 1) rows, then -inf patterns: row 0 about 30 % masked at
    random, row 1 all but one entry, row 2 every entry, row 3 none, row 4
    about 90 %, rows 5+ all but the first and last entry."""
    x = syn.normal_rows(M, N, dtype, seed, "cpu", sigma=2.0)
    rng = np.random.default_rng(seed)
    keep = np.ones((M, N), dtype=bool)
    keep[0] = rng.random(N) >= 0.3
    keep[1] = False
    keep[1, rng.integers(N)] = True
    keep[2] = False
    if M > 4:
        keep[4] = rng.random(N) >= 0.9
        keep[4, rng.integers(N)] = True
    for i in range(5, M):
        keep[i, 1:N - 1] = False
    x[torch.from_numpy(~keep)] = NEG_INF
    return x, keep


def plan_path(op, dtype, M, N):
    return qb.qk_get_plan(op, DT[dtype], M, N)["path"]


# (M, N): shifted kernel (rows of 7), ring (4096), clustered ring (131072),
# masked kernel for long unaligned rows (4097), rows streamed twice (3 * 2^19).
SHAPES = [(6, 7), (6, 4096), (6, 131072), (6, 4097), (5, 3 * 2 ** 19)]


@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_softmax_masked_rows(dtype, M, N):
    if N == 3 * 2 ** 19:
        assert plan_path(qb.QK_OP_SOFTMAX, dtype, M, N) == 4
    x, keep = masked_rows(M, N, dtype, 9100 + N)
    xd = x.to(DEV)
    y = torch.full_like(xd, float("nan"))
    qb.qk_softmax_fwd(xd, y, M, N, DT[dtype])
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    got = to_f64(y)
    ref = oracle.softmax_fwd(to_f64(x))
    assert np.isnan(ref[FULLY_MASKED]).all()
    check_rows(got, ref, dtype, True, f"masked softmax {M}x{N}")
    rows = [i for i in range(M) if i != FULLY_MASKED]
    assert np.all(got[rows][~keep[rows]] == 0.0), "a masked entry got a nonzero probability"

    # backward on the rows with a finite entry: y = 0 at masked entries, so dx = 0 there
    if N > qb.qk_max_row_elements(qb.QK_OP_SOFTMAX_BWD, DT[dtype]):
        return  # beyond the backward kernels' row limit
    Mb = len(rows)
    yb = y[rows].contiguous()
    dy = syn.normal_rows(Mb, N, dtype, 9200 + N, "cpu").to(DEV)
    dx = torch.full_like(yb, float("nan"))
    qb.qk_softmax_bwd(yb, dy, dx, Mb, N, DT[dtype])
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    y64, dy64 = to_f64(yb), to_f64(dy)
    ref_dx = oracle.softmax_bwd(y64, dy64)
    scale = y64 * (np.abs(dy64) + np.sum(np.abs(dy64 * y64), axis=1, keepdims=True))
    gdx = to_f64(dx)
    check_scaled(gdx, ref_dx, scale, dtype, f"masked softmax bwd {M}x{N}")
    assert np.all(gdx[~keep[rows]] == 0.0), "a masked entry got a nonzero gradient"


XENT_SHAPES = [(6, 7), (6, 4096), (6, 131072), (6, 4097)]


@pytest.mark.parametrize("M,N", XENT_SHAPES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_xent_masked_rows(dtype, M, N):
    x, keep = masked_rows(M, N, dtype, 9300 + N)
    # targets: the smallest finite logit of the row, so that loss = lse - x[t]
    # is not a small difference of two large numbers (rows with one finite
    # entry give loss = 0 exactly); row 3's target is masked out below, giving
    # loss = +inf; the fully masked row keeps target 0
    t = np.zeros(M, dtype=np.int64)
    xf = x.to(torch.float64).numpy()
    for i in range(M):
        finite = np.flatnonzero(keep[i])
        t[i] = finite[np.argmin(xf[i, finite])] if finite.size else 0
    x[3, int(t[3])] = NEG_INF
    keep[3, int(t[3])] = False
    targets = torch.from_numpy(t)
    xd, td = x.to(DEV), targets.to(DEV)
    loss = torch.full((M,), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((M,), float("nan"), dtype=torch.float32, device=DEV)
    qb.qk_xent_fwd(xd, td, loss, lse, M, N, DT[dtype])
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    gl, gs = to_f64(loss), to_f64(lse)
    rows = [i for i in range(M) if i not in (FULLY_MASKED, 3)]
    ref_loss, ref_lse = oracle.xent_fwd(to_f64(x[rows]), t[rows])
    check_scalars(gs[rows], ref_lse, f"masked lse {M}x{N}")
    check_scalars(gl[rows], ref_loss, f"masked loss {M}x{N}", loss_denominator(ref_loss, ref_lse))
    ref3_loss, ref3_lse = oracle.xent_fwd(to_f64(x[3:4]), t[3:4])
    check_scalars(gs[3:4], ref3_lse, f"masked-target lse {M}x{N}")
    assert np.isposinf(ref3_loss[0]) and np.isposinf(gl[3]), "a masked target gives loss = +inf"
    assert np.isneginf(gs[FULLY_MASKED]) and np.isnan(gl[FULLY_MASKED])

    # backward on the rows with a finite lse, given the oracle's lse in fp32
    brow = [i for i in range(M) if i != FULLY_MASKED]
    lse32 = torch.from_numpy(np.concatenate([ref_lse[:3 - 1], ref3_lse, ref_lse[3 - 1:]])
                             .astype(np.float32))
    assert lse32.numel() == len(brow)
    xb = x[brow].contiguous()
    tb = targets[brow].contiguous()
    Mb = len(brow)
    dloss = torch.from_numpy(np.random.default_rng(9400 + N).uniform(0.5, 1.5, Mb).astype(np.float32))
    dx = torch.full((Mb, N), float("nan"), dtype=syn.DTYPES[dtype], device=DEV)
    qb.qk_xent_bwd(xb.to(DEV), tb.to(DEV), lse32.to(DEV), dloss.to(DEV), dx, Mb, N, DT[dtype])
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    x64, l64, g64 = to_f64(xb), lse32.double().numpy(), dloss.double().numpy()
    ref_dx = oracle.xent_bwd(x64, tb.numpy(), l64, g64)
    onehot = np.zeros_like(x64)
    onehot[np.arange(Mb), tb.numpy()] = 1.0
    scale = np.abs(g64)[:, None] * (np.exp(x64 - l64[:, None]) + onehot)
    gdx = to_f64(dx)
    check_scaled(gdx, ref_dx, scale, dtype, f"masked xent bwd {M}x{N}")
    kb = keep[brow].copy()
    kb[np.arange(Mb), tb.numpy()] = True  # the target entry carries -1 (times dloss)
    assert np.all(gdx[~kb] == 0.0), "a masked entry got a nonzero gradient"
