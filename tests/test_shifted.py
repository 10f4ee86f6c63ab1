"""Rows that do not start on a 16-byte boundary: the shifted ring kernel (rows of
any length, x and y with the same alignment modulo 16) and the masked kernel it
falls back to, against the fp64 oracle through the C ABI."""
import pytest
import torch

from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
import test_layernorm as tln
from test_parity import DEV, DT_CODE, OP_CODE, check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu

OPS = ("softmax", "rmsnorm", "xent")


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    qb.load_library()
    torch.cuda.set_device(0)
    yield


def shifted_copy(t, elems, fill=None):
    """A copy of t whose data starts `elems` elements past a 16-byte boundary."""
    store = torch.empty(t.numel() + 16, dtype=t.dtype, device=DEV)
    v = store[elems:elems + t.numel()].view(t.shape)
    if fill is None:
        v.copy_(t)
    else:
        v.fill_(fill)
    return v


# Lengths around every plan boundary of the shifted kernel (row groups of
# 8 ... 256 threads of 5 or 9 vectors, clusters of 2 ... 16, streamed
# cross-entropy in equal chunks).
SHIFT_N = [1, 5, 9, 60, 123, 153, 251, 311, 313, 571, 573, 627, 1003, 1143, 1149, 1263, 2045,
           2295, 2301, 2547, 4097, 4599, 4605, 5111, 9207, 9209, 10227, 16385, 18415, 18419,
           32761, 50257, 65537, 131071, 250001]


@pytest.mark.parametrize("N", SHIFT_N)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", OPS)
def test_shifted_lengths(op, dtype, N):
    M = 3 if N > 16384 else max(3, min(29, (1 << 20) // N))
    plan = qb.qk_get_plan(OP_CODE[op], DT_CODE[dtype], M, N)
    inp = syn.make_inputs(op, dtype, M, N, 10000 + N, "cpu")
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = run_gpu(op, dev, dtype)
    check_against_oracle(op, dtype, inp, out, what=f"shifted {dtype} {M}x{N} plan {plan['path']}")


@pytest.mark.parametrize("N", [7, 571, 1001, 1143, 2295, 4097, 4605, 9207, 20001])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_shifted_layernorm(dtype, N):
    full = tln.full_check(dtype, 5, N, seed=10100 + N)
    assert full is not None


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", OPS)
def test_plan_is_the_shifted_kernel(op, dtype):
    """Unaligned N (with aligned pointers) takes path 6 up to its capacity."""
    assert qb.qk_get_plan(OP_CODE[op], DT_CODE[dtype], 64, 4097)["path"] == 6
    if op != "xent":  # rows too long for 16 CTAs of 2304 vectors fall back to the masked kernel
        assert qb.qk_get_plan(OP_CODE[op], DT_CODE[dtype], 4, 400003)["path"] == 2


@pytest.mark.parametrize("M,N", [(4099, 1001), (1023, 5003), (61, 70001)])
@pytest.mark.parametrize("op", OPS)
def test_shifted_many_rows(op, M, N):
    """Many rows per CTA: every slot and both barrier parities reused, rows
    starting at every offset inside a vector."""
    inp = syn.make_inputs(op, "bf16", M, N, 10200 + N, "cpu")
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = run_gpu(op, dev, "bf16")
    rows = torch.tensor(sorted({0, 1, 2, 3, 4, 5, 6, 7, 8, M // 2, M - 2, M - 1}))
    check_against_oracle(op, "bf16", inp, out, rows=rows, what=f"shifted many rows {M}x{N}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("offsets", [(3, 3), (1, 0), (0, 2)])
def test_offset_pointers(op, dtype, offsets):
    """x and y starting some elements past a 16-byte boundary: the same offset
    takes the shifted kernel, different ones the masked kernel."""
    M, N = 7, 4096 + 8
    ox, oy = offsets
    inp = syn.make_inputs(op, dtype, M, N, 10300 + ox * 4 + oy, "cpu")
    dev = {k: v.to(DEV) for k, v in inp.items()}
    dev["x"] = shifted_copy(dev["x"], ox)
    y = shifted_copy(dev["x"], oy, fill=float("nan")) if op != "xent" else None
    out = run_gpu(op, dev, dtype, y=y)
    check_against_oracle(op, dtype, inp, out, what=f"offsets {offsets}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [4097, 65537])
def test_shifted_in_place(dtype, N):
    M = 5
    for op in ("softmax", "rmsnorm"):
        inp = syn.make_inputs(op, dtype, M, N, 10400 + N, "cpu")
        dev = {k: v.to(DEV) for k, v in inp.items()}
        x = shifted_copy(dev["x"], 1)
        dev["x"] = x
        out = run_gpu(op, dev, dtype, y=x)
        check_against_oracle(op, dtype, inp, out, what="shifted, in place")


def test_shifted_xent_targets_and_variants():
    """Targets at both ends of odd rows, out of range, ignored; z-loss."""
    M, N = 8, 50257
    inp = syn.make_inputs("xent", "bf16", M, N, 10500, "cpu")
    t = torch.tensor([0, N - 1, 1, N - 2, -1, N, 7, 25000], dtype=torch.int64)
    inp["targets"] = t
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = run_gpu("xent", dev, "bf16")
    check_against_oracle("xent", "bf16", inp, out, what="shifted targets")
    loss = out["loss"].cpu()
    assert torch.isnan(loss[[4, 5]]).all() and torch.isfinite(loss[[0, 1, 2, 3, 6, 7]]).all()
