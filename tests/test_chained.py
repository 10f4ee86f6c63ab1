"""Dependent calls back to back on one stream, with no synchronisation between
them: each kernel is launched with programmatic dependent launch and may
start (and prefetch its first rows into L2) while the previous one is still
running.  Every stage is checked against the fp64 oracle applied to the exact
bytes it consumed -- the previous stage's device output -- so a stage that
read its input before the producer had finished writing it fails, and so does
a producer whose input a later call overwrote too early."""
import pytest
import torch

from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
import test_layernorm as tln
from test_parity import DEV, DT_CODE, EPS, check_against_oracle

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


def _nan(shape, dtype):
    return torch.full(shape, float("nan"), dtype=dtype, device=DEV)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,N", [(4099, 4096), (300, 1024), (64, 65536), (7, 4097)])
def test_dependent_calls_on_one_stream(dtype, M, N):
    code = DT_CODE[dtype]
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    passes = 3
    inp = [syn.make_inputs("layernorm", dtype, M, N, 12000 + 10 * r + N, "cpu") for r in range(passes)]
    z0 = [syn.make_inputs("softmax", dtype, M, N, 12500 + 10 * r + N, "cpu")["x"] for r in range(passes)]
    g = torch.Generator().manual_seed(12100 + N)
    targets = torch.randint(0, N, (M,), generator=g, dtype=torch.int64)
    w, b, t = inp[0]["w"].to(DEV), inp[0]["b"].to(DEV), targets.to(DEV)
    # every buffer exists before the first launch of the chain
    X = [d["x"].to(DEV) for d in inp]
    Z = [z.to(DEV) for z in z0]
    Y1 = [_nan((M, N), tdt) for _ in range(passes)]
    R1 = [_nan((M,), torch.float32) for _ in range(passes)]
    S2 = [_nan((M, N), tdt) for _ in range(passes)]
    loss = [_nan((M,), torch.float32) for _ in range(passes)]
    lse = [_nan((M,), torch.float32) for _ in range(passes)]
    Y4 = [_nan((M, N), tdt) for _ in range(passes)]
    mean4 = [_nan((M,), torch.float32) for _ in range(passes)]
    rstd4 = [_nan((M,), torch.float32) for _ in range(passes)]
    R6 = [_nan((M,), torch.float32) for _ in range(passes)]
    torch.cuda.synchronize()

    for r in range(passes):
        qb.qk_rmsnorm_fwd(X[r], w, Y1[r], R1[r], M, N, EPS, code)    # a: reads X
        qb.qk_softmax_fwd(Y1[r], S2[r], M, N, code)                  # b: reads a's output
        qb.qk_softmax_fwd(Z[r], X[r], M, N, code)                    # c: overwrites what a read
        qb.qk_xent_fwd(S2[r], t, loss[r], lse[r], M, N, code)        # d: reads b's output
        qb.qk_layernorm_fwd(S2[r], w, b, Y4[r], mean4[r], rstd4[r], M, N, tln.EPS, code)  # e
        qb.qk_rmsnorm_fwd(Y4[r], w, Z[r], R6[r], M, N, EPS, code)   # f: overwrites what c read
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK

    w_cpu, b_cpu = inp[0]["w"], inp[0]["b"]
    for r in range(passes):
        what = f"pass {r} {dtype} {M}x{N}"
        check_against_oracle("rmsnorm", dtype, {"x": inp[r]["x"], "w": w_cpu},
                             {"y": Y1[r], "rstd": R1[r]}, what="a " + what)
        check_against_oracle("softmax", dtype, {"x": Y1[r].cpu()}, {"y": S2[r]}, what="b " + what)
        check_against_oracle("softmax", dtype, {"x": z0[r]}, {"y": X[r]}, what="c " + what)
        s2 = S2[r].cpu()
        check_against_oracle("xent", dtype, {"x": s2, "targets": targets},
                             {"loss": loss[r], "lse": lse[r]}, what="d " + what)
        tln.check({"x": s2, "w": w_cpu, "b": b_cpu},
                  {"y": Y4[r], "mean": mean4[r], "rstd": rstd4[r]}, dtype, what="e " + what)
        check_against_oracle("rmsnorm", dtype, {"x": Y4[r].cpu(), "w": w_cpu},
                             {"y": Z[r], "rstd": R6[r]}, what="f " + what)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_short_launches_get_a_deeper_ring(dtype):
    """Fewer than four items for each resident CTA: three ring slots (when that
    costs no resident CTA), and results unchanged; a long launch keeps the
    table's slot count."""
    code = DT_CODE[dtype]
    N = 4096 if dtype == "f32" else 8192  # 1024 vectors: one ring slot in the table
    short = qb.qk_get_plan(qb.QK_OP_SOFTMAX, code, 512, N)
    long_ = qb.qk_get_plan(qb.QK_OP_SOFTMAX, code, 65536, N)
    assert short["slots"] == 3 and long_["slots"] == 1
    assert short["ctas_per_sm"] == long_["ctas_per_sm"]
    inp = syn.make_inputs("softmax", dtype, 512, N, 12900, "cpu")
    y = _nan((512, N), torch.float32 if dtype == "f32" else torch.bfloat16)
    qb.qk_softmax_fwd(inp["x"].to(DEV), y, 512, N, code)
    torch.cuda.synchronize()
    check_against_oracle("softmax", dtype, inp, {"y": y}, what="short launch")
