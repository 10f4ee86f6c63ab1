"""Backward passes through the C ABI against the fp64 oracle.

Inputs: the forward quantities the backward passes consume (softmax y, RMSNorm
rstd, cross-entropy lse) come from the oracle's forward pass on seeded inputs,
rounded to the working dtype; the same bytes go to both sides.  Gradients can
cancel, so each element is checked against 1e-5 of the magnitude of the terms
that form it (plus one bf16 ulp for bf16 outputs): see parity.check_scaled."""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
from parity import check_scaled, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DT = {"f32": qb.QK_F32, "bf16": qb.QK_BF16}
OPC = {"softmax": qb.QK_OP_SOFTMAX_BWD, "rmsnorm": qb.QK_OP_RMSNORM_BWD, "xent": qb.QK_OP_XENT_BWD}


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    qb.load_library()
    torch.cuda.set_device(0)
    yield
    for op in OPC.values():
        for dt in DT.values():
            qb.qk_set_plan_override(op, dt, None)


def to_dtype(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(syn.DTYPES[dtype])


def make_case(op, dtype, M, N, seed):
    """Host tensors of one backward call (already rounded to dtype) and their fp64 copies."""
    if op == "softmax":
        x = syn.normal_rows(M, N, dtype, seed, "cpu")
        y = to_dtype(oracle.softmax_fwd(to_f64(x)), dtype)
        dy = syn.normal_rows(M, N, dtype, seed + 1, "cpu")
        return {"y": y, "dy": dy}
    if op == "rmsnorm":
        x = syn.normal_rows(M, N, dtype, seed, "cpu")
        w = syn.uniform_weight(N, dtype, seed + 1, "cpu")
        _, r = oracle.rmsnorm_fwd(to_f64(x), to_f64(w), 1e-6)
        dy = syn.normal_rows(M, N, dtype, seed + 2, "cpu")
        return {"x": x, "w": w, "rstd": torch.from_numpy(r).float(), "dy": dy}
    x = syn.normal_rows(M, N, dtype, seed, "cpu", sigma=2 ** 0.5)
    t = syn.uniform_targets(M, N, seed + 1, "cpu")
    _, lse = oracle.xent_fwd(to_f64(x), t.numpy())
    g = syn.uniform_weight(M, "f32", seed + 2, "cpu", lo=0.25, hi=2.0)
    return {"x": x, "targets": t, "lse": torch.from_numpy(lse).float(), "dloss": g}


def run_gpu(op, dtype, case, inplace=False):
    d = {k: v.to(DEV) for k, v in case.items()}
    M, N = (d["y"] if op == "softmax" else d["x"]).shape
    code = DT[dtype]
    if op == "softmax":
        dx = d["dy"] if inplace else torch.full_like(d["y"], float("nan"))
        qb.qk_softmax_bwd(d["y"], d["dy"], dx, M, N, code)
        out = {"dx": dx}
    elif op == "rmsnorm":
        dx = d["dy"] if inplace else torch.full_like(d["x"], float("nan"))
        dw = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
        nbytes = qb.qk_rmsnorm_bwd_workspace_size(M, N, code)
        ws = torch.full((max(nbytes, 16) // 4,), float("nan"), dtype=torch.float32, device=DEV)
        qb.qk_rmsnorm_bwd(d["x"], d["w"], d["rstd"], d["dy"], dx, dw, ws, nbytes, M, N, code)
        out = {"dx": dx, "dw": dw}
    else:
        dx = d["x"] if inplace else torch.full_like(d["x"], float("nan"))
        qb.qk_xent_bwd(d["x"], d["targets"], d["lse"], d["dloss"], dx, M, N, code)
        out = {"dx": dx}
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    return out


def check(op, dtype, case, out, what):
    if op == "softmax":
        y, dy = to_f64(case["y"]), to_f64(case["dy"])
        ref = oracle.softmax_bwd(y, dy)
        scale = y * (np.abs(dy) + np.sum(np.abs(dy * y), axis=1, keepdims=True))
        check_scaled(to_f64(out["dx"]), ref, scale, dtype, f"softmax bwd {what}")
    elif op == "rmsnorm":
        x, w, r, dy = to_f64(case["x"]), to_f64(case["w"]), to_f64(case["rstd"]), to_f64(case["dy"])
        ref_dx, ref_dw = oracle.rmsnorm_bwd(x, w, r, dy)
        N = x.shape[1]
        r2 = r[:, None]
        scale = r2 * np.abs(dy) * w + np.abs(x) * r2 ** 3 * np.sum(np.abs(dy * w * x), axis=1, keepdims=True) / N
        check_scaled(to_f64(out["dx"]), ref_dx, scale, dtype, f"rmsnorm bwd dx {what}")
        check_scaled(to_f64(out["dw"]), ref_dw, np.sum(np.abs(dy * x) * r2, axis=0), "f32",
                     f"rmsnorm bwd dw {what}")
    else:
        x, t = to_f64(case["x"]), case["targets"].numpy()
        lse, g = to_f64(case["lse"]), to_f64(case["dloss"])
        ref = oracle.xent_bwd(x, t, lse, g)
        onehot = np.zeros_like(x)
        ok = (t >= 0) & (t < x.shape[1])
        onehot[np.arange(x.shape[0])[ok], t[ok]] = 1.0
        scale = np.abs(g)[:, None] * (np.exp(x - lse[:, None]) + onehot)
        check_scaled(to_f64(out["dx"]), ref, scale, dtype, f"xent bwd {what}")


def rows_for(N):
    return max(3, min(37, (1 << 21) // N))


@pytest.mark.parametrize("N", [8, 64, 256, 1000, 1024, 4096, 8192, 16384, 65536, 131072])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "xent"])
def test_backward_shapes(op, dtype, N):
    M = rows_for(N)
    case = make_case(op, dtype, M, N, seed=5000 + N)
    check(op, dtype, case, run_gpu(op, dtype, case), f"{dtype} {M}x{N}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "xent"])
def test_backward_in_place(op, dtype):
    case = make_case(op, dtype, 19, 4096, seed=6000)
    check(op, dtype, case, run_gpu(op, dtype, case, inplace=True), "in place")


BWD_PLANS = [
    dict(threads=256, row_threads=8, vec_per_thread=4, cluster=1, slots=2, grid=3),
    dict(threads=256, row_threads=32, vec_per_thread=4, cluster=1, slots=1, grid=2),
    dict(threads=128, row_threads=128, vec_per_thread=4, cluster=1, slots=3, grid=5),
    dict(threads=256, row_threads=256, vec_per_thread=4, cluster=1, slots=2, grid=4),
]
CLUSTER_PLANS = {
    "softmax": dict(threads=256, row_threads=256, vec_per_thread=8, cluster=4, slots=1, grid=8),
    "rmsnorm": dict(threads=256, row_threads=256, vec_per_thread=4, cluster=8, slots=2, grid=16),
}


@pytest.mark.parametrize("pi", range(len(BWD_PLANS) + 1))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "xent"])
def test_backward_forced_plans(op, dtype, pi):
    if pi == len(BWD_PLANS):
        if op not in CLUSTER_PLANS:
            pytest.skip("cross-entropy backward streams rows instead of splitting them")
        plan = CLUSTER_PLANS[op]
    else:
        plan = BWD_PLANS[pi]
    E = 4 if dtype == "f32" else 8
    cap = plan["row_threads"] * plan["vec_per_thread"] * E * plan["cluster"]
    N = max(E, cap - 3 * E)
    if op == "xent" and plan["row_threads"] == plan["threads"]:
        N = 5 * cap + 7 * E  # several chunks per row
    rows_per_step = plan["threads"] // plan["row_threads"]
    M = max(61, 3 * rows_per_step * plan["grid"] + 5) if N <= 8192 else 9
    qb.qk_set_plan_override(OPC[op], DT[dtype], plan)
    try:
        got = qb.qk_get_plan(OPC[op], DT[dtype], M, N)
        assert got["grid"] == plan["grid"] and got["cluster"] == plan["cluster"]
        case = make_case(op, dtype, M, N, seed=7000 + N)
        check(op, dtype, case, run_gpu(op, dtype, case), f"plan {plan}")
    finally:
        qb.qk_set_plan_override(OPC[op], DT[dtype], None)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_xent_backward_bad_targets_and_default_dloss(dtype):
    case = make_case("xent", dtype, 8, 1024, seed=8000)
    case["targets"] = torch.tensor([-1, 1024, 0, 1023, 2 ** 40, 5, -(2 ** 63), 2 ** 63 - 1], dtype=torch.int64)
    d = {k: v.to(DEV) for k, v in case.items()}
    dx = torch.empty_like(d["x"])
    qb.qk_xent_bwd(d["x"], d["targets"], d["lse"], None, dx, 8, 1024, DT[dtype])  # dloss = 1
    torch.cuda.synchronize()
    case["dloss"] = torch.ones(8)
    check("xent", dtype, case, {"dx": dx}, "bad targets, dloss = 1")
    assert torch.isnan(dx[[0, 1, 4, 6, 7]]).all() and torch.isfinite(dx[[2, 3, 5]]).all()


@pytest.mark.parametrize("dtype,M,N", [("bf16", 4096, 4096), ("f32", 300, 16384), ("bf16", 2000, 1024)])
def test_rmsnorm_backward_graph_replays(dtype, M, N):
    """RMSNorm backward (the ring kernel and the fixed-order dw sum) captured
    into a CUDA graph and replayed with new data copied into the same buffers
    before each replay: every replay gives the oracle's dx and dw.  The
    workspace starts as random bytes (it is scratch)."""
    code = DT[dtype]
    cases = [make_case("rmsnorm", dtype, M, N, seed=9150 + i) for i in range(3)]
    d = {k: v.to(DEV) for k, v in cases[0].items()}
    dx = torch.empty_like(d["x"])
    dw = torch.empty((N,), dtype=torch.float32, device=DEV)
    nbytes = qb.qk_rmsnorm_bwd_workspace_size(M, N, code)
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # one eager call first: plan, attributes, occupancy
        qb.qk_rmsnorm_bwd(d["x"], d["w"], d["rstd"], d["dy"], dx, dw, ws, nbytes, M, N, code, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        qb.qk_rmsnorm_bwd(d["x"], d["w"], d["rstd"], d["dy"], dx, dw, ws, nbytes, M, N, code,
                          torch.cuda.current_stream())
    for i, case in enumerate(cases):
        for k in d:
            d[k].copy_(case[k].to(DEV))
        dx.fill_(float("nan"))
        dw.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert qb.qk_get_device_status() == qb.QK_OK
        check("rmsnorm", dtype, case, {"dx": dx, "dw": dw}, f"graph replay {i}")


def test_rmsnorm_backward_is_deterministic():
    case = make_case("rmsnorm", "bf16", 4096, 4096, seed=9000)
    a = run_gpu("rmsnorm", "bf16", case)
    b = run_gpu("rmsnorm", "bf16", case)
    assert torch.equal(a["dw"], b["dw"]) and torch.equal(a["dx"], b["dx"])
    check("rmsnorm", "bf16", case, a, "4096x4096")


@pytest.mark.parametrize("op,dtype,M,N", [("rmsnorm", "bf16", 16384, 4096), ("softmax", "f32", 1024, 4096),
                                          ("xent", "bf16", 1024, 131072)])
def test_backward_benchmark_shapes(op, dtype, M, N):
    """The forward workloads' shapes, checked on every row (oracle in a few seconds)."""
    case = make_case(op, dtype, M, N, seed=9100)
    check(op, dtype, case, run_gpu(op, dtype, case), f"{dtype} {M}x{N}")


# ---- masked path: rows whose length or start is not a multiple of 16 bytes ----

MASKED_N = [1, 3, 7, 101, 513, 571, 1143, 2047, 2049, 2295, 4605, 5001, 8191, 8193, 9207, 20001,
            131071]


@pytest.mark.parametrize("N", MASKED_N)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "xent"])
def test_backward_masked_shapes(op, dtype, N):
    """Ragged rows: softmax and cross-entropy on the shifted ring kernel, RMSNorm
    on the masked kernel (one row per CTA, per cluster of up to 16 CTAs beyond
    8192 elements, persistent over the rows)."""
    M = rows_for(N)
    # softmax and cross-entropy take the shifted ring kernel (path 6)
    assert qb.qk_get_plan(OPC[op], DT[dtype], M, N)["path"] == (5 if op == "rmsnorm" else 6)
    case = make_case(op, dtype, M, N, seed=9300 + N)
    check(op, dtype, case, run_gpu(op, dtype, case), f"masked {dtype} {M}x{N}")


@pytest.mark.parametrize("M,N", [(3000, 1001), (400, 20001), (1500, 5001)])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm"])
def test_backward_masked_many_rows_per_cta(op, M, N):
    """More rows than resident CTAs (clusters): every CTA walks several rows,
    reusing both reduction buffers and both phases of the cluster barrier,
    and RMSNorm's dw partials accumulate over the rows a CTA takes."""
    plan = qb.qk_get_plan(OPC[op], qb.QK_F32, M, N)
    assert plan["path"] == (5 if op == "rmsnorm" else 6) and plan["grid"] // plan["cluster"] < M
    case = make_case(op, "f32", M, N, seed=9400 + N)
    check(op, "f32", case, run_gpu(op, "f32", case), f"masked {M}x{N}")


def _offset(t):
    """A copy of t whose data starts one element past a 16-byte boundary."""
    store = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
    v = store[1:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "xent"])
def test_backward_unaligned_pointers(op, dtype):
    """Aligned N but inputs and outputs one element off a 16-byte boundary."""
    M, N = 9, 4096
    case = make_case(op, dtype, M, N, seed=9500)
    d = {k: v.to(DEV) for k, v in case.items()}
    code = DT[dtype]
    if op == "softmax":
        y, dy = _offset(d["y"]), _offset(d["dy"])
        dx = _offset(torch.full_like(d["y"], float("nan")))
        qb.qk_softmax_bwd(y, dy, dx, M, N, code)
        out = {"dx": dx}
    elif op == "rmsnorm":
        x, dy, w = _offset(d["x"]), _offset(d["dy"]), _offset(d["w"])
        dx = _offset(torch.full_like(d["x"], float("nan")))
        dw = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
        nbytes = qb.qk_rmsnorm_bwd_workspace_size(M, N, code)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV)
        qb.qk_rmsnorm_bwd(x, w, d["rstd"], dy, dx, dw, ws, nbytes, M, N, code)
        out = {"dx": dx, "dw": dw}
    else:
        x = _offset(d["x"])
        dx = _offset(torch.full_like(d["x"], float("nan")))
        qb.qk_xent_bwd(x, d["targets"], d["lse"], d["dloss"], dx, M, N, code)
        out = {"dx": dx}
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    check(op, dtype, case, out, "unaligned pointers")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "xent"])
def test_backward_masked_in_place(op, dtype):
    case = make_case(op, dtype, 13, 1001, seed=9600)
    check(op, dtype, case, run_gpu(op, dtype, case, inplace=True), "masked, in place")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_xent_backward_masked_bad_targets(dtype):
    N = 1001
    case = make_case("xent", dtype, 8, N, seed=9700)
    case["targets"] = torch.tensor([-1, N, 0, N - 1, 2 ** 40, 5, -(2 ** 63), 2 ** 63 - 1], dtype=torch.int64)
    d = {k: v.to(DEV) for k, v in case.items()}
    dx = torch.empty_like(d["x"])
    qb.qk_xent_bwd(d["x"], d["targets"], d["lse"], None, dx, 8, N, DT[dtype])  # dloss = 1
    torch.cuda.synchronize()
    case["dloss"] = torch.ones(8)
    check("xent", dtype, case, {"dx": dx}, "masked, bad targets, dloss = 1")
    assert torch.isnan(dx[[0, 1, 4, 6, 7]]).all() and torch.isfinite(dx[[2, 3, 5]]).all()


def test_masked_rows_beyond_the_limit_are_refused():
    N = 131073  # odd, so masked; beyond 16 clusters x 8192 elements
    for op, dtype in (("softmax", "bf16"), ("rmsnorm", "bf16")):
        case = make_case(op, dtype, 1, N, seed=9800)
        with pytest.raises(qb.QkError) as e:
            run_gpu(op, dtype, case)
        assert e.value.status == qb.QK_ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [4096, 50257])
def test_xent_backward_different_offsets(dtype, N):
    """dlogits not sharing the logits' alignment: the masked kernel."""
    M = 5
    case = make_case("xent", dtype, M, N, seed=9900 + N)
    d = {k: v.to(DEV) for k, v in case.items()}
    x = _offset(d["x"])
    store = torch.full((M * N + 16,), float("nan"), dtype=d["x"].dtype, device=DEV)
    dx = store[2:2 + M * N].view(M, N)
    qb.qk_xent_bwd(x, d["targets"], d["lse"], d["dloss"], dx, M, N, DT[dtype])
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    check("xent", dtype, case, {"dx": dx}, "different offsets")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [4096, 20001])
def test_softmax_backward_different_offsets(dtype, N):
    """dx not sharing the alignment of y and dy: the masked kernel."""
    M = 5
    case = make_case("softmax", dtype, M, N, seed=9950 + N)
    d = {k: v.to(DEV) for k, v in case.items()}
    y, dy = _offset(d["y"]), _offset(d["dy"])
    store = torch.full((M * N + 16,), float("nan"), dtype=d["y"].dtype, device=DEV)
    dx = store[2:2 + M * N].view(M, N)
    qb.qk_softmax_bwd(y, dy, dx, M, N, DT[dtype])
    torch.cuda.synchronize()
    assert qb.qk_get_device_status() == qb.QK_OK
    check("softmax", dtype, case, {"dx": dx}, "different offsets")
