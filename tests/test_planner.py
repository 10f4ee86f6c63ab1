"""The launch planner's documented rules, read back through qk_get_plan on the
device (the occupancy answers come from the GPU), and the results of the
plans those rules pick against the oracle:
  * a one-chunk, unclustered launch of few items per resident CTA gets a
    deeper ring: RMSNorm and LayerNorm three slots below 8 items per CTA,
    softmax three below 4 and two below 8, the others three below 4 -- and
    never at the cost of a resident CTA, except below two items per resident
    CTA, where a third slot may cost up to a third of them;
  * fp32 softmax rows of 4096 switch to 128-thread CTAs of 8 vectors a thread
    below 8 items per resident CTA; cross-entropy rows of 512 vectors to two
    64-thread rows per CTA below 4;
  * a launch of fewer than two items per resident CTA gives every CTA the
    same number of items, except softmax, RMSNorm and LayerNorm CTAs of
    several rows, which keep the full grid;
  * cross-entropy rows of 512 vectors otherwise run one warp a row, 16
    vectors a lane; bf16 softmax rows of 8192 elements 128 x 8 vectors;
  * RMSNorm (softmax) rows of 512 vectors (bf16 4096, fp32 2048 elements)
    at 4-12 (bf16 4-10, fp32 4-8) items per resident CTA run four 64-thread
    rows per 256-thread CTA with three slots, fp32 softmax rows one
    256-thread row per CTA with two slots above that; RMSNorm rows of 2048
    vectors one 512-thread row per CTA with two slots from 10 on;
  * RMSNorm and softmax rows of 64 vectors run sixteen rows per CTA from 1.5
    items per resident CTA on, eight below; fp32 LayerNorm rows of 128 run
    sixteen rows per CTA from 2 to 16 items per resident CTA of the table's
    eight-row plan;
  * a one-chunk, unclustered backward launch of fewer than 8 items per
    resident CTA takes a ring of three slots if that costs no resident CTA,
    else two if that costs at most one per SM; the passes with two inputs
    per item (softmax, RMSNorm) keep the full grid."""
import pytest
import torch

import test_backward as tb
import test_layernorm as tl
from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
from test_parity import DEV, check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu

OP = {"softmax": qb.QK_OP_SOFTMAX, "rmsnorm": qb.QK_OP_RMSNORM, "xent": qb.QK_OP_XENT,
      "layernorm": qb.QK_OP_LAYERNORM, "softmax_bwd": qb.QK_OP_SOFTMAX_BWD,
      "rmsnorm_bwd": qb.QK_OP_RMSNORM_BWD, "xent_bwd": qb.QK_OP_XENT_BWD}
DT = {"f32": qb.QK_F32, "bf16": qb.QK_BF16}


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    qb.load_library()
    torch.cuda.set_device(0)


def plan(op, dtype, M, N):
    return qb.qk_get_plan(OP[op], DT[dtype], M, N)


def items(p, M):
    return -(-M // (p["threads"] // p["row_threads"]))


def resident(p):
    return p["ctas_per_sm"] * torch.cuda.get_device_properties(0).multi_processor_count


def table_resident(op, dtype, N, table_plan):
    """Resident CTAs of the table's own plan (threads, row_threads,
    vec_per_thread, slots), read back with that plan forced: the rules by
    launch length count items per resident CTA of it."""
    th, tpr, vpt, slots = table_plan
    forced = {"path": 3 if op.endswith("_bwd") else 1, "threads": th, "row_threads": tpr, "vec_per_thread": vpt,
              "cluster": 1, "slots": slots,
              "chunks": 0, "ctas_per_sm": 0, "grid": 0, "smem_bytes": 0}
    qb.qk_set_plan_override(OP[op], DT[dtype], forced)
    try:
        return resident(plan(op, dtype, 1 << 20, N))
    finally:
        qb.qk_set_plan_override(OP[op], DT[dtype], None)


@pytest.mark.parametrize("op,dtype,N", [("rmsnorm", "bf16", 1024), ("rmsnorm", "f32", 4096),
                                        ("layernorm", "f32", 2048), ("softmax", "bf16", 4096)])
def test_ring_depth_follows_items_per_cta(op, dtype, N):
    long_ = plan(op, dtype, 1 << 20, N)  # many items per CTA: the table's slots
    for M in (256, 1024, 4096, 16384, 65536):
        p = plan(op, dtype, M, N)
        ipc = items(p, M) / resident(long_)
        if ipc < 2:  # very short: three slots, at most a third of the CTAs lost
            assert p["slots"] >= 3 and 3 * p["ctas_per_sm"] >= 2 * long_["ctas_per_sm"], (M, p, long_)
            continue
        assert p["ctas_per_sm"] == long_["ctas_per_sm"], "a deeper ring never costs a resident CTA"
        ipc = items(p, M) / resident(p)
        t3, t2 = (8, 0) if op in ("rmsnorm", "layernorm") else (4, 8)
        if ipc < t3:  # three slots unless that would cost a resident CTA
            assert p["slots"] >= long_["slots"]
        if t3 <= ipc < t2:  # softmax: two slots (one more 8-16 KiB slot costs no CTA here)
            assert p["slots"] >= 2, (M, p)
        if ipc >= max(t3, t2):
            assert p["slots"] == long_["slots"], (M, p, long_)


def test_short_softmax_rows_of_4096_use_the_128_thread_kernel():
    short = plan("softmax", "f32", 1024, 4096)
    long_ = plan("softmax", "f32", 65536, 4096)
    assert (short["threads"], short["row_threads"], short["vec_per_thread"], short["slots"]) == (128, 128, 8, 3)
    assert (long_["threads"], long_["row_threads"], long_["vec_per_thread"], long_["slots"]) == (256, 256, 4, 1)
    mid = plan("softmax", "f32", 4096, 4096)
    assert (mid["threads"], mid["vec_per_thread"], mid["slots"]) == (128, 8, 2)


def test_short_launches_give_every_cta_the_same_items():
    p = plan("softmax", "f32", 1024, 4096)
    assert 1024 % p["grid"] == 0 and 1024 // p["grid"] == 2, p
    q = plan("softmax", "f32", 2048, 4096)  # three or more items per CTA: the full grid
    assert q["grid"] == resident(q), q
    r = plan("rmsnorm", "bf16", 16384, 256)  # CTAs of 32 rows: the full grid
    n = items(r, 16384)
    assert r["threads"] > r["row_threads"] and n < 2 * resident(r), r
    assert r["grid"] == min(n, resident(r)), r
    x = plan("xent", "bf16", 16384, 256)  # cross-entropy keeps even shares
    n = items(x, 16384)
    assert x["threads"] > x["row_threads"] and n < 2 * resident(x), x
    per = -(-n // min(n, resident(x)))
    assert x["grid"] == -(-n // per), x


def test_cross_entropy_rows_of_512_vectors():
    for dtype, N in (("bf16", 4096), ("f32", 2048)):
        p = plan("xent", dtype, 16384, N)
        assert (p["threads"], p["row_threads"], p["vec_per_thread"], p["slots"]) == (128, 32, 16, 2), p
        s = plan("xent", dtype, 2048, N)
        assert (s["threads"], s["row_threads"], s["vec_per_thread"]) == (128, 64, 8), s
    b = plan("softmax", "bf16", 16384, 8192)
    assert (b["threads"], b["row_threads"], b["vec_per_thread"]) == (128, 128, 8), b


@pytest.mark.parametrize("op,dtype,M,N", [("softmax", "f32", 1024, 4096), ("softmax", "f32", 4096, 4096),
                                          ("xent", "bf16", 2048, 4096), ("xent", "f32", 16384, 2048),
                                          ("rmsnorm", "bf16", 2000, 1024), ("softmax", "bf16", 3000, 8192)])
def test_the_chosen_plans_match_the_oracle(op, dtype, M, N):
    """Every row against the oracle, on ragged row counts where it matters."""
    inp = syn.make_inputs(op, dtype, M, N, 13000 + M, "cpu")
    out = run_gpu(op, {k: v.to(DEV) for k, v in inp.items()}, dtype)
    check_against_oracle(op, dtype, inp, out, what=f"planner {op} {dtype} {M}x{N}")


@pytest.mark.parametrize("op,dtype,N", [("softmax_bwd", "f32", 4096), ("softmax_bwd", "bf16", 4096),
                                        ("xent_bwd", "f32", 4096), ("xent_bwd", "bf16", 16384),
                                        ("rmsnorm_bwd", "f32", 4096)])
def test_backward_ring_depth_follows_items_per_cta(op, dtype, N):
    long_ = plan(op, dtype, 1 << 20, N)  # many items per CTA: the table's ring
    assert long_["cluster"] == 1 and long_["chunks"] == 1
    for M in (1024, 2048, 4096, 8192, 16384, 65536):
        p = plan(op, dtype, M, N)
        assert p["ctas_per_sm"] >= long_["ctas_per_sm"] - 1, "at most one resident CTA for the deeper ring"
        ipc = items(p, M) / (long_["ctas_per_sm"] * torch.cuda.get_device_properties(0).multi_processor_count)
        if ipc < 8:  # each of these shapes has a deeper ring within one CTA per SM
            assert p["slots"] > long_["slots"], (M, p, long_)
            if p["ctas_per_sm"] < long_["ctas_per_sm"]:
                assert p["slots"] == 2, (M, p, long_)
            n, units = items(p, M), min(items(p, M), resident(p))
            if op != "xent_bwd":  # two inputs per item: the full grid
                assert p["grid"] == units, p
            elif n < 2 * units:  # one input: every CTA the same number of items
                per = -(-n // units)
                assert p["grid"] == -(-n // per), p
        else:
            assert p["slots"] == long_["slots"] and p["ctas_per_sm"] == long_["ctas_per_sm"], (M, p, long_)


@pytest.mark.parametrize("op,dtype,M,N", [("softmax", "f32", 1024, 4096), ("softmax", "bf16", 2048, 4096),
                                          ("xent", "f32", 4096, 4096), ("xent", "bf16", 2048, 16384),
                                          ("rmsnorm", "f32", 2048, 4096)])
def test_the_chosen_backward_plans_match_the_oracle(op, dtype, M, N):
    """The deeper-ring backward plans, every row against the oracle."""
    p = plan(op + "_bwd", dtype, M, N)
    assert p["slots"] >= 2, p
    case = tb.make_case(op, dtype, M, N, 14000 + M)
    out = tb.run_gpu(op, dtype, case)
    tb.check(op, dtype, case, out, f"planner {op} bwd {dtype} {M}x{N}")


@pytest.mark.parametrize("op,dtype,M,N", [("xent", "f32", 1024, 4096), ("xent", "bf16", 2048, 4096),
                                          ("xent", "f32", 16384, 256), ("softmax", "f32", 2048, 2048)])
def test_very_short_forward_launches_take_three_slots(op, dtype, M, N):
    """Below two items per resident CTA a forward launch runs a ring of three
    slots; its results against the oracle on every row."""
    p = plan(op, dtype, M, N)
    assert p["slots"] == 3, p
    inp = syn.make_inputs(op, dtype, M, N, 15000 + M, "cpu")
    out = run_gpu(op, {k: v.to(DEV) for k, v in inp.items()}, dtype)
    check_against_oracle(op, dtype, inp, out, what=f"very short {op} {dtype} {M}x{N}")


@pytest.mark.parametrize("op,top,top_f32", [("rmsnorm", 12, 12), ("softmax", 10, 8)])
def test_rows_of_512_vectors(op, top, top_f32):
    """Between 4 and 12 (bf16 softmax 10, fp32 softmax 8) items per resident
    CTA of the table's 128-thread plan: 256-thread CTAs of four 64-thread
    rows, three slots; below it the table's plan; above it the table's plan
    too, except for fp32 softmax: one 256-thread row of 2 vectors a thread,
    two slots; the chosen plans against the oracle on every row."""
    for dtype, N in (("bf16", 4096), ("f32", 2048)):
        hi = top_f32 if dtype == "f32" else top
        long_alt = op == "softmax" and dtype == "f32"
        res = table_resident(op, dtype, N, (128, 128, 4, 1))
        for M in (2048, 4096, 6144, 8192, 10240, 12288, 14336, 16384, 32768, 1 << 20):
            p = plan(op, dtype, M, N)
            got = (p["threads"], p["row_threads"], p["vec_per_thread"])
            if 4 * res <= M < hi * res:
                assert got == (256, 64, 8) and p["slots"] == 3, (dtype, M, p, res)
            elif M >= hi * res and long_alt:
                assert got == (256, 256, 2) and p["slots"] == 2, (dtype, M, p, res)
            else:
                assert got == (128, 128, 4), (dtype, M, p, res)
    for dtype, M, N in (("bf16", 8192, 4096), ("f32", 10000, 2048), ("f32", 30000, 2048)):
        inp = syn.make_inputs(op, dtype, M, N, 16000 + M, "cpu")
        out = run_gpu(op, {k: v.to(DEV) for k, v in inp.items()}, dtype)
        check_against_oracle(op, dtype, inp, out, what=f"planner {op} {dtype} {M}x{N}")


@pytest.mark.parametrize("op,dtype,N", [("rmsnorm", "f32", 256), ("rmsnorm", "bf16", 512),
                                        ("softmax", "f32", 256), ("softmax", "bf16", 512)])
def test_short_rows_of_sixteen_row_ctas(op, dtype, N):
    """Rows of 64 vectors: the table's CTAs of sixteen 16-thread rows from 1.5
    items per resident CTA on, eight 32-thread rows below; three slots either
    way; the plans on both sides of the switch against the oracle on every
    row."""
    table = plan(op, dtype, 1 << 20, N)
    assert (table["threads"], table["row_threads"], table["vec_per_thread"]) == (256, 16, 4), table
    res = resident(table)
    for M in (1024, 4096, 8192, 12288, 16384, 32768, 65536):
        p = plan(op, dtype, M, N)
        got = (p["threads"], p["row_threads"], p["vec_per_thread"])
        assert got == ((256, 32, 2) if 2 * -(-M // 16) < 3 * res else (256, 16, 4)), (M, p, res)
        assert p["slots"] == 3, p
    edge = 24 * res  # 1.5 items per resident CTA of sixteen rows
    for M in (edge - 16 * 37 - 5, edge + 3):  # ragged: not a multiple of the rows per CTA
        inp = syn.make_inputs(op, dtype, M, N, 17000 + M, "cpu")
        out = run_gpu(op, {k: v.to(DEV) for k, v in inp.items()}, dtype)
        check_against_oracle(op, dtype, inp, out, what=f"short rows {op} {dtype} {M}x{N}")


def test_rmsnorm_rows_of_2048_vectors():
    """RMSNorm rows of 2048 vectors (fp32 8192, bf16 16384 elements) from 10
    items per resident CTA of the table's 256 x 8 plan on: one 512-thread row
    of 4 vectors a thread per CTA, two slots; the table's plan below; the
    plans on both sides against the oracle on every row."""
    for dtype, N in (("f32", 8192), ("bf16", 16384)):
        res = table_resident("rmsnorm", dtype, N, (256, 256, 8, 1))
        for M in (1024, 2048, 4096, 8192, 16384, 65536):
            p = plan("rmsnorm", dtype, M, N)
            got = (p["threads"], p["row_threads"], p["vec_per_thread"])
            if M >= 10 * res:
                assert got == (512, 512, 4) and p["slots"] == 2, (dtype, M, p, res)
            else:
                assert got == (256, 256, 8), (dtype, M, p, res)
        for M in (10 * res - 3, 10 * res + 5):
            inp = syn.make_inputs("rmsnorm", dtype, M, N, 19000 + M, "cpu")
            out = run_gpu("rmsnorm", {k: v.to(DEV) for k, v in inp.items()}, dtype)
            check_against_oracle("rmsnorm", dtype, inp, out, what=f"planner rmsnorm {dtype} {M}x{N}")


def test_rmsnorm_backward_f32_rows_of_512_vectors():
    """fp32 RMSNorm backward rows of 2048 elements from 32 items per resident
    CTA of the table's plan (one 128-thread row per CTA, four slots) on: two
    128-thread rows per 256-thread CTA, two slots; the plans on both sides
    against the oracle (dx and dw)."""
    res = table_resident("rmsnorm_bwd", "f32", 2048, (128, 128, 4, 4))
    for M in (1024, 4096, 8192, 16384, 65536):
        p = plan("rmsnorm_bwd", "f32", M, 2048)
        got = (p["threads"], p["row_threads"], p["vec_per_thread"])
        if M >= 32 * res:
            assert got == (256, 128, 4) and p["slots"] == 2, (M, p, res)
        else:
            assert got == (128, 128, 4), (M, p, res)
    for M in (32 * res - 1, 32 * res + 3):
        case = tb.make_case("rmsnorm", "f32", M, 2048, 19500 + M)
        tb.check("rmsnorm", "f32", case, tb.run_gpu("rmsnorm", "f32", case), f"planner rmsnorm bwd f32 {M}x2048")


@pytest.mark.parametrize("op,N,table_plan,long_plan,ipc", [
    ("softmax", 1024, (256, 64, 4, 2), (256, 128, 2, 2), 10),
    ("layernorm", 256, (256, 16, 4, 2), (256, 8, 8, 3), 3)])
def test_fp32_long_launch_rows(op, N, table_plan, long_plan, ipc):
    """fp32 softmax rows of 1024 elements and LayerNorm rows of 256: the long
    plan from `ipc` items per resident CTA of the table's plan on, the table's
    plan (or a short-launch rule) below; the plans on both sides against the
    oracle on every row."""
    res = table_resident(op, "f32", N, table_plan)
    rows = table_plan[0] // table_plan[1]
    edge = ipc * res * rows
    for M in (edge // 2, edge - rows, edge + rows, 2 * edge, 4 * edge):
        p = plan(op, "f32", M, N)
        got = (p["threads"], p["row_threads"], p["vec_per_thread"], p["slots"])
        if -(-M // rows) >= ipc * res:
            assert got == long_plan, (M, p, res)
        else:
            assert got[:3] != long_plan[:3], (M, p, res)
    for M in (edge - rows - 3, edge + 5):
        if op == "layernorm":
            tl.full_check("f32", M, N, 20000 + M, what=f"planner layernorm f32 {M}x{N}")
        else:
            inp = syn.make_inputs(op, "f32", M, N, 20000 + M, "cpu")
            out = run_gpu(op, {k: v.to(DEV) for k, v in inp.items()}, "f32")
            check_against_oracle(op, "f32", inp, out, what=f"planner {op} f32 {M}x{N}")


def test_layernorm_f32_rows_of_128_vectors():
    """fp32 LayerNorm rows of 512 elements: sixteen 16-thread rows of 8 vectors
    a thread per CTA, three slots, from 2 to 16 items per resident CTA of the
    table's eight-row plan; the table's plan outside."""
    table = plan("layernorm", "f32", 1 << 20, 512)
    assert (table["threads"], table["row_threads"], table["vec_per_thread"]) == (256, 32, 4), table
    res = resident(table)
    for M in (1024, 4096, 8192, 16384, 32768, 65536, 131072):
        p = plan("layernorm", "f32", M, 512)
        got = (p["threads"], p["row_threads"], p["vec_per_thread"])
        alt = 2 * res <= -(-M // 8) < 16 * res
        assert got == ((256, 16, 8) if alt else (256, 32, 4)), (M, p, res)
        if alt:
            assert p["slots"] == 3, p
    for M in (16 * res - 9, 16 * res + 5, 128 * res - 9):  # both sides of the lower edge, ragged
        tl.full_check("f32", M, 512, 18000 + M, what=f"planner layernorm f32 {M}x512")
