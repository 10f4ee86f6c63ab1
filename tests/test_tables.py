"""Every plan the host tables can choose has a compiled kernel, for both
dtypes -- checked without a GPU, from the plan tables in qk_api.cu and the
kernel instantiations that the built libqk.so holds (its symbol table).  A
table entry without its kernel would only surface on a GPU, as
QK_ERR_UNSUPPORTED for the shapes that pick it."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
API = os.path.join(ROOT, "memory_bound_row_rmsnorm_gb300", "csrc", "qk_api.cu")
DTYPES = ("float", "__nv_bfloat16")
# template operator codes (qk_internal.h enum Op, qk_bwd_kernels.cuh enum BwdOp)
ROW_OPS = {"kRmsNormTable": 1, "kSoftmaxTable": 0, "kSoftmaxBf16Table": 0, "kXentTable": 2, "kLayerNormTable": 3,
           "kLayerNormF32Table": 3}
BWD_OPS = {"kSoftmaxBwdTable": 10, "kRmsNormBwdTable": 11, "kRmsNormBwdBf16Table": 11, "kXentBwdTable": 12}
SHIFT_OPS = {0: "softmax", 1: "rmsnorm", 2: "xent", 3: "layernorm", 4: "xent backward", 5: "softmax backward"}


@pytest.fixture(scope="module")
def kernels():
    if shutil.which("nm") is None:
        pytest.skip("nm is not available")
    from memory_bound_row_rmsnorm_gb300 import build
    lib = build.build()
    out = subprocess.run(["nm", "-C", lib], capture_output=True, text=True, check=True).stdout
    names = set()
    for m in re.finditer(r"qk::(\w+_kernel)<([^>]*)>\(qk::\w+\)", out):
        args = tuple(a.strip() for a in m.group(2).split(","))
        names.add((m.group(1),) + args)
    assert names, "no kernel symbols found in libqk.so"
    return names


def table(name):
    text = open(API).read()
    m = re.search(r"\b" + name + r"\[\]\s*=\s*\{(.*?)\n\};", text, re.S)
    assert m, name
    return [tuple(x.strip() for x in e.split(",")) for e in re.findall(r"\{([^{}]*)\}", m.group(1))]


def b(v):
    return "true" if v else "false"


@pytest.mark.parametrize("name", sorted(ROW_OPS))
def test_forward_tables(kernels, name):
    rows = table(name)
    assert rows
    for max_nv, th, tpr, vpt, cl, slots in rows:
        for dt in DTYPES:
            key = ("row_kernel", str(ROW_OPS[name]), dt, th, tpr, vpt, b(int(cl) > 1), "false")
            assert key in kernels, f"{name} entry {max_nv}: no {key}"


@pytest.mark.parametrize("name", sorted(BWD_OPS))
def test_backward_tables(kernels, name):
    rows = table(name)
    assert rows
    for max_nv, th, tpr, vpt, cl, slots in rows:
        for dt in DTYPES:
            key = ("bwd_kernel", str(BWD_OPS[name]), dt, th, tpr, vpt, b(int(cl) > 1))
            assert key in kernels, f"{name} entry {max_nv}: no {key}"


def launch_alternatives():
    text = open(API).read()
    m = re.search(r"\bkLaunchAlts\[\]\s*=\s*\{(.*?)\n\};", text, re.S)
    assert m, "kLaunchAlts"
    pat = r"\{(k\w+), (-1|QK_F32|QK_BF16), (\d+), (\d+), (\d+), ([^,]+), (\d+), \{([^{}]*)\}\}"
    return [(g[0], g[1], tuple(x.strip() for x in g[7].split(",")), (int(g[2]), int(g[3])), g[4], g[5])
            for g in re.findall(pat, m.group(1))]


def test_launch_alternatives(kernels):
    """The planner's alternative plans by launch length (kLaunchAlts) have
    their kernels too, for the dtypes each row applies to."""
    ops = {"kSoftmax": ("row_kernel", 0), "kRmsNorm": ("row_kernel", 1), "kXent": ("row_kernel", 2),
           "kOpLayerNorm": ("row_kernel", 3), "kOpSoftmaxBwd": ("bwd_kernel", 10), "kOpRmsNormBwd": ("bwd_kernel", 11),
           "kOpXentBwd": ("bwd_kernel", 12)}
    rows = launch_alternatives()
    assert len(rows) == open(API).read().split("kLaunchAlts[] = {", 1)[1].split("\n};", 1)[0].count("{k")
    for op, dt, (max_nv, th, tpr, vpt, cl, slots), _, _, _ in rows:
        kind, code = ops[op]
        for d in ({"QK_F32": ("float",), "QK_BF16": ("__nv_bfloat16",)}.get(dt, DTYPES)):
            key = (kind, str(code), d, th, tpr, vpt, b(int(cl) > 1))
            if kind == "row_kernel":
                key += ("false",)
            assert key in kernels, f"kLaunchAlts {op} {dt}: no {key}"


def test_launch_alternatives_do_not_overlap():
    """The planner takes the first row that matches; no two rows may match the
    same operator, dtype and row length, so the order of the rows decides
    nothing."""
    rows = launch_alternatives()
    assert rows
    big = 1 << 30
    win = lambda lo2, hi2: (int(lo2), big if hi2 == "kOpenEnd" else int(hi2))
    for i, (op, dt, _, (lo, hi), lo2, hi2) in enumerate(rows):
        assert lo < hi
        w = win(lo2, hi2)
        assert w[0] < w[1], (op, dt, lo2, hi2)
        for op_b, dt_b, _, (lo_b, hi_b), lo2_b, hi2_b in rows[i + 1:]:
            same_dt = dt == dt_b or "-1" in (dt, dt_b)
            wb = win(lo2_b, hi2_b)
            overlap = lo < hi_b and lo_b < hi and w[0] < wb[1] and wb[0] < w[1]
            assert not (op == op_b and same_dt and overlap), (op, dt, lo, hi, w, dt_b, lo_b, hi_b, wb)


def test_two_pass_kernels(kernels):
    """Rows beyond a cluster's capacity (softmax, RMSNorm, LayerNorm): 256 x 8
    two-pass kernels, alone and clustered."""
    for op in (0, 1, 3):
        for dt in DTYPES:
            for cl in ("false", "true"):
                assert ("row_kernel", str(op), dt, "256", "256", "8", cl, "true") in kernels


def test_shifted_table(kernels):
    """Unaligned rows: every row group of the shifted table for the operators
    that use it (LayerNorm and softmax backward skip the narrow 9-vector
    groups), and the clusters of 256 x 8 or 9 for the operators that split
    rows."""
    rows = table("kShiftTable")
    assert rows
    for op in SHIFT_OPS:
        narrow9 = op not in (3, 5)
        for th, tpr, vpt, slots in rows:
            if vpt == "9" and int(tpr) < 256 and not narrow9:
                continue
            for dt in DTYPES:
                key = ("shifted_kernel", str(op), dt, th, tpr, vpt, "false")
                assert key in kernels, f"{SHIFT_OPS[op]}: no {key}"
        if op in (0, 1, 3, 5):
            for vpt in ("8", "9"):
                for dt in DTYPES:
                    assert ("shifted_kernel", str(op), dt, "256", "256", vpt, "true") in kernels


def test_tables_are_ordered():
    """The planner takes the first entry that holds the row, so the forward and
    backward tables grow in max_nv and the shifted table in capacity."""
    for name in list(ROW_OPS) + list(BWD_OPS):
        caps = [int(r[0]) if r[0] != "kStream" else 1 << 62 for r in table(name)]
        assert caps == sorted(caps) and len(set(caps)) == len(caps), name
    caps = [int(r[1]) * int(r[2]) for r in table("kShiftTable")]
    assert caps == sorted(caps), caps
