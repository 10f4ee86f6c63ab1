"""Pins that tie the fp64 oracle to the operators' definitions.

Each ``pin_*`` function takes a loaded oracle library (``oracle.bind(path)``)
and raises AssertionError when the library disagrees with a fact fixed by the
mathematics: a hand-derived closed form, an invariant of the operator, or a
50-digit brute force written here independently of the C code.  They are run
against the real oracle (all must pass) and against deliberately broken copies
of it (each copy must fail at least one), so a plausible slip in the oracle --
a dropped term, a wrong sign, a wrong index, a transposed operand -- cannot
pass unnoticed.

The article (QbitAI on QuACK, section 让内存密集型内核达到“光速”) names the three
operators but prints no formula and no worked example; these checks therefore
follow the textbook definitions of softmax, RMSNorm and cross-entropy.
"""
from __future__ import annotations

import ast
import json
import math
import os
import decimal
from decimal import Decimal

import numpy as np

import oracle

_CTX = decimal.Context(prec=50)
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.json")


# --------------------------------------------------------------------------
# 50-digit evaluation of the closed-form expressions in the golden fixture
# --------------------------------------------------------------------------
def dec(expr: str) -> Decimal:
    """Evaluate an expression built from numbers, + - * /, ln(), sqrt(), exp()."""

    def ev(node):
        if isinstance(node, ast.Expression):
            return ev(node.body)
        if isinstance(node, ast.Constant) and isinstance(node.value, (int, float)):
            return Decimal(str(node.value))
        if isinstance(node, ast.UnaryOp) and isinstance(node.op, ast.USub):
            return -ev(node.operand)
        if isinstance(node, ast.BinOp):
            a, b = ev(node.left), ev(node.right)
            if isinstance(node.op, ast.Add):
                return _CTX.add(a, b)
            if isinstance(node.op, ast.Sub):
                return _CTX.subtract(a, b)
            if isinstance(node.op, ast.Mult):
                return _CTX.multiply(a, b)
            if isinstance(node.op, ast.Div):
                return _CTX.divide(a, b)
        if isinstance(node, ast.Call) and isinstance(node.func, ast.Name) and len(node.args) == 1:
            a = ev(node.args[0])
            fn = {"ln": _CTX.ln, "sqrt": _CTX.sqrt, "exp": _CTX.exp}.get(node.func.id)
            if fn is not None:
                return fn(a)
        raise ValueError(f"unsupported expression: {expr!r}")

    return ev(ast.parse(expr, mode="eval"))


def golden_cases(op: str):
    with open(GOLDEN) as f:
        return [c for c in json.load(f)["cases"] if c["op"] == op]


def _close(got, want, rel, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    err = np.abs(got - want)
    bound = rel * np.maximum(np.abs(want), 1e-300)
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: max rel err {float(np.max(err / np.maximum(np.abs(want), 1e-300)))} > {rel}"


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# Independent 50-digit brute force, unshifted, written from the definitions
# --------------------------------------------------------------------------
def brute_softmax(x):
    out = []
    for row in x:
        e = [_CTX.exp(Decimal(float(v))) for v in row]
        s = sum(e, Decimal(0))
        out.append([float(_CTX.divide(v, s)) for v in e])
    return np.array(out)


def brute_rmsnorm(x, w, eps):
    ys, rs = [], []
    for row in x:
        n = len(row)
        sq = sum((Decimal(float(v)) * Decimal(float(v)) for v in row), Decimal(0))
        r = _CTX.divide(Decimal(1), _CTX.sqrt(_CTX.divide(sq, Decimal(n)) + Decimal(float(eps))))
        ys.append([float(Decimal(float(v)) * r * Decimal(float(wj))) for v, wj in zip(row, w)])
        rs.append(float(r))
    return np.array(ys), np.array(rs)


def brute_xent(x, t):
    loss, lse = [], []
    for row, ti in zip(x, t):
        s = sum((_CTX.exp(Decimal(float(v))) for v in row), Decimal(0))
        l = _CTX.ln(s)
        lse.append(float(l))
        loss.append(float(l - Decimal(float(row[ti]))))
    return np.array(loss), np.array(lse)


# --------------------------------------------------------------------------
# Softmax pins
# --------------------------------------------------------------------------
def pin_softmax_golden(lib):
    for c in golden_cases("softmax"):
        x = np.array([[float(dec(e)) for e in r] for r in c["x"]])
        want = np.array([[float(dec(e)) for e in r] for r in c["y"]])
        _close(oracle.softmax_fwd(x, lib), want, c.get("rel", 1e-14), f"softmax golden {c['derivation']}")


def pin_softmax_rows_sum_to_one(lib):
    for seed, scale in [(1, 1.0), (2, 30.0)]:
        x = _rng(seed).normal(0.0, scale, size=(16, 37))
        y = oracle.softmax_fwd(x, lib)
        assert np.all(y >= 0), "softmax: negative probability"
        assert np.max(np.abs(y.sum(axis=1) - 1.0)) <= 1e-12, "softmax: row sum != 1"


def pin_softmax_shift_invariance(lib):
    x = _rng(3).normal(size=(8, 29))
    y0 = oracle.softmax_fwd(x, lib)
    for c in (-50.0, 3.25, 1.0e3):
        y1 = oracle.softmax_fwd(x + c, lib)
        assert np.max(np.abs(y1 - y0)) <= 1e-11, f"softmax: not shift invariant for c={c}"


def pin_softmax_constant_row(lib):
    for n, c in [(10, 7.5), (1, -3.0), (64, 0.0)]:
        y = oracle.softmax_fwd(np.full((2, n), c), lib)
        assert np.all(y == 1.0 / n), f"softmax: constant row of length {n} != 1/{n}"


def pin_softmax_two_columns(lib):
    x = _rng(4).normal(0, 3, size=(20, 2))
    y = oracle.softmax_fwd(x, lib)
    want = 1.0 / (1.0 + np.exp(x[:, 1] - x[:, 0]))
    _close(y[:, 0], want, 1e-14, "softmax: N=2 logistic closed form")


def pin_softmax_brute_force(lib):
    x = _rng(5).normal(0, 2, size=(4, 8))
    _close(oracle.softmax_fwd(x, lib), brute_softmax(x), 1e-14, "softmax: 4x8 brute force")


# --------------------------------------------------------------------------
# RMSNorm pins
# --------------------------------------------------------------------------
def pin_rmsnorm_golden(lib):
    for c in golden_cases("rmsnorm"):
        x = np.array([[float(dec(e)) for e in r] for r in c["x"]])
        w = np.array([float(dec(e)) for e in c["w"]])
        y, rstd = oracle.rmsnorm_fwd(x, w, float(dec(c["eps"])), lib)
        want_y = np.array([[float(dec(e)) for e in r] for r in c["y"]])
        want_r = np.array([float(dec(e)) for e in c["rstd"]])
        # exact zeros in the expected output must come out as exact zeros
        assert np.all((want_y == 0) == (y == 0)), f"rmsnorm golden zeros {c['derivation']}"
        nz = want_y != 0
        _close(y[nz], want_y[nz], 1e-14, f"rmsnorm golden y {c['derivation']}")
        _close(rstd, want_r, 1e-14, f"rmsnorm golden rstd {c['derivation']}")


def pin_rmsnorm_constant_row(lib):
    w = _rng(6).uniform(0.5, 1.5, size=12)
    for c in (2.5, -0.75, 1e-3):
        y, rstd = oracle.rmsnorm_fwd(np.full((3, 12), c), w, 0.0, lib)
        _close(y, np.sign(c) * np.broadcast_to(w, y.shape), 1e-15, f"rmsnorm: constant row {c}")
        _close(rstd, np.full(3, 1.0 / abs(c)), 1e-15, f"rmsnorm: constant row rstd {c}")
    # with eps > 0 the deviation from sign(c)*w stays within eps / (2 c^2)
    c, eps = 2.0, 1e-6
    y, _ = oracle.rmsnorm_fwd(np.full((1, 12), c), w, eps, lib)
    assert np.max(np.abs(y / w - 1.0)) <= eps / (2 * c * c) * 1.01, "rmsnorm: eps deviation bound"


def pin_rmsnorm_zero_row(lib):
    w = _rng(7).uniform(0.5, 1.5, size=9)
    eps = 1e-6
    y, rstd = oracle.rmsnorm_fwd(np.zeros((2, 9)), w, eps, lib)
    assert np.all(y == 0.0), "rmsnorm: zero row must map to zero"
    _close(rstd, np.full(2, eps ** -0.5), 1e-15, "rmsnorm: zero row rstd = eps^-1/2")


def pin_rmsnorm_scale_invariance(lib):
    rng = _rng(8)
    x = rng.normal(size=(5, 33))
    w = rng.uniform(0.5, 1.5, size=33)
    y0, r0 = oracle.rmsnorm_fwd(x, w, 0.0, lib)
    for a in (3.5, 1e-3):
        y1, r1 = oracle.rmsnorm_fwd(a * x, w, 0.0, lib)
        _close(y1, y0, 1e-13, f"rmsnorm: scale invariance alpha={a}")
        _close(r1 * a, r0, 1e-13, f"rmsnorm: rstd scales as 1/alpha, alpha={a}")


def pin_rmsnorm_normalised_energy(lib):
    rng = _rng(9)
    x = rng.normal(size=(6, 41))
    w = rng.uniform(0.5, 1.5, size=41)
    eps = 0.1
    y, _ = oracle.rmsnorm_fwd(x, w, eps, lib)
    ms = np.mean(x * x, axis=1)
    _close(np.mean((y / w) ** 2, axis=1), ms / (ms + eps), 1e-13, "rmsnorm: mean (y/w)^2 = ms/(ms+eps)")


def pin_rmsnorm_brute_force(lib):
    rng = _rng(10)
    x = rng.normal(size=(4, 8))
    w = rng.uniform(0.5, 1.5, size=8)
    y, r = oracle.rmsnorm_fwd(x, w, 1e-6, lib)
    by, br = brute_rmsnorm(x, w, 1e-6)
    _close(y, by, 1e-14, "rmsnorm: 4x8 brute force y")
    _close(r, br, 1e-14, "rmsnorm: 4x8 brute force rstd")


# --------------------------------------------------------------------------
# Cross-entropy pins
# --------------------------------------------------------------------------
def pin_xent_golden(lib):
    for c in golden_cases("xent"):
        x = np.array([[float(dec(e)) for e in r] for r in c["x"]])
        loss, lse = oracle.xent_fwd(x, np.array(c["target"], dtype=np.int64), lib)
        _close(loss, [float(dec(e)) for e in c["loss"]], 1e-14, f"xent golden loss {c['derivation']}")
        _close(lse, [float(dec(e)) for e in c["lse"]], 1e-14, f"xent golden lse {c['derivation']}")


def pin_xent_is_minus_log_softmax(lib):
    rng = _rng(11)
    x = rng.normal(0, 2 ** 0.5, size=(12, 50))
    t = rng.integers(0, 50, size=12)
    loss, _ = oracle.xent_fwd(x, t, lib)
    p = oracle.softmax_fwd(x, lib)[np.arange(12), t]
    _close(loss, -np.log(p), 1e-12, "xent: loss = -log softmax(x)[t]")


def pin_xent_constant_row(lib):
    for n, c in [(7, 0.0), (1000, -4.25)]:
        loss, lse = oracle.xent_fwd(np.full((2, n), c), np.array([0, n - 1]), lib)
        _close(loss, np.full(2, math.log(n)), 1e-14, f"xent: constant row loss = ln {n}")
        _close(lse, np.full(2, c + math.log(n)), 1e-14, f"xent: constant row lse = c + ln {n}")


def pin_xent_single_column(lib):
    x = np.array([[3.5], [-2.0]])
    loss, lse = oracle.xent_fwd(x, np.array([0, 0]), lib)
    assert np.all(loss == 0.0), "xent: N=1 loss must be 0"
    assert np.all(lse == x[:, 0]), "xent: N=1 lse must equal the logit"


def pin_xent_bounds(lib):
    rng = _rng(12)
    x = rng.normal(0, 3, size=(10, 64))
    loss, lse = oracle.xent_fwd(x, rng.integers(0, 64, size=10), lib)
    mx = x.max(axis=1)
    assert np.all(lse >= mx) and np.all(lse <= mx + math.log(64) + 1e-12), "xent: max <= lse <= max + ln N"
    assert np.all(loss >= 0), "xent: loss must be non-negative"


def pin_xent_out_of_range_target(lib):
    x = _rng(13).normal(size=(3, 6))
    loss, lse = oracle.xent_fwd(x, np.array([6, -1, 2]), lib)
    assert np.isnan(loss[0]) and np.isnan(loss[1]), "xent: out-of-range target must give NaN"
    assert np.isfinite(loss[2]) and np.all(np.isfinite(lse)), "xent: in-range rows stay finite"


def pin_xent_brute_force(lib):
    rng = _rng(14)
    x = rng.normal(0, 2 ** 0.5, size=(4, 8))
    t = rng.integers(0, 8, size=4)
    loss, lse = oracle.xent_fwd(x, t, lib)
    bl, bs = brute_xent(x, t)
    _close(lse, bs, 1e-14, "xent: 4x8 brute force lse")
    _close(loss, bl, 1e-13, "xent: 4x8 brute force loss")




# --------------------------------------------------------------------------
# Backward passes: pinned to finite differences of the (independently pinned)
# forward definitions, to invariants, closed forms and a 50-digit brute force.
# --------------------------------------------------------------------------
def _fd_grad(f, x, h=1e-6):
    """Central-difference gradient of the scalar function f at x."""
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


def pin_softmax_bwd_finite_differences(lib):
    rng = _rng(20)
    x = rng.normal(size=(3, 7))
    g = rng.normal(size=(3, 7))
    dx = oracle.softmax_bwd(oracle.softmax_fwd(x, lib), g, lib)
    fd = _fd_grad(lambda z: float(np.sum(g * oracle.softmax_fwd(z, lib))), x)
    assert np.max(np.abs(dx - fd)) <= 1e-7, "softmax bwd: not the derivative of softmax fwd"


def pin_softmax_bwd_invariants(lib):
    rng = _rng(21)
    y = oracle.softmax_fwd(rng.normal(size=(6, 33)), lib)
    dx = oracle.softmax_bwd(y, rng.normal(size=(6, 33)), lib)
    assert np.max(np.abs(dx.sum(axis=1))) <= 1e-14, "softmax bwd: rows must sum to 0"
    dx0 = oracle.softmax_bwd(y, np.full_like(y, 2.5), lib)
    assert np.max(np.abs(dx0)) <= 1e-15, "softmax bwd: a constant upstream gradient gives 0"


def pin_softmax_bwd_two_columns(lib):
    p = 0.3
    y = np.array([[p, 1 - p]])
    dx = oracle.softmax_bwd(y, np.array([[1.0, 0.0]]), lib)
    _close(dx, [[p * (1 - p), -p * (1 - p)]], 1e-14, "softmax bwd: N=2 closed form")


def pin_softmax_bwd_brute_force(lib):
    rng = _rng(22)
    x = rng.normal(size=(4, 8))
    g = rng.normal(size=(4, 8))
    y = oracle.softmax_fwd(x, lib)
    want = []
    for yr, gr in zip(y, g):
        yd = [Decimal(float(v)) for v in yr]
        gd = [Decimal(float(v)) for v in gr]
        dot = sum((a * b for a, b in zip(yd, gd)), Decimal(0))
        want.append([float(a * (b - dot)) for a, b in zip(yd, gd)])
    dx = oracle.softmax_bwd(y, g, lib)
    assert np.max(np.abs(dx - np.array(want))) <= 1e-15, "softmax bwd: 4x8 brute force"


def pin_rmsnorm_bwd_finite_differences(lib):
    rng = _rng(23)
    x = rng.normal(size=(3, 6))
    w = rng.uniform(0.5, 1.5, size=6)
    g = rng.normal(size=(3, 6))
    eps = 1e-3
    _, r = oracle.rmsnorm_fwd(x, w, eps, lib)
    dx, dw = oracle.rmsnorm_bwd(x, w, r, g, lib)
    fx = _fd_grad(lambda z: float(np.sum(g * oracle.rmsnorm_fwd(z, w, eps, lib)[0])), x)
    fw = _fd_grad(lambda v: float(np.sum(g * oracle.rmsnorm_fwd(x, v, eps, lib)[0])), w)
    assert np.max(np.abs(dx - fx)) <= 1e-7, "rmsnorm bwd: dx is not the derivative of the forward"
    assert np.max(np.abs(dw - fw)) <= 1e-7, "rmsnorm bwd: dw is not the derivative of the forward"


def pin_rmsnorm_bwd_invariants(lib):
    rng = _rng(24)
    x = rng.normal(size=(5, 40))
    w = rng.uniform(0.5, 1.5, size=40)
    g = rng.normal(size=(5, 40))
    y, r = oracle.rmsnorm_fwd(x, w, 0.0, lib)
    dx, dw = oracle.rmsnorm_bwd(x, w, r, g, lib)
    # eps = 0: y(a x) = y(x), so the gradient is orthogonal to x
    assert np.max(np.abs(np.sum(x * dx, axis=1))) <= 1e-12, "rmsnorm bwd: x . dx must vanish at eps=0"
    # dw_j = sum_i dy_ij y_ij / w_j
    _close(dw, np.sum(g * y, axis=0) / w, 1e-12, "rmsnorm bwd: dw = sum dy*y/w")
    # a single column at eps = 0 is a constant +-w: no gradient to x
    dx1, _ = oracle.rmsnorm_bwd(np.array([[1.7], [-0.4]]), np.array([0.9]),
                                np.array([1 / 1.7, 1 / 0.4]), np.array([[2.0], [3.0]]), lib)
    assert np.max(np.abs(dx1)) <= 1e-15, "rmsnorm bwd: N=1, eps=0 has zero dx"


def pin_rmsnorm_bwd_brute_force(lib):
    rng = _rng(25)
    x = rng.normal(size=(4, 8))
    w = rng.uniform(0.5, 1.5, size=8)
    g = rng.normal(size=(4, 8))
    _, r = oracle.rmsnorm_fwd(x, w, 1e-6, lib)
    want_dx, want_dw = [], [Decimal(0)] * 8
    for xr, gr, ri in zip(x, g, r):
        xd = [Decimal(float(v)) for v in xr]
        gd = [Decimal(float(v)) for v in gr]
        wd = [Decimal(float(v)) for v in w]
        rd = Decimal(float(ri))
        dot = sum((a * b * c for a, b, c in zip(gd, wd, xd)), Decimal(0))
        c = rd * rd * rd * dot / Decimal(8)
        want_dx.append([float(rd * a * b - xv * c) for a, b, xv in zip(gd, wd, xd)])
        want_dw = [acc + a * xv * rd for acc, a, xv in zip(want_dw, gd, xd)]
    dx, dw = oracle.rmsnorm_bwd(x, w, r, g, lib)
    _close(dx, want_dx, 1e-12, "rmsnorm bwd: 4x8 brute force dx")
    _close(dw, [float(v) for v in want_dw], 1e-13, "rmsnorm bwd: 4x8 brute force dw")


def pin_xent_bwd_finite_differences(lib):
    rng = _rng(26)
    x = rng.normal(0, 2 ** 0.5, size=(3, 7))
    t = np.array([0, 6, 3])
    g = rng.uniform(0.5, 2.0, size=3)
    _, lse = oracle.xent_fwd(x, t, lib)
    dx = oracle.xent_bwd(x, t, lse, g, lib)
    fd = _fd_grad(lambda z: float(np.sum(g * oracle.xent_fwd(z, t, lib)[0])), x)
    assert np.max(np.abs(dx - fd)) <= 1e-7, "xent bwd: not the derivative of the forward loss"


def pin_xent_bwd_closed_form_and_invariants(lib):
    x = np.array([[0.0, math.log(3.0)]])
    _, lse = oracle.xent_fwd(x, np.array([1]), lib)
    dx = oracle.xent_bwd(x, np.array([1]), lse, np.array([1.0]), lib)
    _close(dx, [[0.25, -0.25]], 1e-14, "xent bwd: softmax - onehot closed form")
    rng = _rng(27)
    x = rng.normal(size=(5, 19))
    t = rng.integers(0, 19, size=5)
    _, lse = oracle.xent_fwd(x, t, lib)
    dx = oracle.xent_bwd(x, t, lse, rng.uniform(0.1, 3, size=5), lib)
    assert np.max(np.abs(dx.sum(axis=1))) <= 1e-14, "xent bwd: rows must sum to 0"
    bad = oracle.xent_bwd(x[:2], np.array([19, -1]), lse[:2], np.ones(2), lib)
    assert np.isnan(bad).all(), "xent bwd: out-of-range target gives NaN gradients"


def pin_xent_bwd_brute_force(lib):
    rng = _rng(28)
    x = rng.normal(size=(4, 8))
    t = rng.integers(0, 8, size=4)
    g = rng.uniform(0.5, 2.0, size=4)
    _, lse = oracle.xent_fwd(x, t, lib)
    want = []
    for xr, ti, gi in zip(x, t, g):
        s = sum((_CTX.exp(Decimal(float(v))) for v in xr), Decimal(0))
        want.append([float(Decimal(float(gi)) * (_CTX.exp(Decimal(float(v))) / s - (1 if j == ti else 0)))
                     for j, v in enumerate(xr)])
    dx = oracle.xent_bwd(x, t, lse, g, lib)
    assert np.max(np.abs(dx - np.array(want))) <= 1e-14, "xent bwd: 4x8 brute force"




# --------------------------------------------------------------------------
# Cross-entropy variants: ignore index, z-loss, mean over rows
# --------------------------------------------------------------------------
def pin_xent_ex_closed_form(lib):
    x = np.array([[0.0, math.log(3.0)], [0.0, math.log(3.0)], [1.0, 2.0]])
    z = 0.5
    loss, lse, mean = oracle.xent_fwd_ex(x, np.array([1, -100, 0]), ignore_index=-100, z=z, lib=lib)
    l4 = math.log(4.0)
    lse2 = math.log(math.e + math.e ** 2)
    want = [math.log(4.0 / 3.0) + z * l4 * l4, 0.0, lse2 - 1.0 + z * lse2 * lse2]
    _close(loss, want, 1e-14, "xent ex: z-loss closed form and ignored row")
    assert abs(mean - (want[0] + want[2]) / 2) <= 1e-14 * abs(mean), "xent ex: mean excludes ignored rows"
    _close(lse, [l4, l4, lse2], 1e-14, "xent ex: lse written on every row")


def pin_xent_ex_reduces_to_plain(lib):
    rng = _rng(30)
    x = rng.normal(size=(6, 17))
    t = rng.integers(0, 17, size=6)
    loss0, lse0 = oracle.xent_fwd(x, t, lib)
    loss, lse, mean = oracle.xent_fwd_ex(x, t, lib=lib)  # no ignore index, z = 0
    _close(loss, loss0, 1e-15, "xent ex: z=0, no ignore index is the plain loss")
    assert abs(mean - np.mean(loss0)) <= 1e-14 * abs(mean), "xent ex: mean of every row"
    all_ignored = oracle.xent_fwd_ex(x, np.full(6, 7), ignore_index=7, lib=lib)[2]
    assert math.isnan(all_ignored), "xent ex: the mean of no rows is NaN"


def pin_xent_ex_no_sentinel_target(lib):
    """Without an ignore index no target value is special: the extreme int64
    targets are out of range and give NaN exactly as in the plain loss, and
    with that value as the ignore index the same row is ignored."""
    rng = _rng(32)
    x = rng.normal(size=(4, 9))
    t = np.array([-(2 ** 63), 3, 2 ** 63 - 1, 0], dtype=np.int64)
    loss0, lse0 = oracle.xent_fwd(x, t, lib)
    assert np.isnan(loss0[[0, 2]]).all() and np.isfinite(loss0[[1, 3]]).all(), "xent: extreme targets"
    loss, lse, _ = oracle.xent_fwd_ex(x, t, lib=lib)
    assert np.isnan(loss[[0, 2]]).all(), "xent ex: INT64_MIN / INT64_MAX targets are out of range"
    _close(loss[[1, 3]], loss0[[1, 3]], 1e-15, "xent ex: in-range rows beside extreme targets")
    g = np.ones(4)
    dx = oracle.xent_bwd_ex(x, t, lse, g, lib=lib)
    assert np.isnan(dx[[0, 2]]).all() and np.isfinite(dx[[1, 3]]).all(), "xent ex bwd: extreme targets"
    loss_i = oracle.xent_fwd_ex(x, t, ignore_index=-(2 ** 63), lib=lib)[0]
    assert loss_i[0] == 0.0 and np.isnan(loss_i[2]), "xent ex: INT64_MIN as the ignore index"
    dx_i = oracle.xent_bwd_ex(x, t, lse, g, ignore_index=-(2 ** 63), lib=lib)
    assert np.all(dx_i[0] == 0.0) and np.isnan(dx_i[2]).all(), "xent ex bwd: INT64_MIN as the ignore index"


def pin_xent_ex_bwd_finite_differences(lib):
    rng = _rng(31)
    x = rng.normal(0, 1.5, size=(4, 6))
    t = np.array([2, -1, 5, 0])
    g = rng.uniform(0.5, 2.0, size=4)
    z = 0.3
    _, lse, _ = oracle.xent_fwd_ex(x, t, ignore_index=-1, z=z, lib=lib)
    dx = oracle.xent_bwd_ex(x, t, lse, g, ignore_index=-1, z=z, lib=lib)
    fd = _fd_grad(lambda q: float(np.sum(g * oracle.xent_fwd_ex(q, t, -1, z, lib)[0])), x)
    assert np.max(np.abs(dx - fd)) <= 1e-7, "xent ex bwd: not the derivative of the forward"
    assert np.all(dx[1] == 0.0), "xent ex bwd: an ignored row has zero gradient"


# --------------------------------------------------------------------------
# LayerNorm
# --------------------------------------------------------------------------
def pin_layernorm_closed_form(lib):
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    w = np.array([1.0, 2.0, 0.5, -1.0])
    b = np.array([0.0, 1.0, -1.0, 0.25])
    y, mean, rstd = oracle.layernorm_fwd(x, w, b, 0.0, lib)
    r = 1.0 / math.sqrt(1.25)  # mean 2.5, population variance 1.25
    want = (np.array([-1.5, -0.5, 0.5, 1.5]) * r) * w + b
    _close(y, [want], 1e-14, "layernorm: (1,2,3,4) closed form")
    _close(mean, [2.5], 1e-15, "layernorm: mean")
    _close(rstd, [r], 1e-14, "layernorm: rstd with the population variance")


def pin_layernorm_constant_row_and_no_bias(lib):
    w = _rng(40).uniform(0.5, 1.5, size=9)
    b = _rng(41).normal(size=9)
    y, mean, rstd = oracle.layernorm_fwd(np.full((2, 9), -3.5), w, b, 1e-5, lib)
    assert np.all(y == b), "layernorm: a constant row maps to the bias"
    _close(rstd, [1e-5 ** -0.5] * 2, 1e-14, "layernorm: constant row rstd = eps^-1/2")
    y0, _, _ = oracle.layernorm_fwd(np.full((1, 9), 2.0), w, None, 1e-5, lib)
    assert np.all(y0 == 0.0), "layernorm: no bias means zero output on a constant row"


def pin_layernorm_invariances(lib):
    rng = _rng(42)
    x = rng.normal(size=(5, 31))
    w = rng.uniform(0.5, 1.5, size=31)
    b = rng.normal(size=31)
    y0, m0, r0 = oracle.layernorm_fwd(x, w, b, 0.0, lib)
    y1, m1, r1 = oracle.layernorm_fwd(3.0 * x + 7.25, w, b, 0.0, lib)
    _close(y1, y0, 1e-12, "layernorm: y(a x + c) = y(x) at eps=0")
    _close(m1, 3.0 * m0 + 7.25, 1e-13, "layernorm: mean is affine")
    _close(r1 * 3.0, r0, 1e-13, "layernorm: rstd scales as 1/a")
    z = (y0 - b) / w
    assert np.max(np.abs(z.mean(axis=1))) <= 1e-13, "layernorm: normalised rows have zero mean"
    _close(np.mean(z * z, axis=1), np.ones(5), 1e-13, "layernorm: normalised rows have unit variance")


def pin_layernorm_brute_force(lib):
    rng = _rng(43)
    x = rng.normal(2.0, 3.0, size=(4, 8))
    w = rng.uniform(0.5, 1.5, size=8)
    b = rng.normal(size=8)
    eps = 1e-3
    y, mean, rstd = oracle.layernorm_fwd(x, w, b, eps, lib)
    ys, ms, rs = [], [], []
    for row in x:
        d = [Decimal(float(v)) for v in row]
        mu = sum(d, Decimal(0)) / Decimal(8)
        var = sum(((v - mu) * (v - mu) for v in d), Decimal(0)) / Decimal(8)
        r = _CTX.divide(Decimal(1), _CTX.sqrt(var + Decimal(eps)))
        ys.append([float((v - mu) * r * Decimal(float(wj)) + Decimal(float(bj))) for v, wj, bj in zip(d, w, b)])
        ms.append(float(mu))
        rs.append(float(r))
    _close(y, ys, 1e-13, "layernorm: 4x8 brute force y")
    _close(mean, ms, 1e-14, "layernorm: 4x8 brute force mean")
    _close(rstd, rs, 1e-14, "layernorm: 4x8 brute force rstd")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
