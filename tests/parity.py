"""Comparison rules between the CUDA path and the fp64 oracle.

Tolerances (fixed before any kernel was run):
  * fp32 outputs y: relative error <= 1e-5; softmax entries also pass with an
    absolute error <= 1e-7 (tiny probabilities).
  * bf16 outputs y: within one bf16 ulp of the fp64 value, where
    ulp(v) = 2^(floor(log2 |v|) - 7); an exact zero must come out as zero.
    The only bf16 softmax entries excused are those whose exact value lies
    below 2^-126, the smallest normal fp32: the kernels form exp in fp32,
    where such a value flushes to 0, so there 0 passes (an error <= 2^-126).
  * rstd, lse: fp32, relative error <= 1e-5.
  * loss: relative error <= 1e-5 against max(|loss|, 1e-3 |lse|), because
    loss = lse - x[t] can cancel.
NaN in the expected value must be NaN in the result and vice versa.
"""
from __future__ import annotations

import numpy as np
import torch

REL_F32 = 1e-5
ABS_SOFTMAX = 1e-7           # fp32 softmax entries only
FP32_MIN_NORMAL = 2.0 ** -126


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of an fp32/bf16 tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def bf16_ulp(ref: np.ndarray) -> np.ndarray:
    a = np.abs(ref)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)


def _nan_agree(got, ref, what):
    gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN pattern differs ({int((gn != rn).sum())} entries)"
    return ~rn


def check_rows(got: np.ndarray, ref: np.ndarray, dtype: str, softmax: bool, what: str) -> None:
    """Element-wise check of an output matrix against the oracle."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    ok_mask = _nan_agree(got, ref, what)
    g, r = got[ok_mask], ref[ok_mask]
    err = np.abs(g - r)
    if dtype == "f32":
        good = err <= REL_F32 * np.abs(r)
    else:
        ulp = bf16_ulp(r)
        good = np.where(r == 0, g == 0, err <= ulp)
    if softmax and dtype == "f32":
        good |= err <= ABS_SOFTMAX
    elif softmax:  # bf16: only where the exact value underflows fp32
        good |= (np.abs(r) < FP32_MIN_NORMAL) & (err <= FP32_MIN_NORMAL)
    if not good.all():
        idx = np.flatnonzero(~good)
        i = idx[np.argmax(err[idx] / np.maximum(np.abs(r[idx]), 1e-300))]
        raise AssertionError(
            f"{what}: {idx.size} of {good.size} outside tolerance; worst got {g[i]!r} "
            f"want {r[i]!r} (|err| {err[i]:.3e})")


def check_scalars(got, ref, what: str, denom=None) -> None:
    """Per-row fp32 scalars (rstd, lse, loss) against the oracle."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ok_mask = _nan_agree(got, ref, what)
    d = np.abs(ref) if denom is None else np.asarray(denom, dtype=np.float64)
    err = np.abs(got - ref)[ok_mask]
    bound = REL_F32 * d[ok_mask]
    bad = ~(err <= bound)
    if bad.any():
        i = np.flatnonzero(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} rows outside tolerance; first got "
                             f"{got[ok_mask][i]!r} want {ref[ok_mask][i]!r}")


def loss_denominator(loss_ref, lse_ref):
    return np.maximum(np.abs(loss_ref), 1e-3 * np.abs(lse_ref))


def check_scaled(got, ref, scale, dtype: str, what: str, rel: float = REL_F32) -> None:
    """Outputs that can cancel (gradients): |got - ref| <= rel * scale, where
    `scale` is the fp64 magnitude of the terms that form each element (so fp32
    rounding of the terms is what is bounded), plus one bf16 ulp of the value
    for bf16 outputs (the final rounding).  NaN must match NaN."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.broadcast_to(np.asarray(scale, dtype=np.float64), ref.shape)
    ok_mask = _nan_agree(got, ref, what)
    g, r, sc = got[ok_mask], ref[ok_mask], scale[ok_mask]
    bound = rel * sc + (bf16_ulp(r) if dtype == "bf16" else 0.0)
    err = np.abs(g - r)
    good = err <= bound
    if not good.all():
        idx = np.flatnonzero(~good)
        i = idx[np.argmax(err[idx] / np.maximum(bound[idx], 1e-300))]
        raise AssertionError(f"{what}: {idx.size} of {good.size} outside tolerance; worst got {g[i]!r} "
                             f"want {r[i]!r} (|err| {err[i]:.3e}, bound {bound[i]:.3e})")
