"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

Only random numbers live here -- none of the operators' arithmetic.  The
distributions follow the benchmark workloads: rows x ~ N(0, sigma^2) drawn in
fp32 and rounded once to the working dtype, RMSNorm weights w ~ U(0.5, 1.5),
cross-entropy targets uniform in [0, N).  LayerNorm rows are offset per row
(x_ij ~ N(s_i, sigma^2), s_i ~ U(-1, 1)) so that the mean it subtracts is
not zero, with w ~ U(0.5, 1.5) and b ~ U(-0.5, 0.5).  Every draw comes from a
torch.Generator seeded explicitly, on the device the tensor is made on.
"""
from __future__ import annotations

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}

# The named workloads: (op, dtype, M, N, sigma of the rows).
WORKLOADS = {
    "softmax_f32_1024x4096": ("softmax", "f32", 1024, 4096, 1.0),
    "rmsnorm_bf16_16384x4096": ("rmsnorm", "bf16", 16384, 4096, 1.0),
    "xent_bf16_8192x131072": ("xent", "bf16", 8192, 131072, 2.0 ** 0.5),  # N(0, 2): variance 2
    "softmax_f32_16384x131072": ("softmax", "f32", 16384, 131072, 1.0),
}
# Backward passes of the same workloads: (op, dtype, M, N, sigma).
BWD_WORKLOADS = {
    "softmax_bwd_f32_1024x4096": ("softmax_bwd", "f32", 1024, 4096, 1.0),
    "rmsnorm_bwd_bf16_16384x4096": ("rmsnorm_bwd", "bf16", 16384, 4096, 1.0),
    "xent_bwd_bf16_8192x131072": ("xent_bwd", "bf16", 8192, 131072, 2.0 ** 0.5),
    "softmax_bwd_f32_16384x131072": ("softmax_bwd", "f32", 16384, 131072, 1.0),
}
# Operators beyond the three the benchmark names: (op, dtype, M, N, sigma).
NEXT_WORKLOADS = {
    "layernorm_bf16_16384x4096": ("layernorm", "bf16", 16384, 4096, 1.0),
}
SWEEP_M = (8192, 16384, 32768)
SWEEP_N = (256, 1024, 4096, 16384, 65536, 262144)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_rows(M: int, N: int, dtype, seed: int, device="cpu", sigma: float = 1.0,
                row_block: int = 4096) -> torch.Tensor:
    """x ~ N(0, sigma^2), drawn in fp32 in blocks of rows, rounded to dtype."""
    dtype = DTYPES.get(dtype, dtype)
    g = _gen(seed, device)
    out = torch.empty((M, N), dtype=dtype, device=device)
    for r0 in range(0, M, row_block):
        r1 = min(M, r0 + row_block)
        blk = torch.randn((r1 - r0, N), generator=g, dtype=torch.float32, device=device)
        if sigma != 1.0:
            blk.mul_(sigma)
        out[r0:r1].copy_(blk)
    return out


def uniform_weight(N: int, dtype, seed: int, device="cpu", lo: float = 0.5, hi: float = 1.5) -> torch.Tensor:
    """RMSNorm weight w ~ U(lo, hi), drawn in fp32, rounded to dtype."""
    dtype = DTYPES.get(dtype, dtype)
    g = _gen(seed, device)
    w = torch.rand((N,), generator=g, dtype=torch.float32, device=device) * (hi - lo) + lo
    return w.to(dtype)


def offset_rows(M: int, N: int, dtype, seed: int, device="cpu", sigma: float = 1.0,
                lo: float = -1.0, hi: float = 1.0, row_block: int = 4096) -> torch.Tensor:
    """x_ij = s_i + sigma * z_ij with s_i ~ U(lo, hi) and z ~ N(0, 1), drawn
    in fp32 (the offsets first, then the rows block by block), rounded to dtype."""
    dtype = DTYPES.get(dtype, dtype)
    g = _gen(seed, device)
    s = torch.rand((M, 1), generator=g, dtype=torch.float32, device=device) * (hi - lo) + lo
    out = torch.empty((M, N), dtype=dtype, device=device)
    for r0 in range(0, M, row_block):
        r1 = min(M, r0 + row_block)
        blk = torch.randn((r1 - r0, N), generator=g, dtype=torch.float32, device=device)
        if sigma != 1.0:
            blk.mul_(sigma)
        out[r0:r1].copy_(blk + s[r0:r1])
    return out


def uniform_targets(M: int, N: int, seed: int, device="cpu") -> torch.Tensor:
    """Cross-entropy targets, int64 uniform in [0, N)."""
    g = _gen(seed, device)
    return torch.randint(0, N, (M,), generator=g, dtype=torch.int64, device=device)


def uniform_rows(M: int, N: int, dtype, seed: int, device="cpu", lo: float = 0.0, hi: float = 1.0,
                 row_block: int = 4096) -> torch.Tensor:
    """Rows ~ U(lo, hi), drawn in fp32 in blocks of rows, rounded to dtype."""
    dtype = DTYPES.get(dtype, dtype)
    g = _gen(seed, device)
    out = torch.empty((M, N), dtype=dtype, device=device)
    for r0 in range(0, M, row_block):
        r1 = min(M, r0 + row_block)
        blk = torch.rand((r1 - r0, N), generator=g, dtype=torch.float32, device=device)
        out[r0:r1].copy_(blk * (hi - lo) + lo)
    return out


def make_inputs(op: str, dtype, M: int, N: int, seed: int, device="cpu", sigma: float = 1.0) -> dict:
    """All inputs of one call of `op`: "softmax", "rmsnorm", "xent", "layernorm", or a
    backward pass ("softmax_bwd", "rmsnorm_bwd", "xent_bwd").  For the backward
    passes the saved forward quantities are stand-ins of the right range
    (probabilities in [0, 2/N), rstd in [0.5, 1.5], lse in [10, 14]); the
    tests build exact ones with the oracle instead."""
    if op == "softmax_bwd":
        return {"y": uniform_rows(M, N, dtype, seed, device, 0.0, 2.0 / N),
                "dy": normal_rows(M, N, dtype, seed + 1, device)}
    if op == "rmsnorm_bwd":
        return {"x": normal_rows(M, N, dtype, seed, device, sigma),
                "w": uniform_weight(N, dtype, seed + 1, device),
                "rstd": uniform_weight(M, "f32", seed + 2, device),
                "dy": normal_rows(M, N, dtype, seed + 3, device)}
    if op == "xent_bwd":
        return {"x": normal_rows(M, N, dtype, seed, device, sigma),
                "targets": uniform_targets(M, N, seed + 1, device),
                "lse": uniform_weight(M, "f32", seed + 2, device, lo=10.0, hi=14.0),
                "dloss": uniform_weight(M, "f32", seed + 3, device)}
    if op == "layernorm":
        return {"x": offset_rows(M, N, dtype, seed, device, sigma),
                "w": uniform_weight(N, dtype, seed + 1, device),
                "b": uniform_weight(N, dtype, seed + 2, device, lo=-0.5, hi=0.5)}
    x = normal_rows(M, N, dtype, seed, device, sigma)
    if op == "softmax":
        return {"x": x}
    if op == "rmsnorm":
        return {"x": x, "w": uniform_weight(N, dtype, seed + 1, device)}
    if op == "xent":
        return {"x": x, "targets": uniform_targets(M, N, seed + 2, device)}
    raise ValueError(op)
