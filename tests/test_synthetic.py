"""The seeded input generators, on CPU: the same seed gives the same bytes,
bf16 inputs are the fp32 draws rounded once, and the draws have the
distributions the workloads name (N(0, sigma^2) rows, w ~ U(0.5, 1.5),
targets uniform in [0, N), LayerNorm rows offset by s_i ~ U(-1, 1))."""
import math

import pytest
import torch

from memory_bound_row_rmsnorm_gb300 import synthetic as syn


@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "xent", "layernorm", "softmax_bwd", "rmsnorm_bwd",
                                "xent_bwd"])
def test_same_seed_same_bytes(op):
    a = syn.make_inputs(op, "bf16", 37, 300, 5, "cpu")
    b = syn.make_inputs(op, "bf16", 37, 300, 5, "cpu")
    c = syn.make_inputs(op, "bf16", 37, 300, 6, "cpu")
    assert a.keys() == b.keys()
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert any(not torch.equal(a[k], c[k]) for k in a)


def test_bf16_is_the_fp32_draw_rounded_once():
    x32 = syn.normal_rows(9000, 64, "f32", 11)  # more than one block of rows
    x16 = syn.normal_rows(9000, 64, "bf16", 11)
    assert torch.equal(x16, x32.to(torch.bfloat16))
    w32 = syn.uniform_weight(4096, "f32", 12)
    assert torch.equal(syn.uniform_weight(4096, "bf16", 12), w32.to(torch.bfloat16))


def test_distributions():
    M, N = 512, 2048
    x = syn.normal_rows(M, N, "f32", 21, sigma=2 ** 0.5).double()
    assert abs(x.mean().item()) < 0.01 and abs(x.var().item() - 2.0) < 0.02
    w = syn.uniform_weight(N, "f32", 22)
    assert w.min().item() >= 0.5 and w.max().item() <= 1.5 and abs(w.mean().item() - 1.0) < 0.03
    t = syn.uniform_targets(M * 8, N, 23)
    assert t.dtype == torch.int64 and t.min().item() >= 0 and t.max().item() < N
    assert abs(t.double().mean().item() - (N - 1) / 2) < 0.05 * N
    ln = syn.make_inputs("layernorm", "f32", M, N, 24, "cpu")
    rows = ln["x"].double()
    s = rows.mean(1)  # the row offsets s_i, up to N(0, 1/N) noise
    assert s.min().item() > -1.0 - 5 / math.sqrt(N) and s.max().item() < 1.0 + 5 / math.sqrt(N)
    assert s.std().item() > 0.4  # spread over U(-1, 1): std 0.577
    assert abs(rows.std(1).mean().item() - 1.0) < 0.02
    b = ln["b"]
    assert b.min().item() >= -0.5 and b.max().item() <= 0.5


def test_named_workloads():
    assert syn.WORKLOADS["rmsnorm_bf16_16384x4096"] == ("rmsnorm", "bf16", 16384, 4096, 1.0)
    op, dt, M, N, sigma = syn.WORKLOADS["xent_bf16_8192x131072"]
    assert (op, dt, M, N) == ("xent", "bf16", 8192, 131072) and sigma ** 2 == pytest.approx(2.0)
    assert syn.SWEEP_M == (8192, 16384, 32768)
    assert syn.SWEEP_N == (256, 1024, 4096, 16384, 65536, 262144)
