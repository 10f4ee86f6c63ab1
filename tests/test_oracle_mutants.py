"""Plant plausible mistakes in a copy of the oracle and check the pins catch
every one.  The mutated copies are compiled into a temporary directory and
loaded beside the real oracle; nothing here touches a GPU or the CUDA path."""
import os

import pytest

import oracle
import oracle_pins

# (description, original text, planted mistake); each original must occur in
# oracle.c exactly once.
MUTANTS = [
    ("softmax: sign of the shift", "s += exp(xi[j] - m);\n\n        for (int64_t j = 0; j < N; ++j)\n            yi[j]",
     "s += exp(xi[j] + m);\n\n        for (int64_t j = 0; j < N; ++j)\n            yi[j]"),
    ("softmax: shift dropped from the sum", "s += exp(xi[j] - m);\n\n        for (int64_t j = 0; j < N; ++j)\n            yi[j]",
     "s += exp(xi[j]);\n\n        for (int64_t j = 0; j < N; ++j)\n            yi[j]"),
    ("softmax: multiply instead of divide", "yi[j] = exp(xi[j] - m) / s;", "yi[j] = exp(xi[j] - m) * s;"),
    ("softmax: min instead of max", "    double *yi = y + i * N;\n\n        double m = -INFINITY;\n        for (int64_t j = 0; j < N; ++j)\n            if (xi[j] > m)",
     "    double *yi = y + i * N;\n\n        double m = INFINITY;\n        for (int64_t j = 0; j < N; ++j)\n            if (xi[j] < m)"),
    ("softmax: transposed row stride", "const double *xi = x + i * N;\n        double *yi = y + i * N;\n\n        double m",
     "const double *xi = x + i * M;\n        double *yi = y + i * N;\n\n        double m"),
    ("softmax: no shift at all", "yi[j] = exp(xi[j] - m) / s;", "yi[j] = exp(xi[j]) / s;"),
    ("rmsnorm: divide by N-1", "sum_sq / (double)N", "sum_sq / (double)(N - 1)"),
    ("rmsnorm: eps outside the root", "1.0 / sqrt(ms + eps)", "1.0 / (sqrt(ms) + eps)"),
    ("rmsnorm: square dropped", "sum_sq += xi[j] * xi[j];", "sum_sq += xi[j];"),
    ("rmsnorm: weight indexed by row", "yi[j] = xi[j] * r * w[j];", "yi[j] = xi[j] * r * w[i];"),
    ("rmsnorm: weight dropped", "yi[j] = xi[j] * r * w[j];", "yi[j] = xi[j] * r;"),
    ("rmsnorm: rms instead of its reciprocal", "double r = 1.0 / sqrt(ms + eps);", "double r = sqrt(ms + eps);"),
    ("rmsnorm: eps times the mean", "1.0 / sqrt(ms + eps)", "1.0 / sqrt(ms * (1.0 + eps))"),
    ("xent: sign of the loss", "? l - xi[t] : NAN", "? xi[t] - l : NAN"),
    ("xent: max dropped from lse", "double l = m + log(s);\n        int64_t t = target[i];\n        loss[i]",
     "double l = log(s);\n        int64_t t = target[i];\n        loss[i]"),
    ("xent: target column off by one", "? l - xi[t] : NAN", "? l - xi[t > 0 ? t - 1 : t] : NAN"),
    ("xent: log2 instead of ln", "double l = m + log(s);\n        int64_t t = target[i];\n        loss[i]",
     "double l = m + log2(s);\n        int64_t t = target[i];\n        loss[i]"),
    ("xent: no range check", "(t >= 0 && t < N) ? l - xi[t] : NAN", "(t > -2 && t <= N) ? l - xi[t] : NAN"),
    ("softmax bwd: sign of the dot", "di[j] = yi[j] * (gi[j] - dot);", "di[j] = yi[j] * (gi[j] + dot);"),
    ("softmax bwd: y dropped from the dot", "dot += gi[j] * yi[j];", "dot += gi[j];"),
    ("softmax bwd: y factor dropped", "di[j] = yi[j] * (gi[j] - dot);", "di[j] = (gi[j] - dot);"),
    ("rmsnorm bwd: r squared for r cubed", "double c = r * r * r * dot / (double)N;", "double c = r * r * dot / (double)N;"),
    ("rmsnorm bwd: mean divisor dropped", "double c = r * r * r * dot / (double)N;", "double c = r * r * r * dot;"),
    ("rmsnorm bwd: w dropped from the dot", "dot += gi[j] * w[j] * xi[j];", "dot += gi[j] * xi[j];"),
    ("rmsnorm bwd: dw without rstd", "dw[j] += gi[j] * xi[j] * r;", "dw[j] += gi[j] * xi[j];"),
    ("rmsnorm bwd: sign of the correction", "di[j] = r * gi[j] * w[j] - xi[j] * c;", "di[j] = r * gi[j] * w[j] + xi[j] * c;"),
    ("xent bwd: one-hot added", "dloss[i] * (p - (j == t ? 1.0 : 0.0))", "dloss[i] * (p + (j == t ? 1.0 : 0.0))"),
    ("xent bwd: lse dropped", "double p = exp(xi[j] - lse[i]);\n            di[j] = ok",
     "double p = exp(xi[j]);\n            di[j] = ok"),
    ("xent bwd: upstream gradient dropped", "dloss[i] * (p - (j == t ? 1.0 : 0.0))", "(p - (j == t ? 1.0 : 0.0))"),
    ("xent ex: z-loss uses lse not lse^2", "l - xi[t] + z * l * l", "l - xi[t] + z * l"),
    ("xent ex: ignored rows counted in the mean", "            total += li;\n            counted += 1;\n        }",
     "            total += li;\n        }\n        counted += 1;"),
    ("xent ex bwd: z-loss gradient factor 1 + z lse", "(1.0 + 2.0 * z * lse[i])", "(1.0 + z * lse[i])"),
    ("xent ex bwd: ignored rows not zeroed", "            if (has_ignore && t == ignore_index) {\n                di[j] = 0.0;",
     "            if (has_ignore && t == ignore_index) {\n                di[j] = dloss[i];"),
    ("xent ex: the ignore index is a sentinel", "        if (has_ignore && t == ignore_index) {\n            li = 0.0;",
     "        if (t == ignore_index) {\n            li = 0.0;"),
    ("xent ex bwd: the ignore index is a sentinel", "            if (has_ignore && t == ignore_index) {\n                di[j] = 0.0;",
     "            if (t == ignore_index) {\n                di[j] = 0.0;"),
    ("layernorm: sample variance", "double var = sq / (double)N;", "double var = sq / (double)(N - 1);"),
    ("layernorm: mean not subtracted in the variance", "sq += (xi[j] - mu) * (xi[j] - mu);", "sq += xi[j] * xi[j];"),
    ("layernorm: eps outside the root", "double r = 1.0 / sqrt(var + eps);", "double r = 1.0 / (sqrt(var) + eps);"),
    ("layernorm: bias dropped", "* w[j] + (b ? b[j] : 0.0);", "* w[j];"),
    ("layernorm: mean not subtracted in y", "yi[j] = (xi[j] - mu) * r * w[j]", "yi[j] = xi[j] * r * w[j]"),
]


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("desc,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(desc, orig, bad, source, tmp_path):
    assert source.count(orig) == 1, f"mutation anchor not unique for {desc!r}"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(orig, bad))
    lib = oracle.bind(oracle.compile_library(str(src), str(tmp_path / f"mutant_{abs(hash(desc))}.so")))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except Exception as e:  # an assertion or any breakdown counts as detection
            caught.append(f"{pin.__name__}: {e}")
    assert caught, f"no pin detects the planted mistake: {desc}"
