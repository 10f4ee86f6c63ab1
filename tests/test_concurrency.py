"""Several host threads calling the library at once, each on its own CUDA
stream, with different operators and shapes (so that the per-thread plan
caches, the per-device lookups and the kernel attribute set-up all run
concurrently), then every result against the fp64 oracle."""
import threading

import pytest
import torch

from memory_bound_row_rmsnorm_gb300 import binding as qb
from memory_bound_row_rmsnorm_gb300 import synthetic as syn
from test_parity import DEV, DT_CODE, check_against_oracle

pytestmark = pytest.mark.gpu

CASES = [("softmax", "f32", 37, 4096), ("rmsnorm", "bf16", 64, 1003), ("xent", "bf16", 19, 50257),
         ("softmax", "bf16", 5, 65536), ("rmsnorm", "f32", 300, 256), ("xent", "f32", 41, 4096),
         ("softmax", "f32", 11, 3001), ("rmsnorm", "bf16", 3, 262144)]


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    qb.load_library()
    torch.cuda.set_device(0)
    yield


def _launch(op, dtype, d, out, stream):
    x = d["x"]
    M, N = x.shape
    code = DT_CODE[dtype]
    if op == "softmax":
        qb.qk_softmax_fwd(x, out["y"], M, N, code, stream)
    elif op == "rmsnorm":
        qb.qk_rmsnorm_fwd(x, d["w"], out["y"], out["rstd"], M, N, 1e-6, code, stream)
    else:
        qb.qk_xent_fwd(x, d["targets"], out["loss"], out["lse"], M, N, code, stream)


def test_threads_on_separate_streams():
    work = []
    for i, (op, dtype, M, N) in enumerate(CASES):
        inp = syn.make_inputs(op, dtype, M, N, 11000 + i, "cpu")
        d = {k: v.to(DEV) for k, v in inp.items()}
        if op == "xent":
            out = {"loss": torch.full((M,), float("nan"), device=DEV),
                   "lse": torch.full((M,), float("nan"), device=DEV)}
        else:
            out = {"y": torch.full_like(d["x"], float("nan"))}
            if op == "rmsnorm":
                out["rstd"] = torch.full((M,), float("nan"), device=DEV)
        work.append((op, dtype, inp, d, out, torch.cuda.Stream()))
    torch.cuda.synchronize()
    errors = []
    barrier = threading.Barrier(len(work))

    def worker(op, dtype, d, out, stream):
        try:
            torch.cuda.set_device(0)
            barrier.wait()
            for _ in range(20):  # the same call repeatedly: writes identical values
                _launch(op, dtype, d, out, stream)
        except Exception as e:  # reported on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(op, dt, d, out, s)) for op, dt, _, d, out, s in work]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert qb.qk_get_device_status() == qb.QK_OK
    for op, dtype, inp, d, out, _ in work:
        check_against_oracle(op, dtype, inp, out, what=f"threaded {op} {dtype} {tuple(d['x'].shape)}")
