"""Device-side failure path: a bounded wait that runs out reports
QK_ERR_TIMEOUT through the status word instead of hanging or faulting.

The test kernel waits on a shared-memory barrier that nothing completes, with
a 20 ms bound; the GPU stays usable and the status word is cleared on read."""
import time

import pytest
import torch

from memory_bound_row_rmsnorm_gb300 import binding as qb

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the gpu tests")
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    assert qb.qk_get_device_status() == qb.QK_OK
    t0 = time.perf_counter()
    qb.qk_test_wait_timeout(20_000_000)
    assert qb.qk_get_device_status() == qb.QK_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    # read-and-clear: the next read is clean, and the context still works
    assert qb.qk_get_device_status() == qb.QK_OK
    x = torch.randn(8, 256, device="cuda")
    y = qb.softmax_fwd(x)
    torch.cuda.synchronize()
    assert torch.allclose(y.sum(1), torch.ones(8, device="cuda"), atol=1e-5)
    assert qb.qk_get_device_status() == qb.QK_OK
