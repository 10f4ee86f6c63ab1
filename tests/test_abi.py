"""The C ABI without a GPU: libqk.so loads, exports every entry point that
include/qk.h declares, and rejects bad arguments on the host before touching a
device.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

from memory_bound_row_rmsnorm_gb300 import binding as qb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qk.h")


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"QK_API\s+[\w\s\*]+?\b(qk_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def lib():
    from memory_bound_row_rmsnorm_gb300 import build
    build.build()
    return qb.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("qk_softmax_fwd", "qk_rmsnorm_fwd", "qk_xent_fwd", "qk_status_string",
                     "qk_get_device_status"):
        assert required in names
    assert sorted(names) == sorted(qb._EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libqk.so does not export {name}"


def test_status_strings(lib):
    for code in range(7):
        s = qb.qk_status_string(code)
        assert s and s != "unknown status"
    assert qb.qk_status_string(99) == "unknown status"


def test_max_row_elements(lib):
    assert qb.qk_max_row_elements(qb.QK_OP_SOFTMAX, qb.QK_F32) == 2 ** 63 - 1  # streamed twice
    assert qb.qk_max_row_elements(qb.QK_OP_RMSNORM, qb.QK_BF16) == 2 ** 63 - 1
    assert qb.qk_max_row_elements(qb.QK_OP_XENT, qb.QK_BF16) == 2 ** 63 - 1
    assert qb.qk_max_row_elements(7, qb.QK_F32) == 0
    assert qb.qk_max_row_elements(qb.QK_OP_SOFTMAX_BWD, qb.QK_F32) == 131072
    assert qb.qk_max_row_elements(qb.QK_OP_RMSNORM_BWD, qb.QK_BF16) == 262144
    assert qb.qk_max_row_elements(qb.QK_OP_XENT_BWD, qb.QK_F32) == 2 ** 63 - 1
    assert qb.qk_max_row_elements(qb.QK_OP_LAYERNORM, qb.QK_F32) == 2 ** 63 - 1  # streamed twice
    assert qb.qk_max_row_elements(qb.QK_OP_LAYERNORM, qb.QK_BF16) == 2 ** 63 - 1


# Fake, never-dereferenced device addresses: every call below must be refused
# by the host-side checks, which run before any CUDA call.
A = 1 << 32


@pytest.mark.parametrize("M,N,dtype,want", [
    (-1, 4, qb.QK_F32, qb.QK_ERR_INVALID_ARG),
    (4, 0, qb.QK_F32, qb.QK_ERR_INVALID_ARG),
    (4, -3, qb.QK_BF16, qb.QK_ERR_INVALID_ARG),
    (4, 4, 7, qb.QK_ERR_INVALID_ARG),
    (2 ** 40, 2 ** 40, qb.QK_F32, qb.QK_ERR_INVALID_ARG),
])
def test_softmax_size_errors(lib, M, N, dtype, want):
    assert lib.qk_softmax_fwd(A, A + (1 << 30), M, N, dtype, None) == want


def test_zero_rows_is_a_no_op(lib):
    assert lib.qk_softmax_fwd(None, None, 0, 4, qb.QK_F32, None) == qb.QK_OK
    assert lib.qk_rmsnorm_fwd(None, None, None, None, 0, 4, 1e-6, qb.QK_BF16, None) == qb.QK_OK
    assert lib.qk_xent_fwd(None, None, None, None, 0, 4, qb.QK_F32, None) == qb.QK_OK


def test_null_pointers(lib):
    assert lib.qk_softmax_fwd(None, A, 4, 4, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG
    assert lib.qk_rmsnorm_fwd(A, None, A + 4096, None, 4, 4, 1e-6, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG
    assert lib.qk_xent_fwd(A, None, A + 4096, None, 4, 4, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG
    assert lib.qk_xent_fwd(A, A + 4096, None, None, 4, 4, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG


def test_misaligned_pointers(lib):
    assert lib.qk_softmax_fwd(A + 2, A + 4096, 4, 4, qb.QK_F32, None) == qb.QK_ERR_MISALIGNED
    assert lib.qk_softmax_fwd(A + 1, A + 4096, 4, 4, qb.QK_BF16, None) == qb.QK_ERR_MISALIGNED
    assert lib.qk_rmsnorm_fwd(A, A + 8192, A + 4096, A + 2 + 16384, 4, 4, 1e-6, qb.QK_F32, None) \
        == qb.QK_ERR_MISALIGNED
    assert lib.qk_xent_fwd(A, A + 4 + 4096, A + 8192, None, 4, 4, qb.QK_F32, None) == qb.QK_ERR_MISALIGNED


def test_overlapping_buffers(lib):
    # partial overlap of x and y (exact aliasing would be allowed)
    assert lib.qk_softmax_fwd(A, A + 16, 4, 4, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG
    # y overlapping w, rstd overlapping x
    assert lib.qk_rmsnorm_fwd(A, A + 4096, A + 4096, None, 4, 4, 1e-6, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG
    assert lib.qk_rmsnorm_fwd(A, A + 4096, A + 8192, A + 32, 4, 4, 1e-6, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG
    # loss overlapping the logits, lse overlapping the targets
    assert lib.qk_xent_fwd(A, A + 4096, A + 8, None, 4, 4, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG
    assert lib.qk_xent_fwd(A, A + 4096, A + 8192, A + 4096, 4, 4, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG


@pytest.mark.parametrize("eps", [-1e-6, float("nan"), float("inf")])
def test_bad_eps(lib, eps):
    assert lib.qk_rmsnorm_fwd(A, A + 4096, A + 8192, None, 4, 4, eps, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG


def test_plan_override_validation(lib):
    bad = qb.qk_plan(threads=256, row_threads=96, vec_per_thread=4, cluster=1)
    assert lib.qk_set_plan_override(qb.QK_OP_SOFTMAX, qb.QK_F32, ctypes.byref(bad)) == qb.QK_ERR_UNSUPPORTED
    big = qb.qk_plan(threads=512, row_threads=512, vec_per_thread=8, cluster=32)
    assert lib.qk_set_plan_override(qb.QK_OP_SOFTMAX, qb.QK_F32, ctypes.byref(big)) == qb.QK_ERR_INVALID_ARG
    ok = qb.qk_plan(threads=256, row_threads=256, vec_per_thread=4, cluster=1)
    assert lib.qk_set_plan_override(qb.QK_OP_SOFTMAX, qb.QK_F32, ctypes.byref(ok)) == qb.QK_OK
    assert lib.qk_set_plan_override(qb.QK_OP_SOFTMAX, qb.QK_F32, None) == qb.QK_OK
    assert lib.qk_set_plan_override(qb.QK_OP_LAYERNORM, qb.QK_BF16, None) == qb.QK_OK
    assert lib.qk_set_plan_override(7, qb.QK_F32, None) == qb.QK_ERR_INVALID_ARG


def test_timeout_hook_argument_checks(lib):
    assert lib.qk_test_wait_timeout(0, None) == qb.QK_ERR_INVALID_ARG
    assert lib.qk_test_wait_timeout(20_000_000_000, None) == qb.QK_ERR_INVALID_ARG


def test_binding_raises_on_error(lib):
    with pytest.raises(qb.QkError) as e:
        qb.qk_softmax_fwd(A, A + 16, 4, 4, qb.QK_F32, 0)
    assert e.value.status == qb.QK_ERR_INVALID_ARG


def test_backward_argument_checks(lib):
    F, B = qb.QK_F32, qb.QK_BF16
    G = 1 << 30  # spacing of fake buffers that must not overlap
    # softmax backward: nulls, element alignment, partial overlap, row limits
    assert lib.qk_softmax_bwd(None, A, A + 8192, 4, 4, F, None) == qb.QK_ERR_INVALID_ARG
    assert lib.qk_softmax_bwd(A + 2, A + 4096, A + 8192, 4, 4, F, None) == qb.QK_ERR_MISALIGNED
    assert lib.qk_softmax_bwd(A, A + 4096, A + 16, 4, 4, F, None) == qb.QK_ERR_INVALID_ARG
    assert lib.qk_softmax_bwd(A, A + 4096, A + 8192, 4, 131076, F, None) == qb.QK_ERR_UNSUPPORTED
    assert lib.qk_softmax_bwd(A, A + G, A + 2 * G, 4, 262148, B, None) == qb.QK_ERR_UNSUPPORTED
    # the masked path (unaligned N) holds rows of up to 131,072 elements
    assert lib.qk_softmax_bwd(A, A + G, A + 2 * G, 4, 131073, B, None) == qb.QK_ERR_UNSUPPORTED
    assert lib.qk_softmax_bwd(None, None, None, 0, 4, F, None) == qb.QK_OK
    # RMSNorm backward: workspace is required; dw must not overlap an input
    args = [A, A + 4096, A + 8192, A + 12288, A + 16384, A + 20480, A + 24576, 1 << 20]
    assert lib.qk_rmsnorm_bwd(*args[:6], None, 0, 4, 8, B, None) == qb.QK_ERR_INVALID_ARG
    bad = list(args)
    bad[5] = A + 16  # dw inside x
    assert lib.qk_rmsnorm_bwd(*bad, 4, 8, B, None) == qb.QK_ERR_INVALID_ARG
    bad = list(args)
    bad[6] = A + 24576 + 4  # workspace not 16-byte aligned
    assert lib.qk_rmsnorm_bwd(*bad, 4, 8, B, None) == qb.QK_ERR_MISALIGNED
    far = [A, A + G, A + 2 * G, A + 3 * G, A + 4 * G, A + 5 * G, A + 6 * G, 1 << 20]
    assert lib.qk_rmsnorm_bwd(*far, 4, 131073, B, None) == qb.QK_ERR_UNSUPPORTED
    n = ctypes.c_size_t(123)
    assert lib.qk_rmsnorm_bwd_workspace_size(-1, 8, B, ctypes.byref(n)) == qb.QK_ERR_INVALID_ARG
    assert lib.qk_rmsnorm_bwd_workspace_size(0, 8, B, ctypes.byref(n)) == qb.QK_OK and n.value == 0
    assert lib.qk_rmsnorm_bwd_workspace_size(4, 8, B, None) == qb.QK_ERR_INVALID_ARG
    # cross-entropy backward: lse is required; dlogits must not overlap the targets
    assert lib.qk_xent_bwd(A, A + 4096, None, None, A + 8192, 4, 8, F, None) == qb.QK_ERR_INVALID_ARG
    assert lib.qk_xent_bwd(A, A + 4096, A + 4608, None, A + 4096, 4, 8, F, None) == qb.QK_ERR_INVALID_ARG


def test_layernorm_argument_checks(lib):
    F, B = qb.QK_F32, qb.QK_BF16
    ln = lib.qk_layernorm_fwd
    # x, w, b, y, mean, rstd, M, N, eps, dtype, stream
    ok = [A, A + 4096, A + 8192, A + 12288, A + 16384, A + 20480]
    assert ln(None, None, None, None, None, None, 0, 4, 1e-5, F, None) == qb.QK_OK  # M == 0
    assert ln(None, *ok[1:], 4, 4, 1e-5, F, None) == qb.QK_ERR_INVALID_ARG
    assert ln(ok[0], None, *ok[2:], 4, 4, 1e-5, F, None) == qb.QK_ERR_INVALID_ARG
    assert ln(*ok[:3], None, *ok[4:], 4, 4, 1e-5, F, None) == qb.QK_ERR_INVALID_ARG
    for eps in (-1.0, float("nan"), float("inf")):
        assert ln(*ok, 4, 4, eps, F, None) == qb.QK_ERR_INVALID_ARG
    assert ln(*ok, 4, 4, 1e-5, 5, None) == qb.QK_ERR_INVALID_ARG
    G = 1 << 30  # unaligned rows beyond the masked kernel's 524,288 elements
    far = [A, A + G, A + 2 * G, A + 3 * G, A + 4 * G, A + 5 * G]
    assert ln(*far, 4, 524289, 1e-5, B, None) == qb.QK_ERR_UNSUPPORTED
    assert ln(*far, 4, 524291, 1e-5, F, None) == qb.QK_ERR_UNSUPPORTED
    assert lib.qk_softmax_fwd(A, A + G, 4, 524289, B, None) == qb.QK_ERR_UNSUPPORTED
    for i, off in ((0, 2), (2, 1), (4, 2), (5, 1)):  # x, b, mean, rstd misaligned
        bad = list(ok)
        bad[i] += off
        assert ln(*bad, 4, 4, 1e-5, F, None) == qb.QK_ERR_MISALIGNED
    bad = list(ok)
    bad[3] = A + 8  # y partly over x
    assert ln(*bad, 4, 4, 1e-5, F, None) == qb.QK_ERR_INVALID_ARG
    bad = list(ok)
    bad[3] = A + 8192  # y over b
    assert ln(*bad, 4, 4, 1e-5, F, None) == qb.QK_ERR_INVALID_ARG
    bad = list(ok)
    bad[4] = A + 20480 + 8  # mean over rstd
    assert ln(*bad, 4, 4, 1e-5, F, None) == qb.QK_ERR_INVALID_ARG
    bad = list(ok)
    bad[5] = A + 4096  # rstd over w
    assert ln(*bad, 4, 4, 1e-5, F, None) == qb.QK_ERR_INVALID_ARG
