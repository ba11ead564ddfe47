"""CPU-only checks of the C ABI: the library loads, exports exactly what
include/moe.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from sparse_moe_layer_12_b300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert _declared() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(libmoe):
    for name in _declared():
        assert hasattr(libmoe, name), name
    assert libmoe.moe_version().decode().startswith("libmoe")


def test_status_strings(libmoe):
    for code, name in B.STATUS.items():
        assert libmoe.moe_status_string(code).decode() == name


def test_workspace_bytes(libmoe):
    s = B.make_shape(8192, 7168, 256, 1, 8, 2048)
    n = B.workspace_bytes(s)
    # x_perm + h + y dominate: (T*k*d + rows*I + rows*d) * 2 bytes
    rows = 8192 * 8 + 8192
    assert B.forward_gathers(s) is False
    assert n >= (8192 * 8 * 7168 + rows * 2048 + rows * 7168) * 2
    assert n < 1.01 * (8192 * 8 * 7168 + rows * 2048 + rows * 7168) * 2 + (1 << 24)
    # decode-sized batches gather routed rows inside the GEMM: no permuted copy
    small = B.make_shape(256, 7168, 256, 1, 8, 2048)
    assert B.forward_gathers(small) is True
    rows = 256 * 9
    assert B.workspace_bytes(small) < 1.01 * (rows * 2048 + rows * 7168) * 2 + (1 << 24)
    assert B.workspace_bytes(B.make_shape(8192, 7000, 256, 1, 8, 2048)) == 0  # d % 128
    assert B.workspace_bytes(B.make_shape(16, 256, 4, 1, 5, 128)) == 0  # k > E
    f8 = B.workspace_bytes(B.make_shape(8192, 7168, 256, 1, 8, 2048, fp8=True))
    assert f8 < n


@pytest.mark.parametrize("shape,code", [
    ((0, 256, 16, 1, 2, 128), 1),      # null pointers with a valid (empty) shape
    ((256, 200, 16, 1, 2, 128), 1),    # d % 128
    ((256, 256, 16, 1, 0, 128), 1),    # k = 0
    ((256, 256, 300, 1, 8, 128), 2),   # E > 256 unsupported
    ((256, 256, 16, 9, 2, 128), 2),    # S > 8 unsupported
    ((256, 256, 32, 1, 17, 128), 2),   # k > 16 unsupported
])
def test_route_rejects_before_launch(libmoe, shape, code):
    s = B.make_shape(*shape)
    st = libmoe.moe_route(ctypes.byref(s), None, None, None, None, None, None, None, None, None, 0, None)
    assert st == code


def test_alignment_and_workspace_are_checked(libmoe):
    s = B.make_shape(256, 256, 16, 1, 2, 128)
    p = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10002)
    args = [p, p, None, p, p, p, p]
    assert libmoe.moe_route(ctypes.byref(s), odd, p, p, None, p, p, p, p, p, 1 << 30, None) == 3
    assert libmoe.moe_route(ctypes.byref(s), p, p, p, None, p, p, p, p, None, 0, None) == 4
    assert libmoe.moe_route(ctypes.byref(s), p, p, p, None, p, p, p, p, p, 16, None) == 4
    assert libmoe.moe_bias_update(ctypes.byref(s), p, p, ctypes.c_float(-1.0), None) == 1
    assert libmoe.moe_quantize_weights_fp8(1, 100, 128, p, p, p, None) == 1
    assert libmoe.moe_debug_wait_timeout(p, 0, None) == 1
    assert len(args) == 7


def test_gather_entries_check_arguments(libmoe):
    s = B.make_shape(256, 256, 16, 1, 2, 128)
    p = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10002)
    # moe_expert_ffn_gather: null perm_token, misaligned x, missing workspace
    assert libmoe.moe_expert_ffn_gather(ctypes.byref(s), p, None, p, p, None, p, None, p, p, 1 << 30, None) == 1
    assert libmoe.moe_expert_ffn_gather(ctypes.byref(s), odd, p, p, p, None, p, None, p, p, 1 << 30, None) == 3
    assert libmoe.moe_expert_ffn_gather(ctypes.byref(s), p, p, p, p, None, p, None, p, None, 0, None) == 4
    f8 = B.make_shape(256, 256, 16, 1, 2, 128, fp8=True)
    assert libmoe.moe_expert_ffn_gather(ctypes.byref(f8), p, p, p, p, None, p, None, p, p, 1 << 30, None) == 1
    # moe_permute tables only: scales without rows are rejected
    assert libmoe.moe_permute(ctypes.byref(s), p, p, p, None, p, p, p, p, 1 << 30, None) == 1
    # dispatch form: gathers for decode-sized batches, copy for large ones, -1 for bad shapes
    assert libmoe.moe_forward_gathers(ctypes.byref(B.make_shape(512, 7168, 256, 1, 8, 2048))) == 1
    assert libmoe.moe_forward_gathers(ctypes.byref(B.make_shape(8192, 7168, 256, 1, 8, 2048))) == 0
    assert libmoe.moe_forward_gathers(ctypes.byref(B.make_shape(256, 200, 16, 1, 2, 128))) == -1
    assert libmoe.moe_forward_gathers(None) == -1


def test_backward_entries_check_arguments(libmoe):
    s = B.make_shape(256, 256, 16, 1, 2, 128)
    p = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10002)
    ws = ctypes.c_void_p(0x100000)
    big = 1 << 40
    n = libmoe.moe_backward_workspace_bytes(ctypes.byref(s))
    # the row buffers alone: x, dy, dx rows (d), [a u], [da du] (2I), h, dh (I) over >= T*k + S*T rows
    assert n >= 2 * (256 * 2 + 256) * (3 * 256 + 6 * 128)
    assert libmoe.moe_backward_workspace_bytes(ctypes.byref(B.make_shape(256, 200, 16, 1, 2, 128))) == 0
    args = [p, p, None] + [p] * 8  # x, w_router, logit_offset = NULL, w_gate_up, w_down ... dw_down
    # null input, misaligned dout, small or missing workspace, FP8 layer
    bad = list(args)
    bad[5] = None  # topk_idx
    assert libmoe.moe_backward(ctypes.byref(s), *bad, ws, big, None) == 1
    bad = list(args)
    bad[6] = odd  # dout
    assert libmoe.moe_backward(ctypes.byref(s), *bad, ws, big, None) == 3
    assert libmoe.moe_backward(ctypes.byref(s), *args, ws, n - 1, None) == 4
    assert libmoe.moe_backward(ctypes.byref(s), *args, None, big, None) == 4
    f8 = B.make_shape(256, 256, 16, 1, 2, 128, fp8=True)
    assert libmoe.moe_backward(ctypes.byref(f8), *args, ws, big, None) == 2


def test_empty_batch_accepts_null_token_buffers(libmoe):
    # T = 0: the token-sized pointers may be NULL (validation passes them and stops at the
    # missing workspace, before anything is launched); with T > 0 they are required
    p = ctypes.c_void_p(0x10000)
    e = B.make_shape(0, 256, 16, 1, 2, 128)
    t = B.make_shape(4, 256, 16, 1, 2, 128)
    assert libmoe.moe_route(ctypes.byref(e), None, p, p, None, None, None, p, p, None, 0, None) == 4
    assert libmoe.moe_route(ctypes.byref(t), None, p, p, None, None, None, p, p, None, 0, None) == 1
    assert libmoe.moe_forward(ctypes.byref(e), None, p, p, None, p, None, p, None, None, None, None, None,
                              ctypes.c_float(0.001), 1, None, 0, None) == 4
    assert libmoe.moe_backward(ctypes.byref(e), None, p, None, p, p, None, None, None, p, p, p, None, 0,
                               None) == 4
    assert libmoe.moe_backward(ctypes.byref(t), None, p, None, p, p, None, None, None, p, p, p, None, 0,
                               None) == 1
