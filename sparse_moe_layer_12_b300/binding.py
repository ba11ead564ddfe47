"""Thin Python binding of libmoe (include/moe.h): argument marshalling only.

Every function takes torch CUDA tensors, checks dtype / shape / device /
contiguity, allocates outputs with torch, and calls the C ABI with raw device
pointers and the current CUDA stream.  No arithmetic of the layer happens here:
if libmoe.so is missing the calls raise; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_BF16, MOE_FP8_E4M3, MOE_FP8_E4M3_POW2 = 0, 1, 2
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_ALIGNMENT",
          4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_DEVICE"}

# every symbol include/moe.h declares
EXPORTS = ["moe_workspace_bytes", "moe_route", "moe_permute", "moe_expert_ffn", "moe_combine",
           "moe_bias_update", "moe_forward", "moe_quantize_weights_fp8", "moe_get_device_status",
           "moe_debug_wait_timeout", "moe_status_string", "moe_version", "moe_expert_ffn_static",
           "moe_expert_ffn_gather", "moe_forward_gathers", "moe_backward_workspace_bytes", "moe_backward",
           "moe_get_static_device_status", "moe_ep_regroup", "moe_quantize_weights_fp8_pow2"]


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("E", ctypes.c_int), ("S", ctypes.c_int),
                ("k", ctypes.c_int), ("I", ctypes.c_int), ("dtype", ctypes.c_int), ("n_group", ctypes.c_int),
                ("topk_group", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_SIGS = {
    "moe_workspace_bytes": (_SZ, [ctypes.POINTER(Shape)]),
    "moe_route": (_I, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute": (_I, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_ffn": (_I, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_ffn_static": (_I, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_expert_ffn_gather": (_I, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_combine": (_I, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P]),
    "moe_bias_update": (_I, [ctypes.POINTER(Shape), _P, _P, _F, _P]),
    "moe_forward": (_I, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _P,
                         _SZ, _P]),
    "moe_quantize_weights_fp8": (_I, [_I, _I, _I, _P, _P, _P, _P]),
    "moe_quantize_weights_fp8_pow2": (_I, [_I, _I, _I, _P, _P, _P, _P]),
    "moe_forward_gathers": (_I, [ctypes.POINTER(Shape)]),
    "moe_backward_workspace_bytes": (_SZ, [ctypes.POINTER(Shape)]),
    "moe_backward": (_I, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_get_device_status": (_I, [_P, _P]),
    "moe_get_static_device_status": (_I, [_P]),
    "moe_ep_regroup": (_I, [_I, _I, _P, _I, _P, _P, _SZ, _P, _P, _I, _P, _I, _P, _P]),
    "moe_debug_wait_timeout": (_I, [_P, ctypes.c_uint, _P]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_version": (ctypes.c_char_p, []),
}

_lib = None

# bytes at the start of a forward workspace that must be zero before its first use
WS_CTRL_BYTES = 2048


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libmoe.so not built: {path} (run python -m sparse_moe_layer_12_b300.build)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn: str, code: int):
    if code != 0:
        raise MoEError(fn, code)


def _need(t: torch.Tensor, dtype, shape, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_shape(T, d, E, S, k, I, fp8=False, n_group=0, topk_group=0, pow2=False) -> Shape:
    """fp8: E4M3 expert GEMMs with FP32 1x128 / 128x128 scales; with pow2 as well, power-of-two
    scales applied by the block-scaled tensor-core MMA."""
    dtype = (MOE_FP8_E4M3_POW2 if pow2 else MOE_FP8_E4M3) if fp8 else MOE_BF16
    return Shape(T, d, E, S, k, I, dtype, n_group, topk_group)


def is_fp8(shape: Shape) -> bool:
    return shape.dtype in (MOE_FP8_E4M3, MOE_FP8_E4M3_POW2)


def forward_gathers(shape: Shape) -> bool:
    """True if moe_forward reads routed rows straight from x for this shape."""
    r = load().moe_forward_gathers(ctypes.byref(shape))
    if r < 0:
        raise MoEError("moe_forward_gathers", 1)
    return r == 1


def workspace_bytes(shape: Shape) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(shape)))


def alloc_workspace(shape: Shape, device="cuda") -> torch.Tensor:
    n = workspace_bytes(shape)
    if n == 0:
        raise ValueError("invalid shape")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:WS_CTRL_BYTES].zero_()  # the control block (status word, router load counters) starts clear
    return ws


def _act_dtype(shape: Shape):
    return torch.float8_e4m3fn if is_fp8(shape) else torch.bfloat16


def moe_route(shape: Shape, x, w_router, bias, logit_offset=None, ws=None):
    T, d, E, k = shape.T, shape.d, shape.E, shape.k
    _need(x, torch.bfloat16, (T, d), "x")
    _need(w_router, torch.bfloat16, (E, d), "w_router")
    _need(bias, torch.float32, (E,), "bias")
    if logit_offset is not None:
        _need(logit_offset, torch.float32, (E,), "logit_offset")
    ws = alloc_workspace(shape, x.device) if ws is None else ws
    idx = torch.empty(T, k, dtype=torch.int32, device=x.device)
    gate = torch.empty(T, k, dtype=torch.float32, device=x.device)
    counts = torch.empty(E, dtype=torch.int32, device=x.device)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=x.device)
    _check("moe_route", load().moe_route(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(bias),
                                         _ptr(logit_offset), _ptr(idx), _ptr(gate), _ptr(counts), _ptr(offsets),
                                         _ptr(ws), ws.numel(), _stream()))
    return idx, gate, counts, offsets


def moe_permute(shape: Shape, x, topk_idx, offsets, ws=None, rows=True, x_perm=None, x_perm_scale=None):
    """rows=False: only the permutation tables (x_perm and its scales are None).
    x_perm / x_perm_scale: optional preallocated outputs."""
    T, d, E, k = shape.T, shape.d, shape.E, shape.k
    fp8 = is_fp8(shape)
    _need(x, torch.bfloat16, (T, d), "x")
    _need(topk_idx, torch.int32, (T, k), "topk_idx")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    ws = alloc_workspace(shape, x.device) if ws is None else ws
    if not rows:
        x_perm = scale = None
    else:
        if x_perm is None:
            x_perm = torch.empty(T * k, d, dtype=_act_dtype(shape), device=x.device)
        _need(x_perm, _act_dtype(shape), (T * k, d), "x_perm")
        scale = x_perm_scale
        if fp8 and scale is None:
            scale = torch.empty(T * k, d // 128, dtype=torch.float32, device=x.device)
        if fp8:
            _need(scale, torch.float32, (T * k, d // 128), "x_perm_scale")
        else:
            scale = None
    perm_token = torch.empty(T * k, dtype=torch.int32, device=x.device)
    inv_pos = torch.empty(T, k, dtype=torch.int32, device=x.device)
    _check("moe_permute", load().moe_permute(ctypes.byref(shape), _ptr(x), _ptr(topk_idx), _ptr(offsets),
                                             _ptr(x_perm), _ptr(scale), _ptr(perm_token), _ptr(inv_pos), _ptr(ws),
                                             ws.numel(), _stream()))
    return x_perm, scale, perm_token, inv_pos


def moe_expert_ffn(shape: Shape, x_perm, x_perm_scale, x, offsets, w_gate_up, w_down, w_gu_scale=None,
                   w_down_scale=None, ws=None, y=None):
    T, d, E, S, k, I = shape.T, shape.d, shape.E, shape.S, shape.k, shape.I
    wdt = _act_dtype(shape)
    _need(x_perm, wdt, (T * k, d), "x_perm")
    _need(x, torch.bfloat16, (T, d), "x")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(w_gate_up, wdt, (E + S, 2 * I, d), "w_gate_up")
    _need(w_down, wdt, (E + S, d, I), "w_down")
    if is_fp8(shape):
        _need(x_perm_scale, torch.float32, (T * k, d // 128), "x_perm_scale")
        _need(w_gu_scale, torch.float32, (E + S, 2 * I // 128, d // 128), "w_gu_scale")
        _need(w_down_scale, torch.float32, (E + S, d // 128, I // 128), "w_down_scale")
    ws = alloc_workspace(shape, x.device) if ws is None else ws
    if y is None:
        y = torch.empty(T * k + S * T, d, dtype=torch.bfloat16, device=x.device)
    else:
        _need(y, torch.bfloat16, (T * k + S * T, d), "y")
    _check("moe_expert_ffn", load().moe_expert_ffn(
        ctypes.byref(shape), _ptr(x_perm), _ptr(x_perm_scale), _ptr(x), _ptr(offsets), _ptr(w_gate_up),
        _ptr(w_gu_scale), _ptr(w_down), _ptr(w_down_scale), _ptr(y), _ptr(ws), ws.numel(), _stream()))
    return y


def moe_expert_ffn_gather(shape: Shape, x, perm_token, offsets, w_gate_up, w_down, w_gu_scale=None,
                          w_down_scale=None, ws=None, y=None):
    """The expert FFN reading routed rows straight from x through perm_token."""
    T, d, E, S, k, I = shape.T, shape.d, shape.E, shape.S, shape.k, shape.I
    wdt = _act_dtype(shape)
    _need(x, torch.bfloat16, (T, d), "x")
    _need(perm_token, torch.int32, (T * k,), "perm_token")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(w_gate_up, wdt, (E + S, 2 * I, d), "w_gate_up")
    _need(w_down, wdt, (E + S, d, I), "w_down")
    if is_fp8(shape):
        _need(w_gu_scale, torch.float32, (E + S, 2 * I // 128, d // 128), "w_gu_scale")
        _need(w_down_scale, torch.float32, (E + S, d // 128, I // 128), "w_down_scale")
    ws = alloc_workspace(shape, x.device) if ws is None else ws
    if y is None:
        y = torch.empty(T * k + S * T, d, dtype=torch.bfloat16, device=x.device)
    else:
        _need(y, torch.bfloat16, (T * k + S * T, d), "y")
    _check("moe_expert_ffn_gather", load().moe_expert_ffn_gather(
        ctypes.byref(shape), _ptr(x), _ptr(perm_token), _ptr(offsets), _ptr(w_gate_up), _ptr(w_gu_scale),
        _ptr(w_down), _ptr(w_down_scale), _ptr(y), _ptr(ws), ws.numel(), _stream()))
    return y


def moe_expert_ffn_static(shape: Shape, x_perm, x_perm_scale, x, offsets, w_gate_up, w_down, w_gu_scale=None,
                          w_down_scale=None, y=None):
    """moe_expert_ffn without a workspace: the library's fixed scratch array is used
    (for callers that cannot allocate device memory; one call at a time)."""
    T, d, E, S, k, I = shape.T, shape.d, shape.E, shape.S, shape.k, shape.I
    wdt = _act_dtype(shape)
    _need(x_perm, wdt, (T * k, d), "x_perm")
    _need(x, torch.bfloat16, (T, d), "x")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(w_gate_up, wdt, (E + S, 2 * I, d), "w_gate_up")
    _need(w_down, wdt, (E + S, d, I), "w_down")
    if is_fp8(shape):
        _need(x_perm_scale, torch.float32, (T * k, d // 128), "x_perm_scale")
        _need(w_gu_scale, torch.float32, (E + S, 2 * I // 128, d // 128), "w_gu_scale")
        _need(w_down_scale, torch.float32, (E + S, d // 128, I // 128), "w_down_scale")
    if y is None:
        y = torch.empty(T * k + S * T, d, dtype=torch.bfloat16, device=x.device)
    else:
        _need(y, torch.bfloat16, (T * k + S * T, d), "y")
    _check("moe_expert_ffn_static", load().moe_expert_ffn_static(
        ctypes.byref(shape), _ptr(x_perm), _ptr(x_perm_scale), _ptr(x), _ptr(offsets), _ptr(w_gate_up),
        _ptr(w_gu_scale), _ptr(w_down), _ptr(w_down_scale), _ptr(y), _stream()))
    return y


def moe_combine(shape: Shape, y, topk_gate, inv_pos, out=None):
    T, d, S, k = shape.T, shape.d, shape.S, shape.k
    _need(y, torch.bfloat16, (T * k + S * T, d), "y")
    _need(topk_gate, torch.float32, (T, k), "topk_gate")
    _need(inv_pos, torch.int32, (T, k), "inv_pos")
    out = torch.empty(T, d, dtype=torch.bfloat16, device=y.device) if out is None else out
    _check("moe_combine", load().moe_combine(ctypes.byref(shape), _ptr(y), _ptr(topk_gate), _ptr(inv_pos),
                                             _ptr(out), _stream()))
    return out


def moe_bias_update(shape: Shape, counts, bias, gamma=0.001):
    _need(counts, torch.int32, (shape.E,), "counts")
    _need(bias, torch.float32, (shape.E,), "bias")
    _check("moe_bias_update", load().moe_bias_update(ctypes.byref(shape), _ptr(counts), _ptr(bias),
                                                     ctypes.c_float(gamma), _stream()))
    return bias


def moe_forward(shape: Shape, x, w_router, bias, w_gate_up, w_down, logit_offset=None, w_gu_scale=None,
                w_down_scale=None, gamma=0.001, update_bias=False, ws=None, out=None, routing_out=True):
    """Whole layer; returns (out, topk_idx, topk_gate, counts) (routing tensors None if routing_out=False)."""
    T, d, E, S, k, I = shape.T, shape.d, shape.E, shape.S, shape.k, shape.I
    wdt = _act_dtype(shape)
    _need(x, torch.bfloat16, (T, d), "x")
    _need(w_router, torch.bfloat16, (E, d), "w_router")
    _need(bias, torch.float32, (E,), "bias")
    _need(w_gate_up, wdt, (E + S, 2 * I, d), "w_gate_up")
    _need(w_down, wdt, (E + S, d, I), "w_down")
    if logit_offset is not None:
        _need(logit_offset, torch.float32, (E,), "logit_offset")
    if is_fp8(shape):
        _need(w_gu_scale, torch.float32, (E + S, 2 * I // 128, d // 128), "w_gu_scale")
        _need(w_down_scale, torch.float32, (E + S, d // 128, I // 128), "w_down_scale")
    ws = alloc_workspace(shape, x.device) if ws is None else ws
    out = torch.empty(T, d, dtype=torch.bfloat16, device=x.device) if out is None else out
    idx = gate = counts = None
    if routing_out:
        idx = torch.empty(T, k, dtype=torch.int32, device=x.device)
        gate = torch.empty(T, k, dtype=torch.float32, device=x.device)
        counts = torch.empty(E, dtype=torch.int32, device=x.device)
    _check("moe_forward", load().moe_forward(
        ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(logit_offset), _ptr(w_gate_up),
        _ptr(w_gu_scale), _ptr(w_down), _ptr(w_down_scale), _ptr(out), _ptr(idx), _ptr(gate), _ptr(counts),
        ctypes.c_float(gamma), 1 if update_bias else 0, _ptr(ws), ws.numel(), _stream()))
    return out, idx, gate, counts


def moe_quantize_weights_fp8(w, pow2=False):
    """bf16 [G, N, K] -> (E4M3 [G, N, K], f32 scales [G, N/128, K/128]); pow2: power-of-two scales."""
    if not (w.is_cuda and w.dtype == torch.bfloat16 and w.dim() == 3 and w.is_contiguous()):
        raise ValueError("w must be a contiguous CUDA bf16 tensor [G, N, K]")
    G, N, K = w.shape
    wq = torch.empty(G, N, K, dtype=torch.float8_e4m3fn, device=w.device)
    sc = torch.empty(G, N // 128, K // 128, dtype=torch.float32, device=w.device)
    name = "moe_quantize_weights_fp8_pow2" if pow2 else "moe_quantize_weights_fp8"
    _check(name, getattr(load(), name)(G, N, K, _ptr(w), _ptr(wq), _ptr(sc), _stream()))
    return wq, sc


def backward_workspace_bytes(shape: Shape) -> int:
    return int(load().moe_backward_workspace_bytes(ctypes.byref(shape)))


def alloc_backward_workspace(shape: Shape, device="cuda") -> torch.Tensor:
    n = backward_workspace_bytes(shape)
    if n == 0:
        raise ValueError("invalid shape")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def moe_backward(shape: Shape, x, w_router, w_gate_up, w_down, topk_idx, dout, logit_offset=None, ws=None,
                 out=None):
    """Gradients of the layer for the routing topk_idx: (dx bf16 [T, d], dw_router f32 [E, d],
    dw_gate_up bf16 [E+S, 2I, d], dw_down bf16 [E+S, d, I]).  `out` may hold those four tensors."""
    T, d, E, S, k, I = shape.T, shape.d, shape.E, shape.S, shape.k, shape.I
    _need(x, torch.bfloat16, (T, d), "x")
    _need(w_router, torch.bfloat16, (E, d), "w_router")
    _need(w_gate_up, torch.bfloat16, (E + S, 2 * I, d), "w_gate_up")
    _need(w_down, torch.bfloat16, (E + S, d, I), "w_down")
    _need(topk_idx, torch.int32, (T, k), "topk_idx")
    _need(dout, torch.bfloat16, (T, d), "dout")
    if logit_offset is not None:
        _need(logit_offset, torch.float32, (E,), "logit_offset")
    ws = alloc_backward_workspace(shape, x.device) if ws is None else ws
    if out is None:
        dev = x.device
        out = (torch.empty(T, d, dtype=torch.bfloat16, device=dev),
               torch.empty(E, d, dtype=torch.float32, device=dev),
               torch.empty(E + S, 2 * I, d, dtype=torch.bfloat16, device=dev),
               torch.empty(E + S, d, I, dtype=torch.bfloat16, device=dev))
    dx, dwr, dwgu, dwd = out
    _need(dx, torch.bfloat16, (T, d), "dx")
    _need(dwr, torch.float32, (E, d), "dw_router")
    _need(dwgu, torch.bfloat16, (E + S, 2 * I, d), "dw_gate_up")
    _need(dwd, torch.bfloat16, (E + S, d, I), "dw_down")
    _check("moe_backward", load().moe_backward(
        ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(logit_offset), _ptr(w_gate_up), _ptr(w_down),
        _ptr(topk_idx), _ptr(dout), _ptr(dx), _ptr(dwr), _ptr(dwgu), _ptr(dwd), _ptr(ws), ws.numel(), _stream()))
    return dx, dwr, dwgu, dwd


def moe_ep_regroup(recv_counts, src, to_local: bool, ws, src_scale=None, dst=None, dst_scale=None,
                   local_offsets=None):
    """Rows between source-major order (as received from the dispatch all-to-all) and
    local expert-major order.  recv_counts int32 [G, E_loc] (CUDA); src [rows, ...]
    (bf16 / E4M3 rows, row bytes a multiple of 16); src_scale f32 [rows, cols] or None.
    Returns (dst, dst_scale, local_offsets int32 [E_loc + 1])."""
    if not (recv_counts.is_cuda and recv_counts.dtype == torch.int32 and recv_counts.dim() == 2
            and recv_counts.is_contiguous()):
        raise ValueError("recv_counts must be a contiguous CUDA int32 tensor [G, E_loc]")
    G, E_loc = recv_counts.shape
    if not (src.is_cuda and src.is_contiguous() and src.dim() == 2):
        raise ValueError("src must be a contiguous CUDA tensor [rows, cols]")
    rows = src.shape[0]
    row_bytes = src.shape[1] * src.element_size()
    dst = torch.empty_like(src) if dst is None else dst
    _need(dst, src.dtype, tuple(src.shape), "dst")
    cols = 0
    if src_scale is not None:
        cols = src_scale.shape[1]
        _need(src_scale, torch.float32, (rows, cols), "src_scale")
        dst_scale = torch.empty_like(src_scale) if dst_scale is None else dst_scale
        _need(dst_scale, torch.float32, (rows, cols), "dst_scale")
    else:
        dst_scale = None
    if local_offsets is None:
        local_offsets = torch.empty(E_loc + 1, dtype=torch.int32, device=src.device)
    _need(local_offsets, torch.int32, (E_loc + 1,), "local_offsets")
    _check("moe_ep_regroup", load().moe_ep_regroup(
        G, E_loc, _ptr(recv_counts), rows, _ptr(src), _ptr(dst), row_bytes, _ptr(src_scale), _ptr(dst_scale), cols,
        _ptr(local_offsets), 1 if to_local else 0, _ptr(ws), _stream()))
    return dst, dst_scale, local_offsets


def moe_get_device_status(ws) -> int:
    return int(load().moe_get_device_status(_ptr(ws), _stream()))


def moe_get_static_device_status() -> int:
    """Reads and clears the status word of moe_expert_ffn_static's array on the current device."""
    return int(load().moe_get_static_device_status(_stream()))


def moe_debug_wait_timeout(ws, limit_us: int):
    _check("moe_debug_wait_timeout", load().moe_debug_wait_timeout(_ptr(ws), limit_us, _stream()))
