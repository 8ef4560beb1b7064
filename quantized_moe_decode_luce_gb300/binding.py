"""ctypes binding of libluce_moe (include/luce_moe.h), same names as the C ABI.

Argument marshalling only: each function checks that its tensors are CUDA,
contiguous and of the right dtype, passes ``data_ptr()`` values and the
current torch stream (or the one given), and raises :class:`LuceError` when
the library returns a status other than ``LUCE_OK``.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback: if the
library has not been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB as LIB_PATH

LUCE_OK = 0
LUCE_ERR_INVALID_ARG = 1
LUCE_ERR_UNSUPPORTED = 2
LUCE_ERR_CUDA = 3
LUCE_FAULT_BAD_ID = 0x1
LUCE_FAULT_TIMEOUT = 0x2
LUCE_FAULT_DESYNC = 0x4

_LIB = None


class LuceError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it was not built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run quantized_moe_decode_luce_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        sigs = {
            "luce_route_topk": [P, P, i32, i32, i32, P, P, P],
            "luce_quantize_q8_1": [P, i32, i32, P, P],
            "luce_moe_group": [P, i32, i32, i32, P, P, P, P],
            "luce_moe_glu_pair": [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f32, P, P, i32, P],
            "luce_moe_prep": [P, P, P, i32, i32, i32, i32, P, P, P, P, P, P, P],
            "luce_moe_layer": [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f32, P, P, P, P, P, P, P, P, P,
                               P, sz, P],
            "luce_moe_down_combine": [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, P, i32, P],
            "luce_argmax": [P, i32, i64, P, P, P, sz, P],
            "luce_argmax_noalloc": [P, i32, i64, P, P, P],
            "luce_argmax_shard": [P, i32, i64, i64, P, P, P, sz, P],
            "luce_argmax_pick": [P, P, i32, i32, P, P, P],
            "luce_rmsnorm_router": [P, P, f32, P, i32, i32, i32, P, P, P],
            "luce_add_rmsnorm_router": [P, P, P, P, f32, P, i32, i32, i32, P, P, P],
            "luce_ep_mask": [P, i64, i32, i32, P, P],
            "luce_add_f32": [P, P, P, i64, P],
            "luce_moe_glu_q4k": [P, P, P, P, P, P, i32, i32, i32, i32, i32, f32, P, P, P],
            "luce_moe_down_combine_q4k": [P, P, P, P, P, i32, i32, i32, i32, i32, P, P],
        }
        for name, args in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.luce_set_pdl.argtypes = [i32]
        L.luce_set_pdl.restype = ctypes.c_int
        L.luce_moe_layer_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.luce_moe_layer_workspace_bytes.restype = sz
        L.luce_argmax_workspace_bytes.argtypes = [i32, i64]
        L.luce_argmax_workspace_bytes.restype = sz
        L.luce_status_string.argtypes = [ctypes.c_int]
        L.luce_status_string.restype = ctypes.c_char_p
        L.luce_get_fault.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        L.luce_get_fault.restype = ctypes.c_int
        L.luce_version.argtypes = []
        L.luce_version.restype = ctypes.c_int
        _LIB = L
    return _LIB


def status_string(status: int) -> str:
    return lib().luce_status_string(int(status)).decode()


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t, dtype=None, name="tensor") -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _check(fn: str, status: int) -> None:
    if status != LUCE_OK:
        raise LuceError(fn, status)


u8, i32, f32 = torch.uint8, torch.int32, torch.float32


def luce_route_topk(logits, bias, k: int, ids, weights, stream=None) -> None:
    T, E = logits.shape
    _check("luce_route_topk", lib().luce_route_topk(
        _ptr(logits, f32, "logits"), _ptr(bias, f32, "bias"), T, E, k, _ptr(ids, i32, "ids"),
        _ptr(weights, f32, "weights"), _stream(stream)))


def luce_quantize_q8_1(x, xq, stream=None) -> None:
    T, K = x.shape
    _check("luce_quantize_q8_1", lib().luce_quantize_q8_1(
        _ptr(x, f32, "x"), T, K, _ptr(xq, u8, "xq"), _stream(stream)))


def luce_moe_group(ids, E: int, counts, offsets, routes, stream=None) -> None:
    T, k = ids.shape
    _check("luce_moe_group", lib().luce_moe_group(
        _ptr(ids, i32, "ids"), T, k, E, _ptr(counts, i32, "counts"), _ptr(offsets, i32, "offsets"),
        _ptr(routes, i32, "routes"), _stream(stream)))


def luce_moe_glu_pair(w_gate, w_up, ws_gate, ws_up, xq, offsets, routes, T: int, k: int, E: int, H: int, I: int,
                      clamp: float, h, hq, variant: int = 0, stream=None) -> None:
    _check("luce_moe_glu_pair", lib().luce_moe_glu_pair(
        _ptr(w_gate, u8, "w_gate"), _ptr(w_up, u8, "w_up"), _ptr(ws_gate, u8, "ws_gate"), _ptr(ws_up, u8, "ws_up"),
        _ptr(xq, u8, "xq"), _ptr(offsets, i32, "offsets"), _ptr(routes, i32, "routes"), T, k, E, H, I,
        float(clamp), _ptr(h, f32, "h"), _ptr(hq, u8, "hq"), variant, _stream(stream)))


def luce_moe_prep(logits, bias, x, k: int, ids, weights, xq, counts, offsets, routes, stream=None) -> None:
    T, E = logits.shape
    H = x.shape[1]
    _check("luce_moe_prep", lib().luce_moe_prep(
        _ptr(logits, f32, "logits"), _ptr(bias, f32, "bias"), _ptr(x, f32, "x"), T, E, k, H, _ptr(ids, i32, "ids"),
        _ptr(weights, f32, "weights"), _ptr(xq, u8, "xq"), _ptr(counts, i32, "counts"),
        _ptr(offsets, i32, "offsets"), _ptr(routes, i32, "routes"), _stream(stream)))


def luce_moe_layer_workspace_bytes(T: int, k: int, H: int, I: int) -> int:
    return int(lib().luce_moe_layer_workspace_bytes(T, k, H, I))


def luce_moe_layer(logits, bias, x, k: int, I: int, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, clamp: float,
                   ids, weights, xq, counts, offsets, routes, h, hq, out, workspace, stream=None) -> None:
    """The whole layer in one launch; `workspace` is a uint8 CUDA tensor of at
    least luce_moe_layer_workspace_bytes(T, k, H, I) bytes, all zero before
    the first call (the library keeps it consistent)."""
    T, E = logits.shape
    H = x.shape[1]
    if workspace is None:
        raise ValueError("workspace is required")
    _check("luce_moe_layer", lib().luce_moe_layer(
        _ptr(logits, f32, "logits"), _ptr(bias, f32, "bias"), _ptr(x, f32, "x"), _ptr(w_gate, u8, "w_gate"),
        _ptr(w_up, u8, "w_up"), _ptr(w_down, u8, "w_down"), _ptr(ws_gate, u8, "ws_gate"), _ptr(ws_up, u8, "ws_up"),
        _ptr(ws_down, u8, "ws_down"), T, E, k, H, I, float(clamp), _ptr(ids, i32, "ids"),
        _ptr(weights, f32, "weights"), _ptr(xq, u8, "xq"), _ptr(counts, i32, "counts"),
        _ptr(offsets, i32, "offsets"), _ptr(routes, i32, "routes"), _ptr(h, f32, "h"), _ptr(hq, u8, "hq"),
        _ptr(out, f32, "out"), _ptr(workspace, u8, "workspace"), workspace.numel(), _stream(stream)))


def luce_set_pdl(enable: bool) -> None:
    _check("luce_set_pdl", lib().luce_set_pdl(1 if enable else 0))


def luce_moe_down_combine(w_down, ws_down, hq, ids, weights, offsets, routes, T: int, k: int, E: int, H: int,
                          I: int, out, variant: int = 0, stream=None) -> None:
    _check("luce_moe_down_combine", lib().luce_moe_down_combine(
        _ptr(w_down, u8, "w_down"), _ptr(ws_down, u8, "ws_down"), _ptr(hq, u8, "hq"), _ptr(ids, i32, "ids"),
        _ptr(weights, f32, "weights"), _ptr(offsets, i32, "offsets"), _ptr(routes, i32, "routes"),
        T, k, E, H, I, _ptr(out, f32, "out"), variant, _stream(stream)))


def luce_argmax_workspace_bytes(R: int, V: int) -> int:
    return int(lib().luce_argmax_workspace_bytes(R, V))


def luce_argmax(logits, idx, val, workspace, stream=None) -> None:
    R, V = logits.shape
    _check("luce_argmax", lib().luce_argmax(
        _ptr(logits, f32, "logits"), R, V, _ptr(idx, i32, "idx"), _ptr(val, f32, "val"),
        _ptr(workspace, u8, "workspace"), workspace.numel() if workspace is not None else 0, _stream(stream)))


def luce_argmax_noalloc(logits, idx, val, stream=None) -> None:
    """The argmax with the library's own fixed scratch (no allocation)."""
    R, V = logits.shape
    _check("luce_argmax_noalloc", lib().luce_argmax_noalloc(
        _ptr(logits, f32, "logits"), R, V, _ptr(idx, i32, "idx"), _ptr(val, f32, "val"), _stream(stream)))


def luce_argmax_shard(logits, v0: int, idx, val, workspace, stream=None) -> None:
    """Argmax of a vocabulary shard whose column 0 is column v0 of the whole vocabulary."""
    R, Vs = logits.shape
    _check("luce_argmax_shard", lib().luce_argmax_shard(
        _ptr(logits, f32, "logits"), R, Vs, int(v0), _ptr(idx, i32, "idx"), _ptr(val, f32, "val"),
        _ptr(workspace, u8, "workspace"), workspace.numel() if workspace is not None else 0, _stream(stream)))


def luce_argmax_pick(vals, idxs, idx, val, stream=None) -> None:
    """vals [S, R] fp32, idxs [S, R] int32 (the shards' results) -> idx [R], val [R]."""
    S, R = vals.shape
    _check("luce_argmax_pick", lib().luce_argmax_pick(
        _ptr(vals, f32, "vals"), _ptr(idxs, i32, "idxs"), S, R, _ptr(idx, i32, "idx"), _ptr(val, f32, "val"),
        _stream(stream)))


def luce_rmsnorm_router(x, gamma, eps: float, w_router, xn, logits, stream=None) -> None:
    """x [T, H], gamma [H], w_router [E, H] (fp32) -> xn [T, H] (or None), logits [T, E]."""
    T, H = x.shape
    E = w_router.shape[0]
    _check("luce_rmsnorm_router", lib().luce_rmsnorm_router(
        _ptr(x, f32, "x"), _ptr(gamma, f32, "gamma"), float(eps), _ptr(w_router, f32, "w_router"), T, E, H,
        _ptr(xn, f32, "xn"), _ptr(logits, f32, "logits"), _stream(stream)))


def luce_add_rmsnorm_router(x, residual, x_sum, gamma, eps: float, w_router, xn, logits, stream=None) -> None:
    """x, residual [T, H] -> x_sum = x + residual (or None), then luce_rmsnorm_router of the sum."""
    T, H = x.shape
    if tuple(residual.shape) != (T, H):
        raise ValueError("residual must have x's shape")
    E = w_router.shape[0]
    _check("luce_add_rmsnorm_router", lib().luce_add_rmsnorm_router(
        _ptr(x, f32, "x"), _ptr(residual, f32, "residual"), _ptr(x_sum, f32, "x_sum"), _ptr(gamma, f32, "gamma"),
        float(eps), _ptr(w_router, f32, "w_router"), T, E, H, _ptr(xn, f32, "xn"), _ptr(logits, f32, "logits"),
        _stream(stream)))


def luce_ep_mask(ids, e0: int, e1: int, ids_out, stream=None) -> None:
    _check("luce_ep_mask", lib().luce_ep_mask(
        _ptr(ids, i32, "ids"), ids.numel(), int(e0), int(e1), _ptr(ids_out, i32, "ids_out"), _stream(stream)))


def luce_add_f32(a, b, out, stream=None) -> None:
    if a.numel() != b.numel() or a.numel() != out.numel():
        raise ValueError("a, b and out must have the same number of elements")
    _check("luce_add_f32", lib().luce_add_f32(
        _ptr(a, f32, "a"), _ptr(b, f32, "b"), _ptr(out, f32, "out"), a.numel(), _stream(stream)))


def luce_moe_glu_q4k(w_gate, w_up, ws_gate, ws_up, xq, ids, E: int, H: int, I: int, clamp: float, h, hq=None,
                     stream=None) -> None:
    """Q4_K gate/up pair + SwiGLU -> h, and its q8_1 blocks -> hq when given."""
    T, k = ids.shape
    _check("luce_moe_glu_q4k", lib().luce_moe_glu_q4k(
        _ptr(w_gate, u8, "w_gate"), _ptr(w_up, u8, "w_up"), _ptr(ws_gate, u8, "ws_gate"), _ptr(ws_up, u8, "ws_up"),
        _ptr(xq, u8, "xq"), _ptr(ids, i32, "ids"), T, k, E, H, I, float(clamp), _ptr(h, f32, "h"),
        _ptr(hq, u8, "hq"), _stream(stream)))


def luce_moe_down_combine_q4k(w_down, ws_down, hq, ids, weights, E: int, H: int, I: int, out, stream=None) -> None:
    """Q4_K down product + masked route-weighted combine -> out."""
    T, k = ids.shape
    _check("luce_moe_down_combine_q4k", lib().luce_moe_down_combine_q4k(
        _ptr(w_down, u8, "w_down"), _ptr(ws_down, u8, "ws_down"), _ptr(hq, u8, "hq"), _ptr(ids, i32, "ids"),
        _ptr(weights, f32, "weights"), T, k, E, H, I, _ptr(out, f32, "out"), _stream(stream)))


def luce_get_fault() -> int:
    bits = ctypes.c_uint(0)
    _check("luce_get_fault", lib().luce_get_fault(ctypes.byref(bits)))
    return int(bits.value)


def luce_version() -> int:
    return int(lib().luce_version())


__all__ = ["LuceError", "lib", "status_string", "luce_route_topk", "luce_quantize_q8_1", "luce_moe_group",
           "luce_moe_glu_pair", "luce_moe_prep", "luce_moe_layer", "luce_moe_layer_workspace_bytes", "luce_set_pdl",
           "luce_moe_down_combine", "luce_argmax", "luce_argmax_workspace_bytes", "luce_argmax_noalloc",
           "luce_argmax_shard", "luce_argmax_pick", "luce_rmsnorm_router", "luce_add_rmsnorm_router", "luce_ep_mask", "luce_add_f32",
           "luce_moe_glu_q4k", "luce_moe_down_combine_q4k",
           "luce_get_fault", "luce_version", "LUCE_OK", "LUCE_ERR_INVALID_ARG", "LUCE_ERR_UNSUPPORTED",
           "LUCE_ERR_CUDA", "LUCE_FAULT_BAD_ID", "LUCE_FAULT_TIMEOUT", "LUCE_FAULT_DESYNC"]
