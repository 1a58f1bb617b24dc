"""Thin Python binding of the C ABI in ``include/moe_nvfp4.h``.

Argument marshalling only: every function here takes torch tensors (or None
for a NULL pointer) where the C call takes pointers, passes their device
addresses and the current CUDA stream, and raises ``MoeError`` on a status
other than MOE_OK. All arithmetic runs in the CUDA library; if the library
is missing the first call raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe_nvfp4.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA = 0, 1, 2, 3
MOE_ERR_WORKSPACE, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE = 4, 5, 6
MOE_W4A16, MOE_W4A4, MOE_MXFP4 = 0, 1, 2
MOE_SCALE_QUANT, MOE_SCALE_DEQUANT = 0, 1
MOE_DEBUG_WAIT_LIMIT, MOE_DEBUG_EXTRA_ARRIVALS, MOE_DEBUG_DISABLE_DECODE_FUSED, MOE_DEBUG_DECODE_STAGE_KB = 1, 2, 3, 4
MOE_DEBUG_FP4_TILE = 5
MOE_DEBUG_F16_TILE = 6

_lib = None


class MoeError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}"
                         + (f" ({last_cuda_error()})" if status == MOE_ERR_CUDA else ""))


class MoeLayerDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("I_shared", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("mode", ctypes.c_int),
                ("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w13_shared", ctypes.c_void_p), ("w2_shared", ctypes.c_void_p),
                ("w_router", ctypes.c_void_p),
                ("x_global_scale", ctypes.c_float), ("h_global_scale", ctypes.c_float),
                ("expert_offset", ctypes.c_int), ("local_experts", ctypes.c_int)]


class MoeGemmArgs(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("gate_up", ctypes.c_int), ("num_groups", ctypes.c_int),
                ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("weights", ctypes.c_void_p), ("last_weights", ctypes.c_void_p),
                ("group_offsets", ctypes.c_void_p), ("a", ctypes.c_void_p),
                ("a_sf", ctypes.c_void_p), ("a_gs", ctypes.c_void_p),
                ("a_row_index", ctypes.c_void_p), ("row_scale", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("out_amax", ctypes.c_void_p), ("rows", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_last_cuda_error": (ctypes.c_char_p, []),
    "moe_route_topk": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_router_gemm": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "moe_nvfp4_quantize_static": (_I, [_P, _I, _I, ctypes.c_float, _P, _P, _P]),
    "moe_mxfp4_quantize": (_I, [_P, _I, _I, _P, _P, _P]),
    "moe_import_global_scale": (_I, [ctypes.c_float, _I, ctypes.POINTER(ctypes.c_float)]),
    "moe_nvfp4_fold_scales": (_I, [_P, _Z, ctypes.c_float, _P, _P]),
    "moe_permute_workspace_size": (_Z, [_I, _I, _I]),
    "moe_permute": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_quantize_workspace_size": (_Z, []),
    "moe_nvfp4_quantize": (_I, [_P, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_prepare_size": (_Z, [_I, _I, _I, _I]),
    "moe_nvfp4_prepare_weights": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_gemm_workspace_size": (_Z, [_I]),
    "moe_gemm_workspace_size_rows": (_Z, [_I, _I, _I]),
    "moe_nvfp4_grouped_gemm": (_I, [ctypes.POINTER(MoeGemmArgs), _P, _Z, _P]),
    "moe_swiglu": (_I, [_P, _I, _I, _P, _P]),
    "moe_combine": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_workspace_size": (_Z, [ctypes.POINTER(MoeLayerDesc)]),
    "moe_nvfp4_forward": (_I, [ctypes.POINTER(MoeLayerDesc), _P, _P, _P, _P, _P, _Z, _P]),
    "moe_get_device_status": (_I, [_P, _P]),
    "moe_set_stage_events": (_I, [ctypes.POINTER(ctypes.c_void_p), _I]),
    "moe_kernel_launches": (ctypes.c_ulonglong, []),
    "moe_permute_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "moe_debug_set": (_I, [_I, ctypes.c_longlong]),
}

MOE_STAGE_COUNT = 8
STAGES = ["route", "permute", "quantize_x", "gemm1_gate_up_swiglu", "quantize_h", "gemm2_down",
          "combine"]


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run nvfp4_mixture_experts_moe_gb300.build.build())")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(s):
    return lib().moe_status_string(int(s)).decode()


def last_cuda_error():
    return lib().moe_last_cuda_error().decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status, what):
    if status != MOE_OK:
        raise MoeError(status, what)


def moe_route_topk(logits, T, E, k, topk_ids, topk_w, stream=None):
    _check(lib().moe_route_topk(_ptr(logits), T, E, k, _ptr(topk_ids), _ptr(topk_w), _stream(stream)),
           "moe_route_topk")


def moe_router_gemm(x, w_router, T, H, E, logits, stream=None):
    _check(lib().moe_router_gemm(_ptr(x), _ptr(w_router), T, H, E, _ptr(logits), _stream(stream)),
           "moe_router_gemm")


def moe_permute_workspace_size(T, k, E):
    return lib().moe_permute_workspace_size(T, k, E)


def moe_permute(topk_ids, T, k, E, counts, offsets, perm, inv_perm, ws, stream=None):
    _check(lib().moe_permute(_ptr(topk_ids), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm),
                             _ptr(inv_perm), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_permute")


def moe_quantize_workspace_size():
    return lib().moe_quantize_workspace_size()


def moe_nvfp4_quantize(x, rows, K, q, sf, gs_out, ws, stream=None):
    _check(lib().moe_nvfp4_quantize(_ptr(x), rows, K, _ptr(q), _ptr(sf), _ptr(gs_out), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)),
           "moe_nvfp4_quantize")


def moe_nvfp4_quantize_static(x, rows, K, gs, q, sf, stream=None):
    _check(lib().moe_nvfp4_quantize_static(_ptr(x), rows, K, float(gs), _ptr(q), _ptr(sf), _stream(stream)),
           "moe_nvfp4_quantize_static")


def moe_mxfp4_quantize(x, rows, K, q, sf, stream=None):
    _check(lib().moe_mxfp4_quantize(_ptr(x), rows, K, _ptr(q), _ptr(sf), _stream(stream)), "moe_mxfp4_quantize")


def moe_import_global_scale(stored, fmt):
    """A checkpoint's stored global scale -> the quant-convention gs (host only)."""
    out = ctypes.c_float(0.0)
    _check(lib().moe_import_global_scale(float(stored), int(fmt), ctypes.byref(out)), "moe_import_global_scale")
    return out.value


def moe_nvfp4_fold_scales(sf_in, n, ratio, sf_out, stream=None):
    _check(lib().moe_nvfp4_fold_scales(_ptr(sf_in), n, float(ratio), _ptr(sf_out), _stream(stream)),
           "moe_nvfp4_fold_scales")


def moe_prepare_size(N, K, mode, gate_up):
    return lib().moe_prepare_size(N, K, mode, gate_up)


def moe_nvfp4_prepare_weights(codes, sf, gs, N, K, mode, gate_up, out, stream=None):
    """``gs`` is a sequence of host floats (one, or gate and up); None for MXFP4."""
    gp = None
    if gs is not None:
        arr = (ctypes.c_float * len(gs))(*[float(v) for v in gs])
        gp = ctypes.cast(arr, ctypes.c_void_p)
    _check(lib().moe_nvfp4_prepare_weights(_ptr(codes), _ptr(sf), gp, N, K, mode, gate_up, _ptr(out),
                                           _stream(stream)),
           "moe_nvfp4_prepare_weights")


def moe_gemm_workspace_size(num_groups):
    return lib().moe_gemm_workspace_size(num_groups)


def moe_gemm_workspace_size_rows(num_groups, rows, K):
    return lib().moe_gemm_workspace_size_rows(num_groups, rows, K)


def moe_nvfp4_grouped_gemm(args: MoeGemmArgs, ws, stream=None):
    _check(lib().moe_nvfp4_grouped_gemm(ctypes.byref(args), _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream)),
           "moe_nvfp4_grouped_gemm")


def moe_swiglu(gu, rows, I, h, stream=None):
    _check(lib().moe_swiglu(_ptr(gu), rows, I, _ptr(h), _stream(stream)), "moe_swiglu")


def moe_combine(y, inv_perm, topk_w, y_shared, T, k, H, out, stream=None):
    _check(lib().moe_combine(_ptr(y), _ptr(inv_perm), _ptr(topk_w), _ptr(y_shared), T, k, H, _ptr(out),
                             _stream(stream)),
           "moe_combine")


def moe_workspace_size(desc: MoeLayerDesc):
    return lib().moe_workspace_size(ctypes.byref(desc))


def moe_nvfp4_forward(desc: MoeLayerDesc, x, logits, out, topk_ids_out, ws, stream=None, ws_bytes=None):
    nbytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().moe_nvfp4_forward(ctypes.byref(desc), _ptr(x), _ptr(logits), _ptr(out), _ptr(topk_ids_out),
                                   _ptr(ws), nbytes, _stream(stream)),
           "moe_nvfp4_forward")


def moe_get_device_status(ws, stream=None):
    """Synchronises and returns (and clears) the device status word of ``ws``."""
    return lib().moe_get_device_status(_ptr(ws), _stream(stream))


def moe_set_stage_events(events):
    """``events``: list of MOE_STAGE_COUNT torch.cuda.Event (or None to clear)."""
    if events is None:
        _check(lib().moe_set_stage_events(None, 0), "moe_set_stage_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().moe_set_stage_events(arr, len(events)), "moe_set_stage_events")


def moe_kernel_launches():
    return int(lib().moe_kernel_launches())


def moe_permute_noalloc(topk_ids, T, k, E, counts, offsets, perm, inv_perm, device_status=None, stream=None):
    """moe_permute without a workspace (fixed device scratch inside the library)."""
    _check(lib().moe_permute_noalloc(_ptr(topk_ids), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm),
                                     _ptr(inv_perm), _ptr(device_status), _stream(stream)),
           "moe_permute_noalloc")


def moe_debug_set(key, value):
    """Test hook (process-wide): see MOE_DEBUG_* in include/moe_nvfp4.h."""
    _check(lib().moe_debug_set(int(key), int(value)), "moe_debug_set")
