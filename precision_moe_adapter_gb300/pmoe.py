"""Thin ctypes binding of libpmoe.so (C ABI in include/pmoe.h).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  Tensors are passed as device pointers (``tensor.data_ptr()``)
together with the current torch stream; integers are accepted as raw
pointers.  There is no CPU fallback: if the library is missing, loading it
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libpmoe.so")

PMOE_OK, PMOE_ERR_INVALID_ARG, PMOE_ERR_UNSUPPORTED, PMOE_ERR_WORKSPACE = 0, 1, 2, 3
PMOE_ERR_CUDA, PMOE_ERR_BAD_INDEX, PMOE_ERR_TIMEOUT = 4, 5, 6
W_INT4_G32_BF16, W_MXFP4_G32_E8M0, W_FP8_B128_F32 = 0, 1, 2
MODE_FUSED, MODE_SCRATCH = 0, 1
ROUTE_FAST, ROUTE_EXACT = 0, 1
OP_PERMUTE, OP_FORWARD, OP_BACKWARD = 0, 1, 2

EXPORTS = ("moe_route", "moe_permute", "moe_chunked_forward", "moe_backward_data", "moe_dequant",
           "adapter_apply", "adapter_grad", "adapter_cayley", "adapter_cayley_grad",
           "moe_workspace_bytes", "moe_scratch_bytes", "moe_ctx_bytes", "moe_clear_status",
           "moe_query_status",
           "pmoe_status_string", "pmoe_launch_count", "pmoe_kernel_timing", "pmoe_kernel_time",
           "moe_grouped_gemm", "moe_grouped_gemm_ws_bytes", "moe_permute_noalloc",
           "dense_linear_ws_bytes", "dense_linear_forward", "dense_linear_backward",
           "moe_adapter_publish", "moe_chunked_forward_slots", "pmoe_debug_expire_gemm_wait")
PERMUTE_NOALLOC_SCRATCH_BYTES = 1 << 20
KT_GEMM_GATE_UP, KT_GEMM_DOWN, KT_GEMM_BWD_G, KT_GEMM_BWD_DX, KT_ROUTER = 0, 1, 2, 3, 4


class PmoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("inter", ctypes.c_int32), ("block", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("w13", ctypes.c_void_p), ("s13", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("s2", ctypes.c_void_p)]


class Adapter(ctypes.Structure):
    _fields_ = [("R_up", ctypes.c_void_p), ("R_down", ctypes.c_void_p),
                ("stride_up", ctypes.c_int64), ("stride_down", ctypes.c_int64)]


class AdapterSlots(ctypes.Structure):
    _fields_ = [("R_up", ctypes.c_void_p * 2), ("R_down", ctypes.c_void_p * 2),
                ("stride_up", ctypes.c_int64), ("stride_down", ctypes.c_int64),
                ("ctrl", ctypes.c_void_p)]


class Routing(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("idx", "w", "counts", "offsets", "perm", "inv_perm", "active", "num_active")]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libpmoe.so (built by ``build.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise FileNotFoundError(
                    f"{LIB_PATH} is missing: build it with precision_moe_adapter_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            _declare(L)
            _lib = L
    return _lib


def _declare(L):
    p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    st = ctypes.c_int
    D, PW, PA, PR = Dims, ctypes.POINTER(Weights), ctypes.POINTER(Adapter), ctypes.POINTER(Routing)
    sig = {
        "moe_route": [D, p, p, p, p, p, p, ctypes.c_int, p, sz, p],
        "moe_permute": [D, p, PR, p, sz, p],
        "moe_permute_noalloc": [D, p, PR, p],
        "moe_adapter_publish": [p, ctypes.c_uint32, ctypes.c_uint32, p],
        "moe_chunked_forward_slots": [D, PW, ctypes.POINTER(AdapterSlots), PR, p, i32, ctypes.c_int,
                                      p, p, p, p, sz, p],
        "dense_linear_forward": [ctypes.c_int, p, p, i32, i32, i32, p, i32, p, p, p, sz, p],
        "dense_linear_backward": [ctypes.c_int, p, p, i32, i32, i32, p, i32, p, p, p, p, p, sz, p],
        "moe_chunked_forward": [D, PW, PA, PR, p, i32, ctypes.c_int, p, p, p, sz, p],
        "moe_backward_data": [D, PW, PA, PR, p, p, p, i32, p, p, p, p, p, sz, p],
        "moe_dequant": [ctypes.c_int, p, p, i64, i64, p, p],
        "moe_grouped_gemm": [ctypes.c_int, p, p, i32, i32, i32, ctypes.c_int, p, p, i32, p, p, sz, p],
        "adapter_apply": [i32, i32, i32, p, p, p, p],
        "adapter_grad": [i32, i32, i32, p, p, p, p, p, p],
        "adapter_cayley": [i32, i32, p, p, p, p],
        "adapter_cayley_grad": [i32, i32, p, p, p, p, p],
        "moe_clear_status": [p, p],
        "moe_query_status": [p, p],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = st
    L.moe_workspace_bytes.argtypes = [D, ctypes.c_int, i32, ctypes.c_int]
    L.moe_workspace_bytes.restype = sz
    L.moe_grouped_gemm_ws_bytes.argtypes = [i32, i32]
    L.moe_grouped_gemm_ws_bytes.restype = sz
    L.dense_linear_ws_bytes.argtypes = [i32, i32, i32]
    L.dense_linear_ws_bytes.restype = sz
    L.moe_scratch_bytes.argtypes = [D, i32, ctypes.c_int]
    L.moe_scratch_bytes.restype = sz
    L.moe_ctx_bytes.argtypes = [D]
    L.moe_ctx_bytes.restype = sz
    L.pmoe_debug_expire_gemm_wait.argtypes = [ctypes.c_uint64]
    L.pmoe_debug_expire_gemm_wait.restype = st
    L.pmoe_status_string.argtypes = [st]
    L.pmoe_status_string.restype = ctypes.c_char_p
    L.pmoe_launch_count.argtypes = []
    L.pmoe_launch_count.restype = ctypes.c_uint64
    L.pmoe_kernel_timing.argtypes = [ctypes.c_int]
    L.pmoe_kernel_timing.restype = st
    L.pmoe_kernel_time.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_int)]
    L.pmoe_kernel_time.restype = st


def status_string(s: int) -> str:
    return lib().pmoe_status_string(s).decode()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(t):
    return t.numel() * t.element_size()


def _check(s: int, where: str):
    if s != PMOE_OK:
        raise PmoeError(s, where)


def dims(T, d, E, k, inter, block) -> Dims:
    return Dims(T, d, E, k, inter, block)


def weights(fmt, w13, s13, w2, s2) -> Weights:
    return Weights(fmt, _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2))


def adapter(R_up=None, R_down=None, stride_up=0, stride_down=0) -> Adapter:
    return Adapter(_ptr(R_up), _ptr(R_down), stride_up, stride_down)


def routing(idx, w, counts, offsets, perm, inv_perm, active, num_active) -> Routing:
    return Routing(*[_ptr(t) for t in (idx, w, counts, offsets, perm, inv_perm, active, num_active)])


# ------------------------------------------------------------------ entry points

def moe_workspace_bytes(dm: Dims, op: int, chunk_C: int = 1, mode: int = MODE_FUSED) -> int:
    return lib().moe_workspace_bytes(dm, op, chunk_C, mode)


def moe_scratch_bytes(dm: Dims, chunk_C: int, mode: int) -> int:
    return lib().moe_scratch_bytes(dm, chunk_C, mode)


def moe_ctx_bytes(dm: Dims) -> int:
    return lib().moe_ctx_bytes(dm)


def pmoe_debug_expire_gemm_wait(wait_ns: int):
    _check(lib().pmoe_debug_expire_gemm_wait(wait_ns), "pmoe_debug_expire_gemm_wait")


def moe_route(dm, X, Wr, bias, logits, idx, w, ws, mode=ROUTE_FAST, stream=None):
    _check(lib().moe_route(dm, _ptr(X), _ptr(Wr), _ptr(bias), _ptr(logits), _ptr(idx), _ptr(w),
                           mode, _ptr(ws), _nbytes(ws), _stream(stream)), "moe_route")


def moe_permute(dm, idx, rt: Routing, ws, stream=None):
    _check(lib().moe_permute(dm, _ptr(idx), ctypes.byref(rt), _ptr(ws), _nbytes(ws),
                             _stream(stream)), "moe_permute")


def adapter_slots(R_up0, R_up1, R_down0, R_down1, stride_up, stride_down, ctrl) -> AdapterSlots:
    a = AdapterSlots()
    a.R_up[0], a.R_up[1] = _ptr(R_up0), _ptr(R_up1)
    a.R_down[0], a.R_down[1] = _ptr(R_down0), _ptr(R_down1)
    a.stride_up, a.stride_down, a.ctrl = stride_up, stride_down, _ptr(ctrl)
    return a


def moe_adapter_publish(ctrl, slot, version, stream=None):
    _check(lib().moe_adapter_publish(_ptr(ctrl), slot, version, _stream(stream)),
           "moe_adapter_publish")


def moe_chunked_forward_slots(dm, wts: Weights, slots: AdapterSlots, rt: Routing, X, chunk_C, mode,
                              Y, ctx, version_out, ws, stream=None):
    _check(lib().moe_chunked_forward_slots(dm, ctypes.byref(wts), ctypes.byref(slots),
                                           ctypes.byref(rt), _ptr(X), chunk_C, mode, _ptr(Y),
                                           _ptr(ctx), _ptr(version_out), _ptr(ws), _nbytes(ws),
                                           _stream(stream)), "moe_chunked_forward_slots")


def dense_linear_ws_bytes(rows, N, K) -> int:
    return int(lib().dense_linear_ws_bytes(rows, N, K))


def dense_linear_forward(fmt, q, s, N, K, block, R, rows, X, Y, ws, stream=None):
    _check(lib().dense_linear_forward(fmt, _ptr(q), _ptr(s), N, K, block, _ptr(R), rows, _ptr(X),
                                      _ptr(Y), _ptr(ws), _nbytes(ws), _stream(stream)),
           "dense_linear_forward")


def dense_linear_backward(fmt, q, s, N, K, block, R, rows, X, dY, dX, dR, ws, stream=None):
    _check(lib().dense_linear_backward(fmt, _ptr(q), _ptr(s), N, K, block, _ptr(R), rows, _ptr(X),
                                       _ptr(dY), _ptr(dX), _ptr(dR), _ptr(ws), _nbytes(ws),
                                       _stream(stream)), "dense_linear_backward")


def moe_permute_noalloc(dm, idx, rt: Routing, stream=None):
    _check(lib().moe_permute_noalloc(dm, _ptr(idx), ctypes.byref(rt), _stream(stream)),
           "moe_permute_noalloc")


def moe_chunked_forward(dm, wts: Weights, adp, rt: Routing, X, chunk_C, mode, Y, ctx, ws,
                        stream=None):
    _check(lib().moe_chunked_forward(dm, ctypes.byref(wts), ctypes.byref(adp) if adp else None,
                                     ctypes.byref(rt), _ptr(X), chunk_C, mode, _ptr(Y), _ptr(ctx),
                                     _ptr(ws), _nbytes(ws), _stream(stream)),
           "moe_chunked_forward")


def moe_backward_data(dm, wts: Weights, adp, rt: Routing, X, dY, ctx, chunk_C, dX, d_topk_w,
                      dR_up, dR_down, ws, stream=None):
    _check(lib().moe_backward_data(dm, ctypes.byref(wts), ctypes.byref(adp) if adp else None,
                                   ctypes.byref(rt), _ptr(X), _ptr(dY), _ptr(ctx), chunk_C,
                                   _ptr(dX), _ptr(d_topk_w), _ptr(dR_up), _ptr(dR_down),
                                   _ptr(ws), _nbytes(ws), _stream(stream)), "moe_backward_data")


def moe_dequant(fmt, q, s, N, K, out, stream=None):
    _check(lib().moe_dequant(fmt, _ptr(q), _ptr(s), N, K, _ptr(out), _stream(stream)),
           "moe_dequant")


def moe_grouped_gemm_ws_bytes(E: int, rows: int) -> int:
    return lib().moe_grouped_gemm_ws_bytes(E, rows)


def moe_grouped_gemm(fmt, q, s, E, N, K, trans, A, offsets, rows, out, ws, stream=None):
    _check(lib().moe_grouped_gemm(fmt, _ptr(q), _ptr(s), E, N, K, trans, _ptr(A), _ptr(offsets),
                                  rows, _ptr(out), _ptr(ws), _nbytes(ws), _stream(stream)),
           "moe_grouped_gemm")


def adapter_apply(rows, dim, b, X, R, Xr, stream=None):
    _check(lib().adapter_apply(rows, dim, b, _ptr(X), _ptr(R), _ptr(Xr), _stream(stream)),
           "adapter_apply")


def adapter_grad(rows, dim, b, X, dXr, R, dX, dR, stream=None):
    _check(lib().adapter_grad(rows, dim, b, _ptr(X), _ptr(dXr), _ptr(R), _ptr(dX), _ptr(dR),
                              _stream(stream)), "adapter_grad")


def adapter_cayley(nblk, b, S, R_bf16, R_f32, stream=None):
    _check(lib().adapter_cayley(nblk, b, _ptr(S), _ptr(R_bf16), _ptr(R_f32), _stream(stream)),
           "adapter_cayley")


def adapter_cayley_grad(nblk, b, S, R_f32, dR, dS, stream=None):
    _check(lib().adapter_cayley_grad(nblk, b, _ptr(S), _ptr(R_f32), _ptr(dR), _ptr(dS),
                                     _stream(stream)), "adapter_cayley_grad")


def moe_clear_status(ws, stream=None):
    _check(lib().moe_clear_status(_ptr(ws), _stream(stream)), "moe_clear_status")


def moe_query_status(ws, stream=None) -> int:
    """Device error word of ``ws`` (PMOE_OK when clean); synchronizes."""
    return lib().moe_query_status(_ptr(ws), _stream(stream))


def pmoe_launch_count() -> int:
    return lib().pmoe_launch_count()


def pmoe_kernel_timing(enable: bool):
    _check(lib().pmoe_kernel_timing(1 if enable else 0), "pmoe_kernel_timing")


def pmoe_kernel_time(which: int):
    """(total ms, launches) of kernel class ``which`` since timing was enabled."""
    ms, n = ctypes.c_double(), ctypes.c_int()
    _check(lib().pmoe_kernel_time(which, ctypes.byref(ms), ctypes.byref(n)), "pmoe_kernel_time")
    return ms.value, n.value
