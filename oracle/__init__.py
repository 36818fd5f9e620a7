"""CPU oracle for the active-expert-chunked low-precision MoE layer.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference arm of ``bench.py`` import this package.  The
product path (``precision_moe_adapter_gb300``) never imports, loads or calls
it, and shares no code with it.

The arithmetic lives in ``pmoe_oracle.c`` (plain C, double-precision
accumulation, OpenMP only across independent tokens / blocks).  This module
compiles it with gcc on first use and exposes one numpy-level function per
step of the method:

  dequant        -- active-expert-chunked dequantization (Orbit announcement, 技艺细节):
                    INT4 group-32 / MXFP4 / FP8 [128,128] weights -> BF16
  route          -- router top-k + softmax over the selected experts
  topk           -- the selection and softmax alone, on given logits
  route_canonical -- router logits in one fixed FP32 summation order
  permute        -- grouping of (token, slot) pairs by expert
  forward        -- per-token definition of the layer (no chunks)
  backward       -- backward-data: dX, d_topk_w, adapter gradients; no base
                    weight gradient (bypass-base-weight-grad backward, Orbit announcement)
  adapter_apply / adapter_grad -- block-diagonal orthogonal (OFT) rotation
  cayley / cayley_grad         -- R = (I+S)(I-S)^-1 per block

Pins: every function is checked against facts other than itself in
``tests/test_oracle_*.py`` (exhaustive format tables against library
conversions, brute-force nearest-BF16, closed forms, finite differences,
textbook special cases).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pmoe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

INT4, MXFP4, FP8 = 0, 1, 2
NO_ROUND = 1


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP).

    Contraction of a*b+c into FMA is disabled so that x86 and Arm hosts give
    identical results."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64


class _Layer(ctypes.Structure):
    _fields_ = [("T", _i), ("d", _i), ("E", _i), ("k", _i), ("I", _i), ("b", _i),
                ("fmt", _i),
                ("w13", _p), ("s13", _p), ("w2", _p), ("s2", _p),
                ("R_up", _p), ("stride_up", _i64), ("R_down", _p), ("stride_down", _i64),
                ("R_up64", _p), ("R_down64", _p)]


def _declare(L):
    L.or_bf16_round.argtypes = [ctypes.c_double]
    L.or_bf16_round.restype = ctypes.c_uint16
    L.or_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.or_bf16_to_double.restype = ctypes.c_double
    L.or_e4m3_value.argtypes = [ctypes.c_uint]
    L.or_e4m3_value.restype = ctypes.c_double
    L.or_dequant.argtypes = [_i, _p, _p, _i64, _i64, _p]
    L.or_route.argtypes = [_i, _i, _i, _i, _p, _p, _p, _p, _i, _p, _p, _p]
    L.or_topk.argtypes = [_i, _i, _p, _p, _i, _p, _p]
    L.or_topk.restype = None
    L.or_route_canonical.argtypes = [_i, _i, _p, _p, _p, _p, _i, _p]
    L.or_route_canonical.restype = None
    L.or_permute.argtypes = [_i, _i, _p, _p, _p, _p, _p, _p, _p]
    L.or_adapter_apply.argtypes = [_i, _i, _i, _p, _p, _p]
    L.or_adapter_grad.argtypes = [_i, _i, _i, _p, _p, _p, _p, _p]
    L.or_cayley.argtypes = [_i, _i, _p, _p]
    L.or_dense_forward.argtypes = [_i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _i, _p, _p]
    L.or_dense_forward.restype = None
    L.or_dense_backward.argtypes = [_i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _i, _p, _p, _p]
    L.or_dense_backward.restype = None
    L.or_cayley.restype = _i
    L.or_cayley_grad.argtypes = [_i, _i, _p, _p, _p]
    L.or_cayley_grad.restype = _i
    L.or_forward.argtypes = [ctypes.POINTER(_Layer), _p, _p, _p, _p, _p, _i, _i, _p, _p, _p]
    L.or_backward.argtypes = [ctypes.POINTER(_Layer), _p, _p, _p, _p, _p, _p, _i, _i,
                              _p, _p, _p, _p, _p]
    L.or_num_threads.restype = _i
    L.or_pre_round.argtypes = [ctypes.POINTER(_Layer), _p, _p, _p, _i, _p]
    L.or_pre_round.restype = None


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return _L().or_num_threads()


# ---------------------------------------------------------------- scalars

def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round doubles to BF16 (RNE), returned as uint16 bit patterns."""
    v = np.ascontiguousarray(v, dtype=np.float64).ravel()
    f = _L().or_bf16_round
    return np.array([f(float(x)) for x in v], dtype=np.uint16)


def e4m3_values() -> np.ndarray:
    """The 256 E4M3 (FN) codes decoded by the oracle, as doubles."""
    f = _L().or_e4m3_value
    return np.array([f(c) for c in range(256)], dtype=np.float64)


# ---------------------------------------------------------------- dequant

def dequant(fmt: int, q: np.ndarray, s: np.ndarray, N: int, K: int) -> np.ndarray:
    """Dequantize one [N, K] weight matrix to BF16 bits (uint16 [N, K])."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s)
    out = np.empty((N, K), dtype=np.uint16)
    _L().or_dequant(fmt, _ptr(q), _ptr(s), N, K, _ptr(out))
    return out


# ---------------------------------------------------------------- routing

def route(X: np.ndarray, Wr: np.ndarray, bias, k: int, toks=None):
    """Router: FP32 logits (double sum), top-k by (logit desc, id asc),
    softmax over the k selected.  Returns (logits f32 [T,E], idx i32 [T,k],
    w f32 [T,k]); rows not in ``toks`` are left zero."""
    X = _c(X, np.uint16)
    Wr = _c(Wr, np.float32)
    bias = _c(bias, np.float32)
    T, d = X.shape
    E = Wr.shape[1]
    toks_a = _c(toks, np.int32)
    n = T if toks is None else len(toks_a)
    logits = np.zeros((T, E), np.float32)
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    _L().or_route(T, d, E, k, _ptr(X), _ptr(Wr), _ptr(bias), _ptr(toks_a), n,
                  _ptr(logits), _ptr(idx), _ptr(w))
    return logits, idx, w


def topk(logits: np.ndarray, k: int, toks=None):
    """Selection and weights from given FP32 logits [T, E] (bias included):
    top-k by (logit desc, id asc), softmax over the k selected in double
    rounded to FP32.  Returns (idx i32 [T,k], w f32 [T,k]); rows not in
    ``toks`` are left zero."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    toks_a = _c(toks, np.int32)
    n = T if toks is None else len(toks_a)
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    _L().or_topk(E, k, _ptr(logits), _ptr(toks_a), n, _ptr(idx), _ptr(w))
    return idx, w


def route_canonical(X: np.ndarray, Wr: np.ndarray, bias, toks=None) -> np.ndarray:
    """The router logits in the library's canonical FP32 summation order
    (32 lane-strided fmaf chains, then a pairwise tree, then + bias):
    f32 [T, E]; rows not in ``toks`` are left zero."""
    X = _c(X, np.uint16)
    Wr = _c(Wr, np.float32)
    bias = _c(bias, np.float32)
    T, d = X.shape
    E = Wr.shape[1]
    toks_a = _c(toks, np.int32)
    n = T if toks is None else len(toks_a)
    logits = np.zeros((T, E), np.float32)
    _L().or_route_canonical(d, E, _ptr(X), _ptr(Wr), _ptr(bias), _ptr(toks_a), n, _ptr(logits))
    return logits


def permute(idx: np.ndarray, E: int):
    """Grouping of the pairs p = t*k + j by expert.  Returns a dict with
    counts [E], offsets [E+1], perm [P], inv_perm [P], active [E] (-1
    padded) and num_active."""
    idx = _c(idx, np.int32).ravel()
    P = idx.size
    out = dict(counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
               perm=np.zeros(P, np.int32), inv_perm=np.zeros(P, np.int32),
               active=np.zeros(E, np.int32))
    na = np.zeros(1, np.int32)
    _L().or_permute(P, E, _ptr(idx), _ptr(out["counts"]), _ptr(out["offsets"]),
                    _ptr(out["perm"]), _ptr(out["inv_perm"]), _ptr(out["active"]), _ptr(na))
    out["num_active"] = int(na[0])
    return out


# ---------------------------------------------------------------- adapter

def cayley(S: np.ndarray) -> np.ndarray:
    """R = (I+S)(I-S)^-1 per block, double [nblk, b, b]."""
    S = _c(S, np.float64)
    b = S.shape[-1]
    nblk = S.size // (b * b)
    R = np.empty(S.shape, np.float64)
    rc = _L().or_cayley(nblk, b, _ptr(S), _ptr(R))
    if rc:
        raise ArithmeticError("singular I - S")
    return R


def cayley_grad(S: np.ndarray, G: np.ndarray) -> np.ndarray:
    """dL/dS (skew) given dL/dR, per block."""
    S = _c(S, np.float64)
    G = _c(G, np.float64)
    b = S.shape[-1]
    nblk = S.size // (b * b)
    dS = np.empty(S.shape, np.float64)
    rc = _L().or_cayley_grad(nblk, b, _ptr(S), _ptr(G), _ptr(dS))
    if rc:
        raise ArithmeticError("singular I - S")
    return dS


def adapter_apply(X: np.ndarray, R: np.ndarray, b: int) -> np.ndarray:
    """bf16(X blockdiag(R)); X bf16 bits [rows, dim], R bf16 bits [dim/b, b, b]."""
    X = _c(X, np.uint16)
    R = _c(R, np.uint16)
    rows, dim = X.shape
    out = np.empty_like(X)
    _L().or_adapter_apply(rows, dim, b, _ptr(X), _ptr(R), _ptr(out))
    return out


def adapter_grad(X, dXr, R, b: int, want_dx: bool = True):
    """Returns (dX bf16 bits or None, dR double [dim/b, b, b])."""
    X = _c(X, np.uint16)
    dXr = _c(dXr, np.uint16)
    R = _c(R, np.uint16)
    rows, dim = X.shape
    dX = np.empty_like(X) if want_dx else None
    dR = np.empty((dim // b, b, b), np.float64)
    _L().or_adapter_grad(rows, dim, b, _ptr(X), _ptr(dXr), _ptr(R), _ptr(dX), _ptr(dR))
    return dX, dR


# ---------------------------------------------------------------- dense linear

def dense_forward(fmt, q, s, N, K, b, R, X, no_round=False, R64=None, X64=None):
    """Dense bypass-base-weight-grad linear with the OFT adapter (see
    or_dense_forward).  q/s: one packed [N, K] matrix; R: BF16 bits
    [K/b, b, b] or None (R64: doubles instead).  X: BF16 bits [rows, K]
    (or X64 doubles).  Returns (Y bf16 bits [rows, N], Y64)."""
    q = _c(q, np.uint8)
    s = np.ascontiguousarray(s)
    R, R64, X64 = _c(R, np.uint16), _c(R64, np.float64), _c(X64, np.float64)
    X = _c(X, np.uint16)
    rows = (X if X is not None else X64).shape[0]
    Y = np.zeros((rows, N), np.uint16)
    Y64 = np.zeros((rows, N), np.float64)
    _L().or_dense_forward(rows, N, K, b, fmt, _ptr(q), _ptr(s), _ptr(R), _ptr(R64), _ptr(X),
                          _ptr(X64), NO_ROUND if no_round else 0, _ptr(Y), _ptr(Y64))
    return Y, Y64


def dense_backward(fmt, q, s, N, K, b, R, X, dY, no_round=False, R64=None, X64=None):
    """Backward-data of the dense linear: dict(dX bf16 bits, dX64, dR double
    [K/b, b, b] or None)."""
    q = _c(q, np.uint8)
    s = np.ascontiguousarray(s)
    R, R64, X64 = _c(R, np.uint16), _c(R64, np.float64), _c(X64, np.float64)
    X, dY = _c(X, np.uint16), _c(dY, np.uint16)
    rows = dY.shape[0]
    dX = np.zeros((rows, K), np.uint16)
    dX64 = np.zeros((rows, K), np.float64)
    dR = None if R is None and R64 is None else np.zeros((K // b, b, b), np.float64)
    _L().or_dense_backward(rows, N, K, b, fmt, _ptr(q), _ptr(s), _ptr(R), _ptr(R64), _ptr(X),
                           _ptr(X64), _ptr(dY), NO_ROUND if no_round else 0, _ptr(dX),
                           _ptr(dX64), _ptr(dR))
    return dict(dX=dX, dX64=dX64, dR=dR)


# ---------------------------------------------------------------- layer

class Layer:
    """The frozen quantized experts plus the (optional) adapter.

    fmt: INT4 / MXFP4 / FP8; w13 [E, 2I, ...] (gate rows then up rows),
    w2 [E, d, ...]; R_up [E or 1, d/b, b, b] and R_down [E or 1, I/b, b, b]
    as BF16 bits, or None for a disabled adapter."""

    def __init__(self, T, d, E, k, I, b, fmt, w13, s13, w2, s2, R_up=None, R_down=None,
                 R_up64=None, R_down64=None):
        self.keep = [np.ascontiguousarray(a) for a in (w13, s13, w2, s2)]
        self.R_up = None if R_up is None else np.ascontiguousarray(R_up, dtype=np.uint16)
        self.R_down = None if R_down is None else np.ascontiguousarray(R_down, dtype=np.uint16)
        self.R_up64 = None if R_up64 is None else np.ascontiguousarray(R_up64, dtype=np.float64)
        self.R_down64 = None if R_down64 is None else np.ascontiguousarray(R_down64, dtype=np.float64)
        if self.R_up is None and self.R_up64 is not None:
            self.R_up = np.zeros(self.R_up64.shape, np.uint16)
        if self.R_down is None and self.R_down64 is not None:
            self.R_down = np.zeros(self.R_down64.shape, np.uint16)
        su = 0 if (self.R_up is None or self.R_up.shape[0] == 1) else d * b
        sd = 0 if (self.R_down is None or self.R_down.shape[0] == 1) else I * b
        self.c = _Layer(T, d, E, k, I, b, fmt, *[_ptr(a) for a in self.keep],
                        _ptr(self.R_up), su, _ptr(self.R_down), sd,
                        _ptr(self.R_up64), _ptr(self.R_down64))
        self.T, self.d, self.E, self.k, self.I, self.b = T, d, E, k, I, b

    def forward(self, X, idx, w, toks=None, no_round=False, want_o=False, X64=None):
        """Y (bf16 bits [T, d]), Y64 (double [T, d]) and optionally o per
        pair (double [T*k, d]); rows not in ``toks`` stay zero.  ``X64``
        (double [T, d]) replaces X when given."""
        X = _c(X, np.uint16) if X is not None else np.zeros((self.T, self.d), np.uint16)
        X64 = _c(X64, np.float64)
        idx = _c(idx, np.int32)
        w = _c(w, np.float32)
        toks_a = _c(toks, np.int32)
        n = self.T if toks is None else len(toks_a)
        Y = np.zeros((self.T, self.d), np.uint16)
        Y64 = np.zeros((self.T, self.d), np.float64)
        o = np.zeros((self.T * self.k, self.d), np.float64) if want_o else None
        _L().or_forward(ctypes.byref(self.c), _ptr(X), _ptr(X64), _ptr(idx), _ptr(w), _ptr(toks_a), n,
                        NO_ROUND if no_round else 0, _ptr(Y), _ptr(Y64), _ptr(o))
        return (Y, Y64, o) if want_o else (Y, Y64)

    def pre_round(self, X, idx, toks):
        """For each pair of the listed tokens (row it*k + j): silu(g) u
        before its rounding to h, and h R_down before its rounding to h~,
        as double [n*k, 2I]."""
        X = _c(X, np.uint16)
        idx = _c(idx, np.int32)
        toks_a = _c(toks, np.int32)
        hx = np.zeros((len(toks_a) * self.k, 2 * self.I), np.float64)
        _L().or_pre_round(ctypes.byref(self.c), _ptr(X), _ptr(idx), _ptr(toks_a), len(toks_a),
                          _ptr(hx))
        return hx

    def backward(self, X, dY, idx, w, toks=None, no_round=False, X64=None):
        """Returns dict(dX bf16 bits, dX64, d_topk_w f32 [T,k], dR_up,
        dR_down double) -- the adapter gradients summed over ``toks``."""
        X = _c(X, np.uint16) if X is not None else np.zeros((self.T, self.d), np.uint16)
        X64 = _c(X64, np.float64)
        dY = _c(dY, np.uint16)
        idx = _c(idx, np.int32)
        w = _c(w, np.float32)
        toks_a = _c(toks, np.int32)
        n = self.T if toks is None else len(toks_a)
        dX = np.zeros((self.T, self.d), np.uint16)
        dX64 = np.zeros((self.T, self.d), np.float64)
        dtw = np.zeros((self.T, self.k), np.float32)
        dR_up = None if self.R_up is None else np.zeros(self.R_up.shape, np.float64)
        dR_dn = None if self.R_down is None else np.zeros(self.R_down.shape, np.float64)
        _L().or_backward(ctypes.byref(self.c), _ptr(X), _ptr(X64), _ptr(dY), _ptr(idx), _ptr(w),
                         _ptr(toks_a), n, NO_ROUND if no_round else 0, _ptr(dX), _ptr(dX64),
                         _ptr(dtw), _ptr(dR_up), _ptr(dR_dn))
        return dict(dX=dX, dX64=dX64, d_topk_w=dtw, dR_up=dR_up, dR_down=dR_dn)
