"""ctypes wrapper around the plain-C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the smoke check and
by the CPU-baseline leg of the benchmark, never by the library's product
path.  It shares no code with the CUDA library.

bf16 values travel as numpy uint16 bit patterns; the oracle widens them to
double exactly.  Every function returns fresh numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

FNV64_BASIS = 0xCBF29CE484222325
CFLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off"]


def build(force: bool = False) -> str:
    """Compile oracle.c with the host C compiler into oracle/liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Lib:
    """The loaded shared object; `path` may name another build of oracle.c
    (the mutation tests load deliberately broken copies this way)."""

    def __init__(self, path=None):
        self.L = C.CDLL(path or build())
        _declare(self.L)


_default = None
_current = None


def lib():
    global _default
    if _current is not None:
        return _current.L
    if _default is None:
        _default = _Lib()
    return _default.L


class use:
    """Context manager: route every function of this module to the oracle
    built at `path` (used only by the mutation tests)."""

    def __init__(self, path):
        self.inst = _Lib(path)

    def __enter__(self):
        global _current
        self.prev = _current
        _current = self.inst
        return self

    def __exit__(self, *exc):
        global _current
        _current = self.prev
        return False


_P = C.c_void_p
_I64 = C.c_int64
_I32 = C.c_int32


def _declare(L):
    L.orc_bf16_to_double.argtypes = [C.c_uint16]
    L.orc_bf16_to_double.restype = C.c_double
    L.orc_double_to_bf16_rne.argtypes = [C.c_double]
    L.orc_double_to_bf16_rne.restype = C.c_uint16
    L.orc_double_to_f32.argtypes = [C.c_double]
    L.orc_double_to_f32.restype = C.c_float
    L.orc_ord_bf16.argtypes = [C.c_uint16]
    L.orc_ord_bf16.restype = C.c_int64
    L.orc_ord_f32.argtypes = [C.c_uint32]
    L.orc_ord_f32.restype = C.c_int64
    for name in ("orc_router_logits_f32in", "orc_router_logits_bf16in", "orc_router_absdot_f32in"):
        getattr(L, name).argtypes = [_P, _I64, _P, _I64, _I64, _I64, _I64, _P]
        getattr(L, name).restype = None
    L.orc_topk.argtypes = [_P, _I64, _I32, _I32, _P]
    L.orc_topk.restype = None
    L.orc_softmax_selected.argtypes = [_P, _I64, _I32, _I32, _P, _P]
    L.orc_softmax_selected.restype = None
    for name in ("orc_margin_f32", "orc_margin_bf16"):
        getattr(L, name).argtypes = [_P, _I64, _I32, _I32, _P, _P, _P, _P, _P]
        getattr(L, name).restype = None
    L.orc_shared_gate.argtypes = [_P, _I64, _P, _I64, _I64, _P, _P]
    L.orc_shared_gate.restype = None
    L.orc_gemm_bf16.argtypes = [_P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _I64]
    L.orc_gemm_bf16.restype = None
    L.orc_fnv64_basis.argtypes = []
    L.orc_fnv64_basis.restype = C.c_uint64
    L.orc_fnv1a64.argtypes = [_P, C.c_size_t, C.c_uint64]
    L.orc_fnv1a64.restype = C.c_uint64
    L.orc_route_hash.argtypes = [_P, _I32, _I64, _I64, C.c_uint64]
    L.orc_route_hash.restype = C.c_uint64
    L.orc_round_bf16_array.argtypes = [_P, _I64, _P]
    L.orc_round_bf16_array.restype = None
    L.orc_round_f32_array.argtypes = [_P, _I64, _P]
    L.orc_round_f32_array.restype = None
    L.orc_bf16_to_double_array.argtypes = [_P, _I64, _P]
    L.orc_bf16_to_double_array.restype = None


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(C.c_void_p)


def _p(a):
    return a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------- formats
def bf16_to_double(bits) -> np.ndarray:
    b, bp = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().orc_bf16_to_double_array(bp, b.size, _p(out))
    return out


def round_bf16(values) -> np.ndarray:
    """Round doubles to bf16 (RNE); returns uint16 bit patterns."""
    v, vp = _c(values, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_round_bf16_array(vp, v.size, _p(out))
    return out


def round_f32(values) -> np.ndarray:
    v, vp = _c(values, np.float64)
    out = np.empty(v.shape, dtype=np.float32)
    lib().orc_round_f32_array(vp, v.size, _p(out))
    return out


def ord_bf16(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    f = lib().orc_ord_bf16
    return np.array([f(int(x)) for x in b.ravel()], dtype=np.int64).reshape(b.shape)


def ord_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint32)
    f = lib().orc_ord_f32
    return np.array([f(int(x)) for x in b.ravel()], dtype=np.int64).reshape(b.shape)


# ---------------------------------------------------------------- router
def router_logits(X, W) -> np.ndarray:
    """Exact-input double dot: X [M,H], W [E,H] (float32, or uint16 bf16 bits)."""
    X = np.asarray(X)
    W = np.asarray(W)
    M, H = X.shape
    E = W.shape[0]
    out = np.empty((M, E), dtype=np.float64)
    if X.dtype == np.uint16:
        xa, xp = _c(X, np.uint16)
        wa, wp = _c(W, np.uint16)
        lib().orc_router_logits_bf16in(xp, H, wp, H, M, H, E, _p(out))
    else:
        xa, xp = _c(X, np.float32)
        wa, wp = _c(W, np.float32)
        lib().orc_router_logits_f32in(xp, H, wp, H, M, H, E, _p(out))
    return out


def router_absdot(X, W) -> np.ndarray:
    """sum_h |X[m,h] W[e,h]| for float32 inputs (tolerance scale)."""
    xa, xp = _c(X, np.float32)
    wa, wp = _c(W, np.float32)
    M, H = xa.shape
    E = wa.shape[0]
    out = np.empty((M, E), dtype=np.float64)
    lib().orc_router_absdot_f32in(xp, H, wp, H, M, H, E, _p(out))
    return out


def topk(logits, k: int) -> np.ndarray:
    """Sequential top-k, lowest index on exact ties; ids [M,k] in rank order."""
    la, lp = _c(logits, np.float64)
    M, E = la.shape
    ids = np.empty((M, k), dtype=np.int32)
    lib().orc_topk(lp, M, E, k, _p(ids))
    return ids


def softmax_selected(logits, ids) -> np.ndarray:
    la, lp = _c(logits, np.float64)
    ia, ip = _c(ids, np.int32)
    M, E = la.shape
    k = ia.shape[1]
    w = np.empty((M, k), dtype=np.float64)
    lib().orc_softmax_selected(lp, M, E, k, ip, _p(w))
    return w


def margin(logits_typed, ids):
    """logits_typed: float32 [M,E] or uint16 bf16 bits [M,E].

    Returns (margin double [M], ulps int64 [M], sel_min_id [M], rej_max_id [M]).
    """
    lt = np.asarray(logits_typed)
    ia, ip = _c(ids, np.int32)
    M, E = lt.shape
    k = ia.shape[1]
    mg = np.empty(M, dtype=np.float64)
    ul = np.empty(M, dtype=np.int64)
    smin = np.empty(M, dtype=np.int32)
    rmax = np.empty(M, dtype=np.int32)
    ptrs = [_p(mg), _p(ul), _p(smin), _p(rmax)]
    if lt.dtype == np.uint16:
        la, lp = _c(lt, np.uint16)
        lib().orc_margin_bf16(lp, M, E, k, ip, *ptrs)
    else:
        la, lp = _c(lt, np.float32)
        lib().orc_margin_f32(lp, M, E, k, ip, *ptrs)
    return mg, ul, smin, rmax


def router_full(X, W, k: int, logit_dtype: str = "f32") -> dict:
    """The whole router step for one call, composed from the pieces above.

    logits are rounded to the logit dtype first; selection, weights and
    margins are then taken on those rounded values (the values a selection
    is a function of)."""
    exact = router_logits(X, W)
    if logit_dtype == "f32":
        typed = round_f32(exact)
        widened = typed.astype(np.float64)
    elif logit_dtype == "bf16":
        typed = round_bf16(exact)
        widened = bf16_to_double(typed)
    else:
        raise ValueError(logit_dtype)
    ids = topk(widened, k)
    w = softmax_selected(widened, ids)
    mg, ul, smin, rmax = margin(typed, ids)
    return {"exact": exact, "logits": typed, "widened": widened, "ids": ids, "weights": w,
            "margin": mg, "margin_ulps": ul, "sel_min_id": smin, "rej_max_id": rmax}


def selection_from_logits(typed, k: int) -> dict:
    """Top-k, weights and margins taken on given logits of the logit dtype
    (float32, or uint16 bf16 bits): used to apply the oracle's selection to
    the GPU's own logits."""
    typed = np.asarray(typed)
    widened = bf16_to_double(typed) if typed.dtype == np.uint16 else typed.astype(np.float64)
    ids = topk(widened, k)
    w = softmax_selected(widened, ids)
    mg, ul, smin, rmax = margin(typed, ids)
    return {"ids": ids, "weights": w, "margin": mg, "margin_ulps": ul,
            "sel_min_id": smin, "rej_max_id": rmax}


# ---------------------------------------------------------------- gate
def shared_gate(X, w):
    xa, xp = _c(X, np.float32)
    wa, wp = _c(w, np.float32)
    M, H = xa.shape
    dot = np.empty(M, dtype=np.float64)
    sig = np.empty(M, dtype=np.float64)
    lib().orc_shared_gate(xp, H, wp, M, H, _p(dot), _p(sig))
    return dot, sig


# ---------------------------------------------------------------- GEMM
def gemm_bf16(A, B, rows=None):
    """A uint16 [M,K], B uint16 [N,K] -> (acc double, absacc double, C uint16).

    rows: optional list of row indices of A to compute (sampled checks)."""
    A = np.asarray(A, dtype=np.uint16)
    if rows is not None:
        A = A[np.asarray(rows)]
    aa, ap = _c(A, np.uint16)
    ba, bp = _c(B, np.uint16)
    M, K = aa.shape
    N = ba.shape[0]
    acc = np.empty((M, N), dtype=np.float64)
    absacc = np.empty((M, N), dtype=np.float64)
    Cm = np.empty((M, N), dtype=np.uint16)
    lib().orc_gemm_bf16(ap, K, bp, K, M, N, K, _p(acc), _p(absacc), _p(Cm), N)
    return acc, absacc, Cm


# ---------------------------------------------------------------- hash
def fnv1a64(data: bytes, basis: int = FNV64_BASIS) -> int:
    buf = (C.c_uint8 * max(1, len(data))).from_buffer_copy(data if data else b"\0")
    return int(lib().orc_fnv1a64(C.cast(buf, C.c_void_p), len(data), C.c_uint64(basis)))


def route_hash(ids, row_begin=None, row_end=None, basis: int = FNV64_BASIS) -> int:
    ia, ip = _c(ids, np.int32)
    M, k = ia.shape
    rb = 0 if row_begin is None else row_begin
    re_ = M if row_end is None else row_end
    return int(lib().orc_route_hash(ip, k, rb, re_, C.c_uint64(basis)))


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
