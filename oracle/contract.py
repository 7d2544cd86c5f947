"""ctypes wrapper around contract.c, the CPU restatement of the library's
documented reduction order (router projection and shared gate).

TEST INFRASTRUCTURE ONLY: imported by the test suite alone.  It shares no
code with the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

from oracle.oracle import CFLAGS

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "contract.c")
_LIB = os.path.join(_HERE, "libcontract.so")
_L = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _lib():
    global _L
    if _L is None:
        _L = C.CDLL(build())
        P, I = C.c_void_p, C.c_int64
        _L.ctr_router_f32in.argtypes = [P, P, I, I, I, P]
        _L.ctr_router_bf16in.argtypes = [P, P, I, I, I, P, P, P]
    return _L


def router_logits(X, W) -> np.ndarray:
    """f32 [M, E] logits in the contract's order; X, W are float32 arrays or
    uint16 bf16 bit patterns (both the same kind)."""
    M, H = X.shape
    E = W.shape[0]
    out = np.empty((M, E), np.float32)
    if X.dtype == np.uint16:
        xa = np.ascontiguousarray(X, np.uint16)
        wa = np.ascontiguousarray(W, np.uint16)
        xs = np.empty(H, np.float32)
        ws = np.empty(E * H, np.float32)
        _lib().ctr_router_bf16in(xa.ctypes.data, wa.ctypes.data, M, E, H, out.ctypes.data,
                                 xs.ctypes.data, ws.ctypes.data)
    else:
        xa = np.ascontiguousarray(X, np.float32)
        wa = np.ascontiguousarray(W, np.float32)
        _lib().ctr_router_f32in(xa.ctypes.data, wa.ctypes.data, M, E, H, out.ctypes.data)
    return out
