"""Oracle for the batch-invariant RMSNorm (TEST INFRASTRUCTURE ONLY:
imported by the test suite alone; it shares no code with the library).

Source: "The Illusion of Determinism in Disaggregated Inference", section
"The physics of the cascade": RMSNorm takes one root-mean-square over the
whole hidden state and divides every element by it, so a one-ULP change in
one element reaches all of them; a batch-invariant normalisation keeps that
statistic's reduction order fixed per row.  Read here with the usual form:

    r[m]    = 1 / sqrt( (1/H) * sum_h x[m, h]^2 + eps )
    y[m, h] = bf16_rne( x[m, h] * r[m] * w[h] )

exact in double before the one rounding to bf16.
"""
from __future__ import annotations

import numpy as np

from oracle import oracle as orc


def _widen(a):
    a = np.asarray(a)
    return orc.bf16_to_double(a) if a.dtype == np.uint16 else a.astype(np.float64)


def rmsnorm(X, w, eps: float):
    """X: float32 [M, H] or uint16 bf16 bits; w: float32 [H] or bf16 bits.
    Returns (r double [M], y_exact double [M, H], y uint16 bf16 bits [M, H])."""
    x = _widen(X)
    wd = _widen(w)
    H = x.shape[1]
    ms = np.sum(x * x, axis=1) / H
    r = 1.0 / np.sqrt(ms + float(np.float32(eps)))
    y = x * r[:, None] * wd[None, :]
    return r, y, orc.round_bf16(y)
