"""Oracle for the grouped expert projection (TEST INFRASTRUCTURE ONLY:
imported by the test suite and the benchmark's CPU-baseline leg, never by
the library; it shares no code with it).

Source: "diag(MODEL-MM-QWEN4-EXP): the MoE expert selections DIFFER, and a
third of the boundaries are exact bf16 ties", section "Why a value tap could
never have said this": after the router picks k experts per token, each
token-slot's row goes through its expert's weights ("the assembled per-slot
expert outputs"), and that grouped expert GEMM -- whose per-expert row counts
change with the batch -- is where the run-to-run difference grows.  Read here
with bf16 experts (the pages' experts are quantised; that format is out of
scope): per slot j of token m,

    Y[m, j, n] = bf16_rne( sum_k X[m, k] * W[ids[m, j], n, k] )

exact in double before the one rounding, and the combined row

    out[m, n] = bf16_rne( sum_j weights[m, j] * Y[m, j, n] )

also exact in double.  Each step reuses the plain oracle's bf16 GEMM on one
row (oracle.gemm_bf16) and numpy double arithmetic; nothing is blocked or
reordered.
"""
from __future__ import annotations

import numpy as np

from oracle import oracle as orc


def expert_outputs(X, ids, W, rows=None):
    """X: uint16 bf16 bits [M, K]; ids: int [M, k]; W: uint16 bf16 bits
    [E, N, K].  Returns (acc double [R, k, N], absacc double [R, k, N],
    Y uint16 bf16 bits [R, k, N]) for the rows R (all rows by default)."""
    X = np.asarray(X, np.uint16)
    ids = np.asarray(ids)
    W = np.asarray(W, np.uint16)
    rows = np.arange(X.shape[0]) if rows is None else np.asarray(rows)
    k = ids.shape[1]
    N = W.shape[1]
    acc = np.empty((len(rows), k, N))
    absacc = np.empty((len(rows), k, N))
    Y = np.empty((len(rows), k, N), np.uint16)
    for r, m in enumerate(rows):
        for j in range(k):
            a, aa, y = orc.gemm_bf16(X[m:m + 1], W[int(ids[m, j])])
            acc[r, j], absacc[r, j], Y[r, j] = a[0], aa[0], y[0]
    return acc, absacc, Y


def combine(Y, weights):
    """Y: uint16 bf16 bits [R, k, N]; weights: float32 [R, k].  Returns
    (acc double [R, N], absacc double [R, N], out uint16 bf16 bits [R, N]):
    the weighted sum over the k slots, exact in double, rounded once."""
    y = orc.bf16_to_double(np.asarray(Y, np.uint16))
    w = np.asarray(weights, np.float64)[:, :, None]
    acc = np.sum(w * y, axis=1)
    absacc = np.sum(np.abs(w * y), axis=1)
    return acc, absacc, orc.round_bf16(acc)
