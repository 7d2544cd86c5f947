"""Helpers shared by the GPU tests: moving synthetic inputs to the device and
the tolerances the parity tests use (each derived in its docstring)."""
from __future__ import annotations

import numpy as np

U = 2.0 ** -24     # unit roundoff of binary32


def dev_f32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def host_bf16_bits(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def router_logit_tol(absdot: np.ndarray) -> np.ndarray:
    """F32 router logits: |gpu - exact| <= 2e-6 * sum_h |x_h w_h|.

    The stated 2e-6 relative tolerance is read relative to the dot
    product's own scale sum|x w| (a plain relative error is unbounded where
    a logit is near zero).  The rigorous bound for this reduction order is
    (H/16 + 5) * 2^-24 * sum|x w| (a chain of H/16 roundings, four tree
    levels, one final rounding); typical errors are far below both."""
    return 2e-6 * absdot


def softmax_tol(widened_logits_row_gaps: np.ndarray, k: int) -> np.ndarray:
    """Relative tolerance of an f32 weight w_j = exp(d_j)/sum exp(d_i) with
    d_j = l_j - l_0 rounded once: |d|*u (rounding of d, amplified by exp),
    2 ulps of expf, k roundings in the sum, one in the division; doubled for
    numerator and denominator."""
    return (np.abs(widened_logits_row_gaps) + k + 8) * 2.0 * U


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significant bits)."""
    a = np.abs(v).astype(np.float64)
    a = np.where(a == 0, 2.0 ** -126, a)
    e = np.floor(np.log2(a))
    return np.exp2(np.maximum(e - 7, -133))


def gemm_tol(ref: np.ndarray, absacc: np.ndarray, K: int) -> np.ndarray:
    """bf16 GEMM: one bf16 ULP of the exact result, plus an absolute floor
    (K/8) * 2^-24 * sum_k |a_k b_k| for f32 accumulation over K/16
    tensor-core steps (with slack for rounding inside a step), which only
    matters where the result nearly cancels."""
    return bf16_ulp(ref) + (K / 8.0) * U * absacc
