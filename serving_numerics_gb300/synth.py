"""Seeded synthetic inputs shaped like the workloads on the source pages.

This module only draws random numbers and lays them out; it holds none of
the method's arithmetic.  Both the CUDA path and the CPU oracle are fed
from here.  bf16 tensors are returned as numpy uint16 bit patterns.

Workloads:
  * tiny m-scan       H=256,  E=64,  k=4,  W ~ N(0, 0.02^2) f32, X ~ N(0,1) f32
  * 256-expert router H=2048, E=256, k=8,  W, w_sg ~ N(0, 0.02^2), X ~ N(0,1), per layer
  * tie-heavy bf16    H=2048, E=512, k=10, X, W on the grid {-1, +1} * 2^-8 (bf16-exact)
  * projection GEMM   A [M,K], B [N,K] ~ N(0,1)/64 rounded to bf16
  * mixed prefill     16 request lengths ~ U[5, 300]
"""
from __future__ import annotations

import numpy as np

# stream ids keep every (workload, layer, tensor) draw independent
_S_X, _S_W, _S_WSG, _S_A, _S_B, _S_LEN, _S_MISC, _S_ATTN = range(8)


def rng(seed: int, *path: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), *map(int, path)]))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) with torch's CPU
    conversion; returns the uint16 patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_exact(x: np.ndarray) -> np.ndarray:
    """bf16 patterns of float32 values that are already bf16-representable."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "values are not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


TINY = dict(H=256, E=64, k=4)
ROUTER256 = dict(H=2048, E=256, k=8)
TIE512 = dict(H=2048, E=512, k=10)


# ---------------------------------------------------------------- router
def router_weights(seed: int, layer: int, E: int, H: int, std: float = 0.02) -> np.ndarray:
    return (rng(seed, _S_W, layer).standard_normal((E, H)) * std).astype(np.float32)


def shared_gate_weights(seed: int, layer: int, H: int, std: float = 0.02) -> np.ndarray:
    return (rng(seed, _S_WSG, layer).standard_normal(H) * std).astype(np.float32)


def tokens(seed: int, layer: int, request: int, n: int, H: int) -> np.ndarray:
    """Hidden states of one request's n tokens at one layer, X ~ N(0,1)."""
    return rng(seed, _S_X, layer, request).standard_normal((n, H)).astype(np.float32)


def tiny_mscan(seed: int = 0, max_m: int = 96, fixed_len: int = 19):
    """Gate weights, a fixed 19-token request and a pool of co-arrival
    tokens that brings the total to at most max_m."""
    H, E = TINY["H"], TINY["E"]
    W = router_weights(seed, 0, E, H)
    req = tokens(seed, 0, 0, fixed_len, H)
    pool = tokens(seed, 0, 1, max_m - fixed_len, H)
    return W, req, pool


# ---------------------------------------------------------------- tie-heavy bf16
def grid_bf16(g: np.random.Generator, shape, q: int, p_zero: float) -> np.ndarray:
    """Integers in {-q..q} (zero with probability p_zero, else uniform over
    the non-zero values) times 2^-8, as exact bf16 patterns."""
    mag = g.integers(1, q + 1, shape)
    sign = np.where(g.random(shape) < 0.5, -1, 1)
    v = np.where(g.random(shape) < p_zero, 0, mag * sign).astype(np.float64)
    return bf16_bits_exact((v * 2.0 ** -8).astype(np.float32))


# grid parameters chosen with the oracle: with X, W in {-1, +1} * 2^-8 and
# seed 0, 78 of the 240 token-slots of the 48-call workload (32.5%) tie
# exactly at the k-boundary, against 79/240 on the page that measured it
TIE_Q = 1
TIE_PZERO = 0.0


def tie_heavy_call(seed: int, call: int, n_tokens: int = 5, q: int = TIE_Q, p_zero: float = TIE_PZERO):
    H, E = TIE512["H"], TIE512["E"]
    X = grid_bf16(rng(seed, _S_X, call), (n_tokens, H), q, p_zero)
    W = grid_bf16(rng(seed, _S_W, call), (E, H), q, p_zero)
    return X, W


# ---------------------------------------------------------------- GEMM
def gemm_a(seed: int, M: int, K: int, layer: int = 0) -> np.ndarray:
    return to_bf16_bits(rng(seed, _S_A, layer).standard_normal((M, K)).astype(np.float32) / 64)


def gemm_b(seed: int, N: int, K: int, layer: int = 0) -> np.ndarray:
    return to_bf16_bits(rng(seed, _S_B, layer).standard_normal((N, K)).astype(np.float32) / 64)


# ---------------------------------------------------------------- mixed prefill
def request_lengths(seed: int = 0, n: int = 16, lo: int = 5, hi: int = 300) -> np.ndarray:
    return rng(seed, _S_LEN).integers(lo, hi + 1, n)


# ---------------------------------------------------------------- attention
# The prefill attention workload: 16 query heads sharing 2 key/value heads of
# dimension 128 (16 x 128 = the hidden size 2048 above), 4096 query tokens
# in 8 requests of mixed length, five of them behind a cached prefix.
ATTN_HEADS, ATTN_KV_HEADS, ATTN_D = 16, 2, 128
ATTN_Q_LENS = (1024, 768, 512, 512, 384, 384, 256, 256)
ATTN_PREFIX = (0, 2048, 1024, 0, 3072, 512, 0, 1536)


def attention_offsets(q_lens, prefix):
    """(q_offsets, kv_offsets) of requests with q_lens queries after
    prefix cached tokens each: 0, then running sums."""
    q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    kv = np.concatenate([[0], np.cumsum(np.asarray(q_lens) + np.asarray(prefix))]).astype(np.int32)
    return q, kv


def attention_inputs(seed: int, Tq: int, Tkv: int, heads: int, kv_heads: int, D: int = ATTN_D):
    """q [Tq, heads, D], k and v [Tkv, kv_heads, D] as bf16 bit patterns of
    standard normal draws."""
    g = rng(seed, _S_ATTN)
    q = to_bf16_bits(g.standard_normal((Tq, heads, D)).astype(np.float32))
    k = to_bf16_bits(g.standard_normal((Tkv, kv_heads, D)).astype(np.float32))
    v = to_bf16_bits(g.standard_normal((Tkv, kv_heads, D)).astype(np.float32))
    return q, k, v


# ---------------------------------------------------------------- device pools
def device_normal(shape, seed: int, std: float, dtype, device="cuda"):
    """Seeded normal draws made on the GPU with torch's generator, for
    benchmark pools too large to draw on the host quickly."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(dtype)
