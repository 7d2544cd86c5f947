"""Pins for oracle/moe.py (the grouped expert projection and the weighted
combine), each against something other than the oracle itself: one-hot
experts select input columns exactly; an integer grid has an exact product
computed here with integers; relabelling the experts leaves every slot's
output unchanged; the combine has closed forms for one slot, dyadic weights
and a zero weight."""
import numpy as np

from oracle import moe
from oracle import oracle as orc
from serving_numerics_gb300 import synth


def bf16_bits(v):
    return synth.bf16_bits_exact(np.asarray(v, np.float32))


def test_one_hot_experts_pick_columns():
    """W[e][n, :] is the unit vector of column (3e + n) mod K, so slot j of
    token m must return X[m, (3 ids[m,j] + n) mod K] exactly: this pins the
    expert index, the [N, K] orientation of each expert and the slot order."""
    g = np.random.default_rng(0)
    M, K, N, E, k = 7, 64, 16, 5, 3
    X = synth.gemm_a(1, M, K)
    W = np.zeros((E, N, K), np.uint16)
    for e in range(E):
        for n in range(N):
            W[e, n, (3 * e + n) % K] = 0x3F80                # 1.0
    ids = g.integers(0, E, (M, k))
    _, _, Y = moe.expert_outputs(X, ids, W)
    for m in range(M):
        for j in range(k):
            cols = (3 * ids[m, j] + np.arange(N)) % K
            assert np.array_equal(Y[m, j], X[m, cols])


def test_integer_grid_is_exact():
    g = np.random.default_rng(1)
    M, K, N, E, k = 5, 128, 24, 4, 2
    Xi = g.integers(-3, 4, (M, K))
    Wi = g.integers(-2, 3, (E, N, K))
    ids = g.integers(0, E, (M, k))
    acc, _, Y = moe.expert_outputs(bf16_bits(Xi * 0.25), ids, bf16_bits(Wi * 0.5))
    for m in range(M):
        for j in range(k):
            want = (Wi[ids[m, j]] @ Xi[m]).astype(np.int64) * 0.125   # exact in double; one bf16 rounding
            assert np.array_equal(acc[m, j], want)
            assert np.array_equal(Y[m, j], orc.round_bf16(want))


def test_relabelling_experts_changes_nothing():
    g = np.random.default_rng(2)
    M, K, N, E, k = 6, 64, 16, 6, 3
    X = synth.gemm_a(2, M, K)
    W = np.stack([synth.gemm_b(2, N, K, layer=e) for e in range(E)])
    ids = g.integers(0, E, (M, k))
    perm = g.permutation(E)                      # new label of expert e is perm[e]
    W2 = np.empty_like(W)
    W2[perm] = W
    _, _, Y = moe.expert_outputs(X, ids, W)
    _, _, Y2 = moe.expert_outputs(X, perm[ids], W2)
    assert np.array_equal(Y, Y2)


def test_combine_closed_forms():
    g = np.random.default_rng(3)
    R, k, N = 4, 3, 10
    Y = bf16_bits(g.integers(-16, 17, (R, k, N)) * 0.125)
    one = np.zeros((R, k), np.float32)
    one[:, 1] = 1.0
    assert np.array_equal(moe.combine(Y, one)[2], Y[:, 1])                 # a single slot of weight 1
    w = np.tile(np.array([0.25, 0.75, 0.0], np.float32), (R, 1))
    yv = orc.bf16_to_double(Y)
    assert np.array_equal(moe.combine(Y, w)[0], 0.25 * yv[:, 0] + 0.75 * yv[:, 1])   # dyadic: exact
    Y3 = Y.copy()
    Y3[:, 2] = bf16_bits(np.full((R, N), 1000.0))                         # zero weight: no effect
    assert np.array_equal(moe.combine(Y3, w)[2], moe.combine(Y, w)[2])
    assert np.array_equal(moe.combine(Y, 2 * w)[0], 2 * moe.combine(Y, w)[0])   # linear, exact doubling
