"""bi_moe_expert_gemm on the GPU: the grouped expert projection against the
oracle (oracle/moe.py), and its invariance: a token's per-slot outputs and
combined row are byte-identical whatever else shares the batch, although
every expert's row count -- and so the grouping, the padding and the tile a
row lands in -- changes with the batch ("diag(MODEL-MM-QWEN4-EXP): ...",
section "Why a value tap could never have said this")."""
import numpy as np
import pytest

from oracle import moe
from oracle import oracle as orc
from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def routed(seed, M, E, k):
    """Distinct experts per token (the router's top-k), skewed so that some
    experts get many rows and some none, and dyadic-ish weights summing to 1."""
    g = np.random.default_rng(seed)
    p = g.dirichlet(np.full(E, 0.3))
    ids = np.stack([g.choice(E, k, replace=False, p=p) for _ in range(M)]).astype(np.int32)
    w = g.random((M, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    return ids, w.astype(np.float32)


def experts(seed, E, N, K):
    return np.stack([synth.gemm_b(seed, N, K, layer=e) for e in range(E)])


def run(bi, X, ids, w, W):
    import torch
    out = bi.moe_expert_gemm(gu.dev_bf16(X), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                             gu.dev_bf16(W))
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    return gu.host_bf16_bits(out["Y"]), gu.host_bf16_bits(out["out"])


def check_against_oracle(X, ids, w, W, Y, out, rows=None):
    rows = np.arange(X.shape[0]) if rows is None else np.asarray(rows)
    K = X.shape[1]
    acc, absacc, _ = moe.expert_outputs(X, ids, W, rows=rows)
    got = orc.bf16_to_double(Y[rows])
    assert np.all(np.abs(got - acc) <= gu.gemm_tol(acc, absacc, K)), "per-slot outputs off"
    # the combine, against the oracle's combine of the GPU's own per-slot rows
    cacc, cabs, _ = moe.combine(Y[rows], w[rows])
    k = ids.shape[1]
    tol = gu.bf16_ulp(cacc) + (k + 1) * gu.U * cabs
    assert np.all(np.abs(orc.bf16_to_double(out[rows]) - cacc) <= tol), "combined rows off"


@pytest.mark.parametrize("M,k,E,N,K", [(1, 2, 4, 256, 64), (37, 4, 8, 272, 192), (300, 2, 2, 512, 256),
                                       (129, 8, 64, 128, 128)])
def test_moe_parity(bi, M, k, E, N, K):
    """Ragged N (272), experts with several 128-row tiles (E=2, 300 tokens),
    experts with no rows (E=64, skewed routing), single tokens."""
    ids, w = routed(M + E, M, E, k)
    X = synth.gemm_a(60, M, K, layer=M)
    W = experts(61, E, N, K)
    Y, out = run(bi, X, ids, w, W)
    check_against_oracle(X, ids, w, W, Y, out)


def test_moe_integer_grid_exact(bi):
    g = np.random.default_rng(7)
    M, k, E, N, K = 50, 3, 5, 256, 256
    ids, w = routed(7, M, E, k)
    X = synth.bf16_bits_exact((g.integers(-2, 3, (M, K)) * 0.25).astype(np.float32))
    W = synth.bf16_bits_exact((g.integers(-1, 2, (E, N, K)) * 0.5).astype(np.float32))
    Y, _ = run(bi, X, ids, w, W)
    _, _, Yref = moe.expert_outputs(X, ids, W)
    assert np.array_equal(Y, Yref)


def test_moe_identity_experts(bi):
    """Expert e = the identity scaled by 2^-e: every slot returns its token's
    row times an exact power of two."""
    M, k, E, K = 40, 3, 4, 128
    ids, w = routed(8, M, E, k)
    X = synth.gemm_a(62, M, K)
    W = np.zeros((E, K, K), np.uint16)
    for e in range(E):
        W[e][np.arange(K), np.arange(K)] = synth.bf16_bits_exact(np.array([2.0 ** -e], np.float32))[0]
    Y, _ = run(bi, X, ids, w, W)
    xv = orc.bf16_to_double(X)
    for j in range(k):
        want = orc.round_bf16(xv * (2.0 ** -ids[:, j])[:, None])
        assert np.array_equal(Y[:, j], want)


def test_moe_request_invariant_to_batch(bi):
    """A 19-token request solo and inside batches of 64, 300 and 2000 tokens
    (placed first, in the middle, last): its per-slot rows and combined rows
    are byte-identical, although the experts' row counts all change."""
    E, k, N, K = 16, 4, 256, 512
    W = experts(63, E, N, K)
    ids_r, w_r = routed(9, 19, E, k)
    X_r = synth.gemm_a(64, 19, K)
    Y0, out0 = run(bi, X_r, ids_r, w_r, W)
    n = 0
    for M, off in ((64, 0), (300, 140), (2000, 1981)):
        ids_o, w_o = routed(10 + M, M - 19, E, k)
        X_o = synth.gemm_a(65, M - 19, K, layer=M)
        X = np.concatenate([X_o[:off], X_r, X_o[off:]])
        ids = np.concatenate([ids_o[:off], ids_r, ids_o[off:]])
        w = np.concatenate([w_o[:off], w_r, w_o[off:]])
        Y, out = run(bi, X, ids, w, W)
        assert Y[off:off + 19].tobytes() == Y0.tobytes(), f"per-slot rows differ at M={M}"
        assert out[off:off + 19].tobytes() == out0.tobytes(), f"combined rows differ at M={M}"
        n += 1
    assert n == 3


def test_moe_full_size_sampled(bi):
    """M=4096 tokens, top-8 of 256 experts, N=1024, K=2048 (the benchmark's
    launch): sampled token rows against the oracle."""
    M, k, E, N, K = 4096, 8, 256, 1024, 2048
    ids, w = routed(11, M, E, k)
    X = synth.gemm_a(66, M, K)
    W = experts(67, E, N, K)
    Y, out = run(bi, X, ids, w, W)
    check_against_oracle(X, ids, w, W, Y, out, rows=[0, 1, 2047, 4095])


def test_moe_bad_id_sets_the_error_word(bi):
    import torch
    M, k, E, N, K = 8, 2, 4, 256, 64
    ids, w = routed(12, M, E, k)
    ids[3, 1] = E + 5                                      # out of range
    X = synth.gemm_a(68, M, K)
    W = experts(69, E, N, K)
    o = bi.moe_expert_gemm(gu.dev_bf16(X), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), gu.dev_bf16(W))
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == bi.BI_ERR_INVALID_ARG
    assert bi.bi_get_last_device_error() == 0              # read and cleared
    Y = gu.host_bf16_bits(o["Y"])
    keep = np.ones((M, k), bool)
    keep[3, 1] = False
    acc, absacc, _ = moe.expert_outputs(X, np.where(keep, ids, 0), W)
    got = orc.bf16_to_double(Y)
    tol = gu.gemm_tol(acc, absacc, K)
    assert np.all((np.abs(got - acc) <= tol)[keep])        # every other slot is still right
