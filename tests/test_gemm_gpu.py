"""bi_gemm_bf16 on the GPU against the CPU oracle, and its M-invariance.

Parity: within one bf16 ULP of the exact product (plus the f32-accumulation
floor where the result nearly cancels) on shapes that span several 128x256
tiles with ragged M and N tails; bit-exact where every partial sum is exact
in f32 (integer grid, identity weight).  Invariance: every row of every M in
the sweep is byte-identical to the same row computed in other batches, at
any row position inside the 128-row tile."""
import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def gemm(bi, A_bits, B_bits):
    import torch
    a = gu.dev_bf16(A_bits)
    b = gu.dev_bf16(B_bits)
    c = bi.gemm_bf16(a, b)
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    return gu.host_bf16_bits(c)


def check_close(orc, C_bits, A, B, rows=None):
    acc, absacc, ref = orc.gemm_bf16(A, B, rows=rows)
    got = orc.bf16_to_double(C_bits if rows is None else C_bits[np.asarray(rows)])
    K = A.shape[1]
    tol = gu.gemm_tol(acc, absacc, K)
    bad = np.abs(got - acc) > tol
    assert not bad.any(), f"{bad.sum()} elements off; worst {np.max(np.abs(got - acc) / tol)} x tol"
    # and within one ULP of the correctly rounded result, in ordinal terms
    d = np.abs(orc.ord_bf16(C_bits.ravel() if rows is None else C_bits[np.asarray(rows)].ravel())
               - orc.ord_bf16(ref.ravel()))
    return d


@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (5, 272, 128), (130, 512, 192), (257, 528, 320),
                                   (384, 256, 1024)])
def test_gemm_parity_small(bi, orc, M, N, K):
    A = synth.gemm_a(10, M, K, layer=M)
    B = synth.gemm_b(10, N, K, layer=N)
    C = gemm(bi, A, B)
    d = check_close(orc, C, A, B)
    assert np.mean(d == 0) > 0.97


def test_gemm_integer_grid_exact(bi, orc):
    """Every partial sum is an exact f32 value: the result must equal the
    correctly rounded exact product bit for bit."""
    g = np.random.default_rng(3)
    M, N, K = 300, 512, 4096
    A = synth.bf16_bits_exact((g.integers(-2, 3, (M, K)) * 2.0 ** -3).astype(np.float32))
    B = synth.bf16_bits_exact((g.integers(-1, 2, (N, K)) * 2.0 ** -3).astype(np.float32))
    C = gemm(bi, A, B)
    rows = [0, 1, 127, 128, 255, 299]
    _, _, ref = orc.gemm_bf16(A, B, rows=rows)
    assert np.array_equal(C[rows], ref)


def test_gemm_identity(bi, orc):
    M, K = 200, 256
    A = synth.gemm_a(11, M, K)
    B = np.zeros((K, K), np.uint16)
    B[np.arange(K), np.arange(K)] = 0x3F80
    C = gemm(bi, A, B)
    assert np.array_equal(orc.bf16_to_double(C), orc.bf16_to_double(A))


def test_gemm_full_size_sampled(bi, orc):
    """M=4096, N=K=4096 (the benchmark's launch configuration): sampled rows
    against the oracle (every column)."""
    M, N, K = 4096, 4096, 4096
    A = synth.gemm_a(12, M, K)
    B = synth.gemm_b(12, N, K)
    C = gemm(bi, A, B)
    rows = [0, 127, 128, 2049, 4095]
    d = check_close(orc, C, A, B, rows=rows)
    assert np.mean(d == 0) > 0.97


def test_gemm_m_invariance_sweep(bi, orc):
    """Every row at M in {1,19,64,65,75,128,1024,2560,4096,8192} is
    byte-identical to the same row of the M=8192 product; sampled rows also
    equal their M=1 solo products.  At M = 2560 and 4096 the tiles of the
    last partial wave run as 128-column halves (N = 128 tensor-core steps),
    so those rows also check that the instruction width does not change the
    bits.  Self-counting: the number of compared rows is the sum of the M
    values plus the solo samples."""
    N, K = 4096, 4096
    Mmax = 8192
    A = synth.gemm_a(13, Mmax, K)
    B = synth.gemm_b(13, N, K)
    full = gemm(bi, A, B)
    compared = 0
    for M in (1, 19, 64, 65, 75, 128, 1024, 2560, 4096, 8192):
        C = gemm(bi, A[:M], B)
        assert C.tobytes() == full[:M].tobytes(), f"rows differ at M={M}"
        compared += M
    solo_rows = [0, 1, 63, 64, 127, 128, 129, 1000, 2559, 4095, 8191]
    for r in solo_rows:
        C = gemm(bi, A[r:r + 1], B)
        assert C.tobytes() == full[r:r + 1].tobytes(), f"row {r} solo differs"
        compared += 1
    assert compared == 1 + 19 + 64 + 65 + 75 + 128 + 1024 + 2560 + 4096 + 8192 + len(solo_rows)
    check_close(orc, full, A, B, rows=[0, 8191])


def test_gemm_row_position_invariance(bi):
    """A 19-row request placed at different offsets inside a batch (so its
    rows land on different tensor-memory lanes and tiles) gives the same
    bytes."""
    N, K = 512, 2048
    req = synth.gemm_a(14, 19, K)
    B = synth.gemm_b(14, N, K)
    solo = gemm(bi, req, B)
    other = synth.gemm_a(15, 400, K)
    for off in (0, 1, 37, 109, 127, 128, 200, 381):
        batch = np.concatenate([other[:off], req, other[off:]])
        C = gemm(bi, batch, B)
        assert C[off:off + 19].tobytes() == solo.tobytes(), f"offset {off}"
