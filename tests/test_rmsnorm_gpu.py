"""bi_rmsnorm on the GPU: within one bf16 ULP of the exact oracle, bit for
bit equal to the f32 restatement of its documented order (the contract
sum of squares from oracle/contract.c, then IEEE single-precision divide,
square root and products, each rounded once), and byte-identical per row
whatever the batch ("The Illusion of Determinism in Disaggregated
Inference", section "The physics of the cascade")."""
import numpy as np
import pytest

from oracle import contract
from oracle import oracle as orc
from oracle import rmsnorm as ref
from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

EPS = 1e-6


def run(bi, X, w):
    import torch
    x = gu.dev_f32(X) if X.dtype == np.float32 else gu.dev_bf16(X)
    wd = gu.dev_f32(w) if w.dtype == np.float32 else gu.dev_bf16(w)
    y, r = bi.rmsnorm(x, wd, EPS)
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    return gu.host_bf16_bits(y), gu.host(r)


def f32_restatement(X, w):
    """The documented order in numpy float32 (IEEE: every operation rounded
    once), with the contract's sum of squares."""
    xf = orc.bf16_to_double(X).astype(np.float32) if X.dtype == np.uint16 else X
    wf = orc.bf16_to_double(w).astype(np.float32) if w.dtype == np.uint16 else w
    H = X.shape[1]
    ss = np.array([contract.router_logits(X[m:m + 1], X[m:m + 1])[0, 0] for m in range(X.shape[0])], np.float32)
    r = np.float32(1.0) / np.sqrt(ss / np.float32(H) + np.float32(EPS))
    y = (xf * r[:, None]) * wf[None, :]
    return r, orc.round_bf16(y.astype(np.float64))


# short, ragged and long rows, f32 and bf16; a block's share of rows staged
# in several chunks (M = 8000: 53 rows a block, 27 at a time; H = 32768: one
# 128 KB row at a time)
@pytest.mark.parametrize("M,H,dt", [(1, 2048, "f32"), (37, 264, "f32"), (300, 2048, "f32"), (19, 8, "f32"),
                                    (50, 2048, "bf16"), (33, 1032, "bf16"), (2000, 3328, "f32"),
                                    (45, 3336, "f32"), (1300, 6656, "bf16"), (21, 6664, "bf16"),
                                    (8000, 2048, "f32"), (400, 32768, "f32"), (700, 32768, "bf16")])
def test_rmsnorm_parity_and_order(bi, M, H, dt):
    X = synth.tokens(70, 0, M, M, H)
    w = (1.0 + 0.1 * synth.shared_gate_weights(70, M, H)).astype(np.float32)
    if dt == "bf16":
        X, w = synth.to_bf16_bits(X), synth.to_bf16_bits(w)
    y, r = run(bi, X, w)
    r_ex, y_ex, _ = ref.rmsnorm(X, w, EPS)
    assert np.all(np.abs(r - r_ex) <= (H / 32 + 8) * gu.U * r_ex)
    assert np.all(np.abs(orc.bf16_to_double(y) - y_ex) <= gu.bf16_ulp(y_ex) + 1e-30)
    r_c, y_c = f32_restatement(X, w)
    assert r.view(np.uint32).tobytes() == r_c.view(np.uint32).tobytes()
    assert np.array_equal(y, y_c)


def test_rmsnorm_rows_invariant_to_batch(bi):
    H = 2048
    w = (1.0 + 0.1 * synth.shared_gate_weights(71, 0, H)).astype(np.float32)
    req = synth.tokens(71, 0, 0, 19, H)
    pool = synth.tokens(71, 0, 1, 4096, H)
    y0, r0 = run(bi, req, w)
    n = 0
    for M, off in ((20, 1), (64, 0), (700, 300), (4096, 4077)):
        X = np.concatenate([pool[:off], req, pool[off:M - 19]])
        y, r = run(bi, X, w)
        assert y[off:off + 19].tobytes() == y0.tobytes() and r[off:off + 19].tobytes() == r0.tobytes(), M
        n += 1
    assert n == 4
