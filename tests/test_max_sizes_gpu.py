"""The largest shapes the entry points accept (include/bi.h: H = BI_MAX_H,
E = BI_MAX_E, k = BI_MAX_K): the router (matrix-vector twin and tiles, f32
and bf16 inputs), the shared gate fused into it (rows too long to stage, so
read from device memory) and RMSNorm hold the reduction contract bit for bit
on sampled rows, and the selection is the oracle's selection of the returned
logits ("batch changed the model's mind", section "The fix: m-invariant
twins"; "The Illusion of Determinism in Disaggregated Inference", section
"The physics of the cascade")."""
import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

H_MAX, E_MAX, K_MAX = 32768, 1024, 32


@pytest.mark.parametrize("M,dt", [(3, "f32"), (100, "f32"), (70, "bf16")])
def test_router_at_max_h_e_k(bi, orc, M, dt):
    import torch
    from oracle import contract
    X = synth.tokens(61, 0, 0, M, H_MAX)
    W = synth.router_weights(61, M, E_MAX, H_MAX)
    if dt == "bf16":
        X, W = synth.to_bf16_bits(X), synth.to_bf16_bits(W)
        x, w = gu.dev_bf16(X), gu.dev_bf16(W)
    else:
        x, w = gu.dev_f32(X), gu.dev_f32(W)
    out = bi.router_topk(x, w, K_MAX)
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    lg = gu.host(out["logits"])
    rows = np.arange(M) if M <= 4 else np.array([0, 31, 32, 63, M - 1])
    want = contract.router_logits(X[rows], W)
    assert lg[rows].view(np.uint32).tobytes() == want.view(np.uint32).tobytes()
    sel = orc.selection_from_logits(lg, K_MAX)
    assert np.array_equal(gu.host(out["ids"]), sel["ids"])
    assert np.array_equal(gu.host(out["margin_ulps"]), sel["margin_ulps"])


def test_fused_gate_at_max_h(bi):
    import torch
    from oracle import contract
    M = 40
    X = synth.tokens(62, 0, 0, M, H_MAX)
    W = synth.router_weights(62, 0, 256, H_MAX)
    wsg = synth.shared_gate_weights(62, 0, H_MAX)
    out = bi.router_gate_topk(gu.dev_f32(X), gu.dev_f32(W), gu.dev_f32(wsg), 8)
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    rows = np.array([0, 17, 39])
    want = contract.router_logits(X[rows], wsg[None, :])[:, 0]
    assert gu.host(out["gate_dot"])[rows].view(np.uint32).tobytes() == want.view(np.uint32).tobytes()


def test_rmsnorm_at_max_h(bi):
    import torch
    from oracle import contract
    from oracle import oracle as o
    M, eps = 24, 1e-6
    X = synth.tokens(63, 0, 0, M, H_MAX)
    w = (1.0 + 0.1 * synth.shared_gate_weights(63, 0, H_MAX)).astype(np.float32)
    y, r = bi.rmsnorm(gu.dev_f32(X), gu.dev_f32(w), eps)
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    rows = [0, 11, 23]
    ss = np.array([contract.router_logits(X[m:m + 1], X[m:m + 1])[0, 0] for m in rows], np.float32)
    want_r = np.float32(1.0) / np.sqrt(ss / np.float32(H_MAX) + np.float32(eps))
    assert gu.host(r)[rows].view(np.uint32).tobytes() == want_r.view(np.uint32).tobytes()
    want_y = o.round_bf16(((X[rows] * want_r[:, None]) * w[None, :]).astype(np.float64))
    assert np.array_equal(gu.host_bf16_bits(y)[rows], want_y)
