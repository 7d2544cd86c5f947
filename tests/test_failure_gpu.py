"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes gives up, the sticky device error word reports BI_ERR_TIMEOUT to
the host, reading it clears it, and the context keeps working."""
import time

import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(bi, orc):
    import torch
    assert bi.bi_get_last_device_error() == bi.BI_OK            # start clean
    t = time.perf_counter()
    assert bi.bi_selftest_wait_timeout(20000) == bi.BI_OK       # 20 ms bound
    assert bi.bi_get_last_device_error() == bi.BI_ERR_TIMEOUT
    elapsed = time.perf_counter() - t
    assert 0.015 < elapsed < 5.0
    assert bi.bi_get_last_device_error() == bi.BI_OK            # read clears it
    # the context is usable: a normal router call still matches the oracle
    X = synth.tokens(50, 0, 0, 8, 256)
    W = synth.router_weights(50, 0, 64, 256)
    out = bi.router_topk(gu.dev_f32(X), gu.dev_f32(W), 4, "f32")
    torch.cuda.synchronize()
    sel = orc.selection_from_logits(out["logits"].cpu().numpy(), 4)
    assert np.array_equal(out["ids"].cpu().numpy(), sel["ids"])
    assert bi.bi_get_last_device_error() == bi.BI_OK


def test_selftest_rejects_bad_limits(bi):
    assert bi.bi_selftest_wait_timeout(0) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_selftest_wait_timeout(2000001) == bi.BI_ERR_INVALID_ARG


def _every_kernel(bi):
    """One small call per kernel family of the library, each returning its
    output tensors: the cluster router, the split router and its staged-gate
    selection, the persistent router, the dense and grouped tensor-core
    GEMMs, RMSNorm in one chunk and in several, and prefill attention with
    one head and two heads to a block and with a context past the first key
    chunk."""
    import torch
    dev = "cuda"
    H, E, k = 2048, 256, 8
    W = synth.device_normal((E, H), 901, 0.02, torch.float32, dev)
    w_sg = synth.device_normal((H,), 902, 0.02, torch.float32, dev)
    X4 = synth.device_normal((4, H), 903, 1.0, torch.float32, dev)
    X300 = synth.device_normal((300, H), 904, 1.0, torch.float32, dev)
    X2k = synth.device_normal((2048, H), 905, 1.0, torch.float32, dev)
    A = synth.device_normal((256, 1024), 906, 1.0, torch.bfloat16, dev)
    B = synth.device_normal((512, 1024), 907, 0.05, torch.bfloat16, dev)
    Xm = synth.device_normal((64, 256), 908, 1.0, torch.bfloat16, dev)
    Wm = synth.device_normal((8, 256, 256), 909, 0.05, torch.bfloat16, dev)
    ids = torch.stack([torch.randperm(8, generator=torch.Generator().manual_seed(910 + i))[:2]
                       for i in range(64)]).to(torch.int32).to(dev)
    wts = torch.full((64, 2), 0.5, dtype=torch.float32, device=dev)
    Xn = synth.device_normal((8000, H), 911, 1.0, torch.float32, dev)
    wn = synth.device_normal((H,), 912, 1.0, torch.float32, dev)

    def attn(seed, q_lens, prefix, heads, kv_heads):
        qo, ko = synth.attention_offsets(q_lens, prefix)
        q, kk, v = (gu.dev_bf16(a) for a in synth.attention_inputs(seed, qo[-1], ko[-1], heads, kv_heads))
        return lambda: list(bi.attention_prefill(q, kk, v, qo, ko, 0.0883883))

    def router(x):
        return lambda: [bi.router_topk(x, W, k)[n] for n in ("logits", "ids", "weights")]

    def gated(x):
        return lambda: [bi.router_gate_topk(x, W, w_sg, k)[n] for n in ("logits", "ids", "gate_dot")]

    return [
        ("router cluster", router(X4)),
        ("router split", router(X300)),
        ("router split, staged gate", gated(X300[:256])),
        ("router persistent", gated(X2k)),
        ("gemm", lambda: [bi.gemm_bf16(A, B)]),
        ("grouped gemm", lambda: list(bi.moe_expert_gemm(Xm, ids, wts, Wm).values())),
        ("rmsnorm", lambda: list(bi.rmsnorm(X300, wn, 1e-6))),
        ("rmsnorm chunked", lambda: list(bi.rmsnorm(Xn, wn, 1e-6))),
        ("attention, head pairs", attn(913, (300, 200), (0, 150), 16, 2)),
        ("attention, one head", attn(914, (200, 70), (100, 0), 3, 1)),
        ("attention, past a key chunk", attn(915, (32,), (8300,), 4, 2)),
    ]


def test_every_kernel_drains_after_a_wait_ran_out(bi):
    """With a timeout already in the error word, a wait of any kernel that is
    not satisfied within its first polls gives up (and its block then lets
    its own copies and tensor-core operations finish before it frees its
    tensor memory and exits): every call still ends, the word reads
    BI_ERR_TIMEOUT, and afterwards every call gives its bytes from before
    again, so the context, its shared and tensor memory included, is
    intact."""
    import torch
    calls = _every_kernel(bi)
    ref = {name: [t.clone() for t in fn()] for name, fn in calls}
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == bi.BI_OK
    assert bi.bi_selftest_wait_timeout(1000) == bi.BI_OK        # the word now holds a timeout
    t = time.perf_counter()
    for _, fn in calls:
        fn()
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t
    assert bi.bi_get_last_device_error() == bi.BI_ERR_TIMEOUT
    assert elapsed < 60.0
    for name, fn in calls:
        got = fn()
        torch.cuda.synchronize()
        for a, b in zip(ref[name], got):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name
    assert bi.bi_get_last_device_error() == bi.BI_OK
