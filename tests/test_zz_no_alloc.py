"""bi_router_topk_noalloc: the router for callers that cannot provide device
memory beyond their inputs and outputs (a plugin or embedded runtime handed
device pointers but no allocator; bi_router_topk needs a caller workspace for
large batches).  Its partial sums live in a fixed array compiled into the
library.

Checked through the C ABI against bi_router_topk on the same inputs, on two
calls in a row (the array keeps the previous call's contents, which must not
leak into the next), on two calls queued back to back on one stream with no
host synchronisation between them, with the device's free memory unchanged
across a call, and for the rejection of a problem too large for the array.
This file is collected last on purpose; it passes alone in a fresh process
and after the rest of the suite."""
import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

FIELDS = ("logits", "ids", "weights", "margin", "margin_ulps")


def outputs(torch, M, E, k, logit_dtype):
    dev = "cuda"
    return {
        "logits": torch.full((M, E), 7.0, dtype=torch.float32 if logit_dtype == "f32" else torch.bfloat16, device=dev),
        "ids": torch.full((M, k), -1, dtype=torch.int32, device=dev),
        "weights": torch.full((M, k), 7.0, dtype=torch.float32, device=dev),
        "margin": torch.full((M,), 7.0, dtype=torch.float32, device=dev),
        "margin_ulps": torch.full((M,), -1, dtype=torch.int32, device=dev),
    }


def call(bi, fn, x, w, k, logit_dtype):
    import torch
    M, H = x.shape
    E = w.shape[0]
    o = outputs(torch, M, E, k, logit_dtype)
    ind = bi.BI_F32 if x.dtype == torch.float32 else bi.BI_BF16
    ld = bi.BI_F32 if logit_dtype == "f32" else bi.BI_BF16
    args = (x, w, ind, ld, M, H, E, k, o["logits"], o["ids"], o["weights"], o["margin"], o["margin_ulps"])
    if fn is bi.bi_router_topk:
        fn(*args, workspace=bi.router_workspace(M, E))
    else:
        fn(*args)
    torch.cuda.synchronize()
    return host(torch, o)


def host(torch, o):
    return {f: o[f].contiguous().view(torch.uint8).cpu().numpy().tobytes() if o[f].dtype == torch.bfloat16
            else o[f].cpu().numpy() for f in FIELDS}


CASES = [(1, 2048, 256, 8, "f32"), (19, 2048, 256, 8, "f32"), (64, 2048, 256, 8, "f32"),
         (5, 256, 64, 4, "f32"), (256, 256, 64, 4, "f32"), (16, 2048, 1024, 32, "f32")]


@pytest.mark.parametrize("M,H,E,k,ld", CASES)
def test_noalloc_matches_router_topk_twice(bi, M, H, E, k, ld):
    assert bi.bi_get_last_device_error() == 0
    for call_no in range(2):                      # two calls in a row, different inputs
        X = synth.tokens(60 + call_no, 0, M, M, H)
        W = synth.router_weights(60 + call_no, M, E, H)
        x, w = gu.dev_f32(X), gu.dev_f32(W)
        ref = call(bi, bi.bi_router_topk, x, w, k, ld)
        got = call(bi, bi.bi_router_topk_noalloc, x, w, k, ld)
        for f in FIELDS:
            a, b = np.asarray(ref[f]), np.asarray(got[f])
            assert a.tobytes() == b.tobytes(), f"{f} differs on call {call_no} (tolerance: identical bytes)"
    assert bi.bi_get_last_device_error() == 0


def test_noalloc_bf16_tie_grid_twice(bi):
    for call_no in range(2):
        X, W = synth.tie_heavy_call(0, call_no, n_tokens=5)
        x, w = gu.dev_bf16(X), gu.dev_bf16(W)
        ref = call(bi, bi.bi_router_topk, x, w, 10, "bf16")
        got = call(bi, bi.bi_router_topk_noalloc, x, w, 10, "bf16")
        for f in FIELDS:
            assert np.asarray(ref[f]).tobytes() == np.asarray(got[f]).tobytes(), f


def test_noalloc_rejects_problems_beyond_its_array(bi):
    import torch
    E, H, k = 256, 2048, 8
    limit_m = bi.BI_NOALLOC_SCRATCH_BYTES // (16 * 4 * E)      # 64 tokens at E = 256
    for M, want in ((limit_m, bi.BI_OK), (limit_m + 1, bi.BI_ERR_UNSUPPORTED_SHAPE)):
        x = torch.zeros((M, H), dtype=torch.float32, device="cuda")
        w = torch.zeros((E, H), dtype=torch.float32, device="cuda")
        o = outputs(torch, M, E, k, "f32")
        st = bi.bi_router_topk_noalloc(x, w, bi.BI_F32, bi.BI_F32, M, H, E, k, o["logits"], o["ids"],
                                       None, None, None, check=False)
        assert st == want, (M, st)
    torch.cuda.synchronize()


def test_noalloc_back_to_back_on_one_stream(bi):
    """Two calls with different inputs and outputs queued on one stream with
    no synchronisation between them (the second call's kernels may start
    while the first call's selection still reads the shared array; the
    array is written only after each kernel's wait on its predecessor): each
    output equals its own bi_router_topk result."""
    import torch
    M, H, E, k = 48, 2048, 256, 8
    xs = [gu.dev_f32(synth.tokens(70 + i, 0, 0, M, H)) for i in range(2)]
    ws = [gu.dev_f32(synth.router_weights(70 + i, 0, E, H)) for i in range(2)]
    refs = [call(bi, bi.bi_router_topk, xs[i], ws[i], k, "f32") for i in range(2)]
    outs = [outputs(torch, M, E, k, "f32") for _ in range(2)]
    torch.cuda.synchronize()
    for i in range(2):
        o = outs[i]
        bi.bi_router_topk_noalloc(xs[i], ws[i], bi.BI_F32, bi.BI_F32, M, H, E, k, o["logits"], o["ids"],
                                  o["weights"], o["margin"], o["margin_ulps"])
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    for i in range(2):
        got = host(torch, outs[i])
        for f in FIELDS:
            assert np.asarray(got[f]).tobytes() == np.asarray(refs[i][f]).tobytes(), (i, f)


def test_noalloc_call_leaves_free_memory_unchanged(bi):
    """After a first call on the device, a call allocates nothing: the
    device's free memory is the same before and after it."""
    import torch
    M, H, E, k = 64, 2048, 256, 8
    x = gu.dev_f32(synth.tokens(72, 0, 0, M, H))
    w = gu.dev_f32(synth.router_weights(72, 0, E, H))
    o = outputs(torch, M, E, k, "f32")
    args = (x, w, bi.BI_F32, bi.BI_F32, M, H, E, k, o["logits"], o["ids"], o["weights"], o["margin"],
            o["margin_ulps"])
    bi.bi_router_topk_noalloc(*args)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        bi.bi_router_topk_noalloc(*args)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
