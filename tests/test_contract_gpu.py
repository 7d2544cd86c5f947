"""The router projection and the shared gate hold the documented reduction
order bit for bit: every logit and gate dot equals the CPU restatement of
the contract (oracle/contract.c: 16 partitions owning the 8-wide blocks of
every 128-wide slab, one f32 fused multiply-add chain each, a pairwise tree
of the partials), for every work split the library picks (the one-launch
cluster router at every token tile it compiles, whole tiles,
partition-split tiles, whole tiles plus a split tail, the no-allocation
entry), for f32 and bf16 inputs, and for bf16 logits (the same f32 value
rounded to nearest even once).

This is stronger than the tolerance parity of test_router_gpu.py: it pins
the order itself, which is what makes the results independent of M ("batch
changed the model's mind", section "The fix: m-invariant twins")."""
import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def gpu_logits(bi, X, W, k, logit_dtype, noalloc=False):
    import torch
    x = gu.dev_f32(X) if X.dtype == np.float32 else gu.dev_bf16(X)
    w = gu.dev_f32(W) if W.dtype == np.float32 else gu.dev_bf16(W)
    M, E = X.shape[0], W.shape[0]
    lg = torch.empty((M, E), dtype=torch.float32 if logit_dtype == "f32" else torch.bfloat16, device="cuda")
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    ind = bi.BI_F32 if X.dtype == np.float32 else bi.BI_BF16
    lod = bi.BI_F32 if logit_dtype == "f32" else bi.BI_BF16
    if noalloc:
        bi.bi_router_topk_noalloc(x, w, ind, lod, M, X.shape[1], E, k, lg, ids)
    else:
        bi.bi_router_topk(x, w, ind, lod, M, X.shape[1], E, k, lg, ids, workspace=bi.router_workspace(M, E))
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    return gu.host(lg) if logit_dtype == "f32" else gu.host_bf16_bits(lg)


# (M, H, E, k): the cluster router (M <= 112, E <= 512) at token tiles of
# 1, 2, 4, 8 and 16 rows, 2 to 32 experts per block, one-slab and ragged H
# (H = 8: a single 8-wide block); partition-split tiles one block to an SM
# (and E = 1024 at small M), two-block tiles two to an SM, whole tiles +
# split tail (E = 1024, M = 8300: group sums past 64 MiB); ragged H and E
SHAPES = [(1, 2048, 256, 8), (7, 264, 96, 5), (20, 2048, 256, 8), (33, 2048, 32, 4), (3, 8, 64, 4),
          (64, 136, 1024, 32), (100, 2048, 256, 8), (112, 2048, 512, 10), (128, 2048, 512, 10), (57, 4104, 256, 8),
          (300, 136, 64, 4), (700, 264, 256, 8), (1300, 2048, 256, 8), (1235, 128, 256, 8),
          (8300, 136, 1024, 16)]


@pytest.mark.parametrize("M,H,E,k", SHAPES)
def test_router_f32_logits_are_the_contract(bi, M, H, E, k):
    from oracle import contract
    X = synth.tokens(50, 0, M, M, H)
    W = synth.router_weights(50, M, E, H)
    got = gpu_logits(bi, X, W, k, "f32")
    want = contract.router_logits(X, W)
    assert got.view(np.uint32).tobytes() == want.view(np.uint32).tobytes(), \
        f"{np.sum(got.view(np.uint32) != want.view(np.uint32))} logits differ"


@pytest.mark.parametrize("M,H,E,k", [(5, 2048, 512, 10), (50, 2048, 512, 10), (700, 2048, 256, 8),
                                     (1400, 2048, 256, 8)])
def test_router_bf16_inputs_and_logits_are_the_contract(bi, orc, M, H, E, k):
    from oracle import contract
    X = synth.to_bf16_bits(synth.tokens(51, 0, M, M, H))
    W = synth.to_bf16_bits(synth.router_weights(51, M, E, H))
    want = contract.router_logits(X, W)
    got = gpu_logits(bi, X, W, k, "f32")
    assert got.view(np.uint32).tobytes() == want.view(np.uint32).tobytes()
    got_b = gpu_logits(bi, X, W, k, "bf16")
    want_b = orc.round_bf16(want.astype(np.float64))
    assert np.array_equal(got_b, want_b)


def test_router_noalloc_is_the_contract(bi):
    from oracle import contract
    M, H, E, k = 40, 2048, 256, 8
    X = synth.tokens(52, 0, 0, M, H)
    W = synth.router_weights(52, 0, E, H)
    got = gpu_logits(bi, X, W, k, "f32", noalloc=True)
    assert got.view(np.uint32).tobytes() == contract.router_logits(X, W).view(np.uint32).tobytes()


def test_router_full_size_sampled_rows_are_the_contract(bi):
    """M = 4096 (the benchmark's launch: two-block tiles, two to an SM):
    sampled rows across the batch."""
    from oracle import contract
    M, H, E, k = 4096, 2048, 256, 8
    X = synth.tokens(53, 0, 0, M, H)
    W = synth.router_weights(53, 0, E, H)
    got = gpu_logits(bi, X, W, k, "f32")
    rows = np.array([0, 31, 32, 1999, 3647, 3648, 3700, 4095])
    want = contract.router_logits(X[rows], W)
    assert got[rows].view(np.uint32).tobytes() == want.view(np.uint32).tobytes()


@pytest.mark.parametrize("M,H", [(1, 2048), (33, 264), (4096, 2048)])
def test_shared_gate_dot_is_the_contract(bi, M, H):
    import torch
    from oracle import contract
    X = synth.tokens(54, 0, 0, M, H)
    w = synth.shared_gate_weights(54, 0, H)
    dot, _ = bi.shared_gate(gu.dev_f32(X), gu.dev_f32(w))
    torch.cuda.synchronize()
    rows = np.arange(M) if M <= 64 else np.array([0, 1, 2047, 4095])
    want = contract.router_logits(X[rows], w[None, :])[:, 0]
    assert gu.host(dot)[rows].view(np.uint32).tobytes() == want.view(np.uint32).tobytes()


# (M, H, E, k, dtype): every work split, f32 and bf16 inputs; rows up to 96 KB
# per block are staged in shared memory, the last two are too long for that
# and read the gate rows from device memory directly
FUSED = [(1, 2048, 256, 8, "f32"), (20, 264, 96, 5, "f32"), (100, 2048, 256, 8, "f32"), (1300, 2048, 256, 8, "f32"),
         (5, 2048, 512, 10, "bf16"), (700, 2048, 256, 8, "bf16"), (4096, 2048, 256, 8, "f32"),
         (70, 4096, 64, 4, "f32"), (203, 6000, 64, 4, "bf16"),
         # the persistent projection with the gate: ragged M, E and H, bf16
         (2500, 2056, 96, 5, "bf16"), (2432, 264, 128, 6, "f32")]


@pytest.mark.parametrize("M,H,E,k,dt", FUSED)
def test_router_gate_fused_is_the_two_calls(bi, M, H, E, k, dt):
    """bi_router_gate_topk gives the router outputs of bi_router_topk byte
    for byte, and a gate dot that is the contract's (and, for f32 inputs,
    bi_shared_gate's bytes, dot and sigmoid)."""
    import torch
    from oracle import contract
    X = synth.tokens(55, 0, M, M, H)
    W = synth.router_weights(55, M, E, H)
    w = synth.shared_gate_weights(55, M, H)
    if dt == "bf16":
        X, W, w = synth.to_bf16_bits(X), synth.to_bf16_bits(W), synth.to_bf16_bits(w)
        x, Wd, wd = gu.dev_bf16(X), gu.dev_bf16(W), gu.dev_bf16(w)
    else:
        x, Wd, wd = gu.dev_f32(X), gu.dev_f32(W), gu.dev_f32(w)
    fused = bi.router_gate_topk(x, Wd, wd, k)
    plain = bi.router_topk(x, Wd, k)
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    for f in ("logits", "ids", "weights", "margin", "margin_ulps"):
        assert fused[f].cpu().numpy().tobytes() == plain[f].cpu().numpy().tobytes(), f
    rows = np.arange(M) if M <= 1300 else np.array(sorted({r for r in (0, 5, 63, 64, M // 2, 3647, 3648, M - 65,
                                                                       M - 64, M - 1) if r < M}))
    want = contract.router_logits(X[rows], w[None, :])[:, 0]
    assert gu.host(fused["gate_dot"])[rows].view(np.uint32).tobytes() == want.view(np.uint32).tobytes()
    if dt == "f32":
        d, sg = bi.shared_gate(x, wd)
        torch.cuda.synchronize()
        assert gu.host(fused["gate_dot"]).tobytes() == gu.host(d).tobytes()
        assert gu.host(fused["gate_sigmoid"]).tobytes() == gu.host(sg).tobytes()
