"""The persistent router projection (large batches: at least one 64 x 64 x
8-partition item per SM): every CTA takes the same number of slab steps, so
an item may be cut between two CTAs, the second continuing the first's FMA
chains from the accumulators it handed over.

The bits must not depend on where the cuts fall: every logit equals the CPU
restatement of the reduction contract (oracle/contract.c) at shapes whose
cuts land inside items, with ragged M, E and H (a last slab with one 8-wide
block), for f32 and bf16 inputs and logits.  The hand-off flags carry a
per-call epoch, so a workspace full of arbitrary bytes, one left by another
plan, repeated calls and CUDA-graph replays must all give the same bytes.

Source pages: "batch changed the model's mind" ("The fix: m-invariant
twins"); "The Illusion of Determinism ..." ("The engineering cost of
determinism")."""
import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _dev(a):
    return gu.dev_f32(a) if a.dtype == np.float32 else gu.dev_bf16(a)


def _call(bi, x, w, M, H, E, k, in_bf16, logit_bf16, ws, stream=None):
    import torch
    lg = torch.empty((M, E), dtype=torch.bfloat16 if logit_bf16 else torch.float32, device="cuda")
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((M, k), dtype=torch.float32, device="cuda")
    mg = torch.empty(M, dtype=torch.float32, device="cuda")
    mu = torch.empty(M, dtype=torch.int32, device="cuda")
    bi.bi_router_topk(x, w, bi.BI_BF16 if in_bf16 else bi.BI_F32, bi.BI_BF16 if logit_bf16 else bi.BI_F32,
                      M, H, E, k, lg, ids, wt, mg, mu, workspace=ws, stream=stream)
    return {"logits": lg, "ids": ids, "weights": wt, "margin": mg, "margin_ulps": mu}


def _bytes(out):
    return {f: t.cpu().numpy().tobytes() for f, t in out.items()}


def _is_persistent(bi, M, E):
    m, c, n = bi.router_plan(M, E)
    return m < 0 and (c, n) == (2, 2)


def _require_persistent(bi, M, E):
    """On a 152-SM GB300 these shapes must take the persistent kernel (its
    block must fit an SM); elsewhere the SM count may put them on another
    plan."""
    import torch
    if _is_persistent(bi, M, E):
        return
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        pytest.fail(f"M={M} E={E}: plan {bi.router_plan(M, E)}, not the persistent kernel")
    pytest.skip("this GPU's SM count puts the shape on another plan")


# (M, H, E, k, inputs): cuts inside items (item counts not a multiple of the
# SM count), ragged M (not a multiple of 64), ragged E (96: one full and one
# half expert tile), ragged H (2056: a 17th slab with a single 8-wide block;
# 136: a second slab where only the first half's partition 0 has data)
CASES = [(1217, 2048, 256, 8, "f32"), (2500, 2056, 96, 5, "f32"), (3000, 136, 1024, 32, "f32"),
         (1999, 2048, 256, 8, "bf16"), (2432, 264, 128, 6, "bf16")]


@pytest.mark.parametrize("M,H,E,k,dt", CASES)
def test_persistent_logits_are_the_contract(bi, orc, M, H, E, k, dt):
    import torch
    from oracle import contract
    _require_persistent(bi, M, E)
    X = synth.tokens(71, 0, M, M, H)
    W = synth.router_weights(71, M, E, H)
    if dt == "bf16":
        X, W = synth.to_bf16_bits(X), synth.to_bf16_bits(W)
    want = contract.router_logits(X, W)
    x, w = _dev(X), _dev(W)
    ws = bi.router_workspace(M, E)
    got = _call(bi, x, w, M, H, E, k, dt == "bf16", False, ws)
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    g = gu.host(got["logits"])
    assert g.view(np.uint32).tobytes() == want.view(np.uint32).tobytes(), \
        f"{np.sum(g.view(np.uint32) != want.view(np.uint32))} logits differ"
    sel = orc.selection_from_logits(g, k)
    assert np.array_equal(gu.host(got["ids"]), sel["ids"])
    # bf16 logits: the same f32 values rounded to nearest even once
    got_b = _call(bi, x, w, M, H, E, k, dt == "bf16", True, ws)
    torch.cuda.synchronize()
    assert np.array_equal(gu.host_bf16_bits(got_b["logits"]), orc.round_bf16(want.astype(np.float64)))


def test_persistent_workspace_contents_do_not_matter(bi):
    """A fresh workspace of 0xFF bytes, one of random bytes, one that another
    plan (two-block tiles, M = 1000) has just filled with group sums, and the
    same workspace over five back-to-back calls: identical bytes each time."""
    import torch
    M, H, E, k = 4096, 2048, 256, 8
    _require_persistent(bi, M, E)
    X = synth.tokens(72, 0, 0, M, H)
    W = synth.router_weights(72, 0, E, H)
    x, w = gu.dev_f32(X), gu.dev_f32(W)
    n = bi.router_workspace_bytes(M, E)
    ref = _bytes(_call(bi, x, w, M, H, E, k, False, False, bi.router_workspace(M, E)))
    torch.cuda.synchronize()
    ff = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
    assert _bytes(_call(bi, x, w, M, H, E, k, False, False, ff)) == ref
    g = torch.Generator(device="cuda").manual_seed(5)
    rnd = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
    assert _bytes(_call(bi, x, w, M, H, E, k, False, False, rnd)) == ref
    # another plan's group sums over the epoch and flag words
    _call(bi, x[:1000], w, 1000, H, E, k, False, False, rnd)
    assert _bytes(_call(bi, x, w, M, H, E, k, False, False, rnd)) == ref
    outs = [_call(bi, x, w, M, H, E, k, False, False, rnd) for _ in range(5)]
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    for o in outs:
        assert _bytes(o) == ref


def test_persistent_graph_replays(bi):
    """The call captured once in a CUDA graph and replayed on new inputs
    copied into the same buffers: each replay equals the direct call on
    those inputs (the epoch advances inside the graph, once per replay)."""
    import torch
    M, H, E, k = 2048, 2048, 256, 8
    _require_persistent(bi, M, E)
    w = gu.dev_f32(synth.router_weights(73, 0, E, H))
    xs = [gu.dev_f32(synth.tokens(73, r, 0, M, H)) for r in range(3)]
    ws = bi.router_workspace(M, E)
    refs = []
    for x in xs:
        refs.append(_bytes(_call(bi, x, w, M, H, E, k, False, False, bi.router_workspace(M, E))))
    torch.cuda.synchronize()
    xin = torch.empty_like(xs[0])
    xin.copy_(xs[0])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _call(bi, xin, w, M, H, E, k, False, False, ws, stream=s)    # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        out = _call(bi, xin, w, M, H, E, k, False, False, ws, stream=s)
    for r in (1, 2, 0, 1):
        xin.copy_(xs[r])
        graph.replay()
        torch.cuda.synchronize()
        assert _bytes(out) == refs[r], r
    assert bi.bi_get_last_device_error() == 0
