"""Router parity: bi_router_topk on the GPU against the CPU oracle.

The library splits each 32x64 tile's 16 partitions over 1, 2, 4, 8 or 16
thread blocks depending on M (from one tile per SM on, two blocks of 8; for
batches whose group sums would pass 64 MiB, whole tiles plus a split tail);
the cases below cover every split in every input/logit dtype, including E
that is not a multiple of the 64-expert tile.

Logits within the stated tolerance of the exact dot; ids bit-exact wherever
the oracle's margin exceeds twice that tolerance; the oracle's top-k applied
to the GPU's OWN logits bit-exact against the GPU ids for every token;
margins (value and ULPs) and weights against the oracle on the GPU's own
logits.  Shapes span several 32x32 tiles with ragged tails and every
partition split the library chooses (small M spreads partitions over more
thread blocks)."""
import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def run_router(bi, X, W, k, logit_dtype):
    import torch
    x = gu.dev_f32(X) if X.dtype == np.float32 else gu.dev_bf16(X)
    w = gu.dev_f32(W) if W.dtype == np.float32 else gu.dev_bf16(W)
    out = bi.router_topk(x, w, k, logit_dtype)
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    logits = gu.host(out["logits"]) if logit_dtype == "f32" else gu.host_bf16_bits(out["logits"])
    return {"logits": logits, "ids": gu.host(out["ids"]), "weights": gu.host(out["weights"]),
            "margin": gu.host(out["margin"]), "margin_ulps": gu.host(out["margin_ulps"])}


def check_selection_on_own_logits(orc, g, k):
    """Everything downstream of the logits, given the GPU's own logits."""
    sel = orc.selection_from_logits(g["logits"], k)
    assert np.array_equal(g["ids"], sel["ids"]), "top-k of the GPU logits must match the oracle exactly"
    ul = np.minimum(sel["margin_ulps"], np.iinfo(np.int32).max)
    assert np.array_equal(g["margin_ulps"].astype(np.int64), ul)
    mref = sel["margin"]
    assert np.all(np.abs(g["margin"] - mref) <= gu.U * np.abs(mref) + 1e-45)
    widened = orc.bf16_to_double(g["logits"]) if g["logits"].dtype == np.uint16 else g["logits"].astype(np.float64)
    rows = np.arange(len(widened))[:, None]
    gaps = widened[rows, sel["ids"]] - widened[rows, sel["ids"][:, :1]]
    tol = gu.softmax_tol(gaps, k) * sel["weights"]
    assert np.all(np.abs(g["weights"] - sel["weights"]) <= tol)
    return sel


CASES_F32 = [
    # (M, H, E, k)
    (1, 256, 64, 4), (19, 256, 64, 4), (37, 256, 64, 4), (96, 256, 64, 4),
    (1, 2048, 256, 8), (7, 2048, 256, 8), (75, 2048, 256, 8), (300, 2048, 256, 8),
    (1100, 2048, 256, 8), (520, 200, 128, 6), (3000, 136, 1024, 32),
    (33, 264, 96, 5), (5, 8, 32, 1), (70, 136, 1024, 32), (600, 264, 96, 5),
    # at least a tile per SM: every tile as two 8-partition blocks, two blocks
    # to an SM (the shallow ring)
    (1300, 2048, 256, 8), (4904, 128, 64, 4), (400, 136, 1024, 32),
]


@pytest.mark.parametrize("M,H,E,k", CASES_F32)
def test_router_f32_parity(bi, orc, M, H, E, k):
    X = synth.tokens(1, 0, M, M, H)
    W = synth.router_weights(1, M, E, H)
    g = run_router(bi, X, W, k, "f32")
    exact = orc.router_logits(X, W)
    absdot = orc.router_absdot(X, W)
    err = np.abs(g["logits"].astype(np.float64) - exact)
    assert np.all(err <= gu.router_logit_tol(absdot)), f"max err/absdot = {np.max(err / absdot)}"
    check_selection_on_own_logits(orc, g, k)
    ref = orc.router_full(X, W, k, "f32")
    safe = ref["margin"] > 2 * np.max(gu.router_logit_tol(absdot), axis=1)
    assert np.array_equal(g["ids"][safe], ref["ids"][safe])
    assert safe.mean() > 0.5


@pytest.mark.parametrize("M", [1, 5, 64, 200, 700])
def test_router_bf16_logits_tie_grid(bi, orc, M):
    """Tie-heavy grid inputs: f32 sums are exact in any order, so the bf16
    logits, ids, ties and margins must equal the oracle bit for bit."""
    X, W = synth.tie_heavy_call(0, 100 + M, n_tokens=M)
    k = synth.TIE512["k"]
    g = run_router(bi, X, W, k, "bf16")
    ref = orc.router_full(X, W, k, "bf16")
    assert np.array_equal(g["logits"], ref["logits"])
    assert np.array_equal(g["ids"], ref["ids"])
    assert np.array_equal(g["margin_ulps"].astype(np.int64), ref["margin_ulps"])
    assert np.array_equal(g["margin"].astype(np.float64), ref["margin"])
    check_selection_on_own_logits(orc, g, k)


def test_tie_heavy_workload_counts(bi, orc):
    """The 48-call x 5-token tie-heavy workload: the GPU's exact-tie count at
    the k-boundary equals the oracle's (78 of 240), every tie goes to the
    lower index, and each call's route hash matches the oracle's."""
    import torch
    slots = gpu_ties = orc_ties = 0
    for call in range(48):
        X, W = synth.tie_heavy_call(0, call)
        g = run_router(bi, X, W, 10, "bf16")
        ref = orc.router_full(X, W, 10, "bf16")
        assert np.array_equal(g["ids"], ref["ids"])
        slots += len(g["ids"])
        gpu_ties += int(np.sum(g["margin_ulps"] == 0))
        orc_ties += int(np.sum(ref["margin_ulps"] == 0))
        h = bi.route_hash(torch.from_numpy(g["ids"]).cuda(), [0, len(g["ids"])])
        torch.cuda.synchronize()
        assert int(h.cpu().numpy().view(np.uint64)[0]) == orc.route_hash(ref["ids"])
    assert slots == 240
    assert gpu_ties == orc_ties == 78


@pytest.mark.parametrize("M", [40, 900, 1400])
def test_router_bf16_in_f32_logits(bi, orc, M):
    X = synth.to_bf16_bits(synth.tokens(2, 0, 0, M, 512))
    W = synth.to_bf16_bits(synth.router_weights(2, 0, 128, 512))
    g = run_router(bi, X, W, 6, "f32")
    exact = orc.router_logits(X, W)
    absdot = np.abs(orc.bf16_to_double(X)) @ np.abs(orc.bf16_to_double(W)).T
    assert np.all(np.abs(g["logits"] - exact) <= gu.router_logit_tol(absdot))
    check_selection_on_own_logits(orc, g, 6)


@pytest.mark.parametrize("M", [50, 1000, 1300])
def test_router_f32_in_bf16_logits(bi, orc, M):
    """General f32 inputs, bf16 logits.  The GPU rounds its f32 sum (itself
    within the f32 tolerance of the exact dot) to bf16, so it lies within
    one bf16 ULP plus the f32 tolerance of the exact logit; one ULP alone
    cannot hold for logits near zero, where the f32 error exceeds a bf16
    ULP.  Away from zero the ordinal distance is at most one."""
    X = synth.tokens(3, 0, 0, M, 2048)
    W = synth.router_weights(3, 0, 512, 2048)
    g = run_router(bi, X, W, 10, "bf16")
    ref = orc.router_full(X, W, 10, "bf16")
    absdot = orc.router_absdot(X, W)
    got = orc.bf16_to_double(g["logits"])
    assert np.all(np.abs(got - ref["exact"]) <= gu.bf16_ulp(ref["exact"]) + gu.router_logit_tol(absdot))
    big = np.abs(ref["exact"]) >= 2.0 ** 8 * gu.router_logit_tol(absdot)
    d = np.abs(orc.ord_bf16(g["logits"]) - orc.ord_bf16(ref["logits"]))
    assert big.mean() > 0.9 and np.max(d[big]) <= 1
    check_selection_on_own_logits(orc, g, 10)


def test_router_full_size_sampled(bi, orc):
    """M = 4096 (the benchmark's launch configuration): sampled rows against
    the oracle, all rows' selection against the oracle on GPU logits."""
    M, H, E, k = 4096, 2048, 256, 8
    X = synth.tokens(4, 0, 0, M, H)
    W = synth.router_weights(4, 0, E, H)
    g = run_router(bi, X, W, k, "f32")
    rows = np.array([0, 1, 31, 32, 33, 1000, 2047, 2048, 3647, 3648, 3700, 4064, 4095])
    exact = orc.router_logits(X[rows], W)
    absdot = orc.router_absdot(X[rows], W)
    assert np.all(np.abs(g["logits"][rows] - exact) <= gu.router_logit_tol(absdot))
    check_selection_on_own_logits(orc, g, k)


def test_router_nan_and_zero_rules(bi, orc):
    """A NaN logit ranks first; -0 and +0 tie and go to the lower index
    (inputs built so that whole logit columns are NaN / signed zeros)."""
    M, H, E, k = 4, 128, 64, 3
    X = synth.tokens(5, 0, 0, M, H)
    W = synth.router_weights(5, 0, E, H)
    W[7, :] = 0.0          # +0 logits (f32 chain from +0 with zero products)
    W[3, :] = -0.0
    W[40, 0] = np.nan      # NaN logits
    g = run_router(bi, X, W, k, "f32")
    assert np.all(g["ids"][:, 0] == 40)
    sel = orc.selection_from_logits(g["logits"], k)
    assert np.array_equal(g["ids"], sel["ids"])


@pytest.mark.parametrize("E,M,H", [(64, 5000, 2048), (256, 1300, 2048), (1024, 400, 2048), (1024, 8300, 136)])
def test_router_splits_bit_identical(bi, E, M, H):
    """The same tokens under different work splits: the first and the last
    300 rows of an M-token batch, each also computed as a 300-token batch,
    give identical bytes in every output.  The M-token batches run as
    two-block tiles; at E = 1024, M = 8300 the group sums would pass 64 MiB,
    so rows 0..8191 run as whole tiles and the last rows as a split tail.
    As 300-token batches the rows are split differently again."""
    import torch
    k = 8
    X = synth.tokens(6, 0, 0, M, H)
    w = gu.dev_f32(synth.router_weights(6, 0, E, H))
    big = bi.router_topk(gu.dev_f32(X), w, k, "f32")
    for a in (0, M - 300):
        small = bi.router_topk(gu.dev_f32(X[a:a + 300]), w, k, "f32")
        torch.cuda.synchronize()
        for f in ("logits", "ids", "weights", "margin", "margin_ulps"):
            assert small[f].cpu().numpy().tobytes() == big[f][a:a + 300].cpu().numpy().tobytes(), (a, f)


def test_router_plan_reports_the_cut(bi):
    """bi_router_plan on a 152-SM GB300: one cluster launch up to 112 rows
    (E <= 512), partition-split tiles below a tile half per SM, two-block
    tiles once their blocks fill the SMs, the persistent projection from one
    64 x 64 x 8-partition item per SM, whole tiles plus a split tail where
    the group sums would pass 64 MiB."""
    import torch
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("plan thresholds are stated for 152 SMs")
    for M in (1, 64, 112):
        m, c, n = bi.router_plan(M, 256)
        assert m == M and c in (-16, -8) and n == 1, (M, m, c, n)
    assert bi.router_plan(128, 256) == (0, 8, 2)       # past the cluster router: 16 tiles, 8 blocks each
    assert bi.router_plan(129, 256) == (0, 4, 2)       # 20 tiles: 4 blocks each fill 80 SMs
    assert bi.router_plan(4096, 256) == (-152, 2, 2)     # the persistent projection: 512 items, 152 CTAs
    assert bi.router_plan(1217, 256) == (-152, 2, 2)     # 160 items
    assert bi.router_plan(1216, 256) == (-152, 2, 2)     # 152 items: one a CTA
    assert bi.router_plan(1152, 256) == (0, 2, 2)        # 144 items: fewer than the SMs, two-block tiles
    assert bi.router_plan(256, 256) == (0, 4, 2)
    assert bi.router_plan(640, 256) == (0, 2, 2)       # 80 tiles: 160 two-block halves
    assert bi.router_plan(1024, 256) == (0, 2, 2)
    assert bi.router_plan(8300, 1024) == (8192, 2, 3)
    assert bi.router_plan(64, 1024)[2] == 2            # E = 1024: always the tiled kernels


def test_router_two_streams_separate_workspaces(bi):
    """Two tiled calls (M > 128, so their group sums go through the caller's
    workspace) queued on two streams with no ordering between them, each with
    its own workspace: every output is byte-identical to the same call run
    alone.  The library keeps no buffer of its own that the two could share."""
    import torch
    M, H, E, k = 3000, 2048, 256, 8
    Xa = gu.dev_f32(synth.tokens(61, 0, 0, M, H))
    Xb = gu.dev_f32(synth.tokens(61, 1, 0, M, H))
    wa = gu.dev_f32(synth.router_weights(61, 0, E, H))
    wb = gu.dev_f32(synth.router_weights(61, 1, E, H))
    ref_a = bi.router_topk(Xa, wa, k)
    torch.cuda.synchronize()
    ref_b = bi.router_topk(Xb, wb, k)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    wsa, wsb = bi.router_workspace(M, E), bi.router_workspace(M, E)
    assert wsa is not None and wsa.numel() == bi.router_workspace_bytes(M, E)
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):
        with torch.cuda.stream(sa):
            oa = bi.router_topk(Xa, wa, k, workspace=wsa, stream=sa)
        with torch.cuda.stream(sb):
            ob = bi.router_topk(Xb, wb, k, workspace=wsb, stream=sb)
        outs.append((oa, ob))
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    for oa, ob in outs:
        for f in ("logits", "ids", "weights", "margin", "margin_ulps"):
            assert oa[f].cpu().numpy().tobytes() == ref_a[f].cpu().numpy().tobytes(), f
            assert ob[f].cpu().numpy().tobytes() == ref_b[f].cpu().numpy().tobytes(), f
