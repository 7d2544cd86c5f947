"""bi_shared_gate and bi_route_trace_hash on the GPU against the oracle."""
import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,H", [(1, 2048), (3, 256), (17, 2048), (75, 136), (1000, 2048), (64, 8)])
def test_shared_gate_parity(bi, orc, M, H):
    import torch
    X = synth.tokens(20, 0, M, M, H)
    w = synth.shared_gate_weights(20, M, H)
    dot, sig = bi.shared_gate(gu.dev_f32(X), gu.dev_f32(w))
    torch.cuda.synchronize()
    rdot, rsig = orc.shared_gate(X, w)
    absdot = np.abs(X.astype(np.float64)) @ np.abs(w.astype(np.float64))
    assert np.all(np.abs(gu.host(dot) - rdot) <= gu.router_logit_tol(absdot))
    # sigmoid: the dot error times the slope, plus a few f32 roundings
    slope = rsig * (1 - rsig)
    assert np.all(np.abs(gu.host(sig) - rsig) <= slope * gu.router_logit_tol(absdot) + 8 * gu.U * rsig)


def test_shared_gate_matches_router_order(bi):
    """The gate dot and the router use one reduction contract: a gate
    vector used as a router row gives the same bits."""
    import torch
    M, H, E = 50, 2048, 32
    X = synth.tokens(21, 0, 0, M, H)
    W = synth.router_weights(21, 0, E, H)
    x = gu.dev_f32(X)
    out = bi.router_topk(x, gu.dev_f32(W), 2, "f32")
    dot, _ = bi.shared_gate(x, gu.dev_f32(W[5]))
    torch.cuda.synchronize()
    assert gu.host(out["logits"])[:, 5].tobytes() == gu.host(dot).tobytes()


def test_route_hash_parity(bi, orc):
    import torch
    g = np.random.default_rng(22)
    M, E, k = 777, 256, 8
    ids = np.stack([g.choice(E, k, replace=False) for _ in range(M)]).astype(np.int32)
    offs = [0, 5, 5, 300, 301, 777]
    h = bi.route_hash(torch.from_numpy(ids).cuda(), offs)
    torch.cuda.synchronize()
    got = h.cpu().numpy().view(np.uint64)
    for r in range(len(offs) - 1):
        assert int(got[r]) == orc.route_hash(ids, offs[r], offs[r + 1])
    # chaining through the device basis (in place, as layers chain)
    h2 = h.clone()
    bi.bi_route_trace_hash(torch.from_numpy(ids).cuda(), M, k, offs, h2, h2)
    torch.cuda.synchronize()
    got2 = h2.cpu().numpy().view(np.uint64)
    for r in range(len(offs) - 1):
        assert int(got2[r]) == orc.route_hash(ids, offs[r], offs[r + 1], basis=int(got[r]))
    # order of ids within a row does not matter (a set is hashed)
    perm = np.stack([g.permutation(r) for r in ids]).astype(np.int32)
    h3 = bi.route_hash(torch.from_numpy(perm).cuda(), offs)
    torch.cuda.synchronize()
    assert np.array_equal(h3.cpu().numpy(), h.cpu().numpy())


@pytest.mark.parametrize("k", [3, 8, 12, 32])
def test_route_hash_any_id_values(bi, orc, k):
    """Ids of every byte length (0, one byte, two, three, four, negative)
    and every sort width: the kernel folds the high zero bytes of an id into
    one step, so each length takes its own path; all must equal the oracle's
    byte-by-byte FNV-1a.  Ranges longer than 32 rows cross the warp's row
    batches."""
    import torch
    g = np.random.default_rng(23 + k)
    M = 170
    classes = [np.zeros(1, np.int64), np.arange(1, 256), np.arange(256, 65536, 97),
               np.arange(65536, 1 << 24, 40009), np.arange(1 << 24, (1 << 31) - 1, 9_000_011),
               -np.arange(1, 1 << 31, 7_000_003)]
    pool = np.concatenate(classes)
    ids = g.choice(pool, size=(M, k)).astype(np.int32)
    offs = [0, 1, 40, 100, 100, 170]
    h = bi.route_hash(torch.from_numpy(ids).cuda(), offs)
    torch.cuda.synchronize()
    got = h.cpu().numpy().view(np.uint64)
    for r in range(len(offs) - 1):
        assert int(got[r]) == orc.route_hash(ids, offs[r], offs[r + 1]), f"range {r}, k={k}"
