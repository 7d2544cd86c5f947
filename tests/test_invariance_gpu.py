"""The pages' central claim, checked GPU against GPU: a request's logits,
expert ids, weights, margins and route hash are byte-identical solo versus
inside any batch, for every total token count M swept ("batch changed the
model's mind", sections "m-scan: the staircase", "16% of routing decisions"
and "The fix: m-invariant twins"; "The Illusion of Determinism in
Disaggregated Inference", section "The engineering cost of determinism":
cache miss at M = N versus cache hit at M = N mod block_size).

Every sweep counts its own comparisons and asserts the derivable total, so
a sweep that silently compared nothing cannot pass."""
import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

FIELDS = ("logits", "ids", "weights", "margin", "margin_ulps")


def route(bi, x, w, k, logit_dtype="f32"):
    return bi.router_topk(x, w, k, logit_dtype)


def rows_bytes(out, a, b):
    return {f: out[f][a:b].contiguous().cpu().numpy().tobytes() for f in FIELDS}


def test_tiny_mscan(bi):
    """H=256, E=64, top-4: the fixed 19-token request solo, then with
    co-arrivals bringing M to 20..96, placed first, in the middle and last."""
    import torch
    W, req, pool = synth.tiny_mscan(0)
    w = gu.dev_f32(W)
    solo = rows_bytes(route(bi, gu.dev_f32(req), w, 4), 0, 19)
    n = 0
    for M in range(20, 97):
        co = pool[:M - 19]
        for pos in ("first", "middle", "last"):
            off = {"first": 0, "middle": len(co) // 2, "last": len(co)}[pos]
            X = np.concatenate([co[:off], req, co[off:]])
            out = route(bi, gu.dev_f32(X), w, 4)
            torch.cuda.synchronize()
            assert rows_bytes(out, off, off + 19) == solo, f"M={M} {pos}"
            n += 1
    assert n == 77 * 3


M_SWEEP = [1, 2, 4, 8, 16, 19, 32] + list(range(35, 65)) + [65, 75, 96, 128, 256, 512, 1024, 2048, 4096]
# batches of at least a tile per SM (two-block tiles), with the request last
TAIL_SWEEP = [1235, 1300, 1400, 2500, 3000, 4096]


def test_router256_m_sweep(bi):
    """H=2048, E=256, top-8 plus the shared gate: the 19-token request is
    byte-identical solo and inside batches of every M in the sweep (M < 19
    compares a prefix of it).  The library spreads partitions over 16, 8, 4,
    2 or 1 thread blocks depending on M; the bytes must not change."""
    import torch
    H, E, k = 2048, 256, 8
    W = gu.dev_f32(synth.router_weights(30, 0, E, H))
    wsg = gu.dev_f32(synth.shared_gate_weights(30, 0, H))
    req = synth.tokens(30, 0, 0, 19, H)
    pool = synth.tokens(30, 0, 1, 4096, H)
    solo_x = gu.dev_f32(req)
    solo = rows_bytes(route(bi, solo_x, W, k), 0, 19)
    sd, ss = bi.shared_gate(solo_x, wsg)
    solo_gate = (sd.cpu().numpy().tobytes(), ss.cpu().numpy().tobytes())
    n = 0
    for M in M_SWEEP:
        if M <= 19:
            X = req[:M]
            off, cnt = 0, M
        else:
            off = (M - 19) // 2
            X = np.concatenate([pool[:off], req, pool[off:M - 19]])
            cnt = 19
        x = gu.dev_f32(X)
        out = route(bi, x, W, k)
        d, s = bi.shared_gate(x, wsg)
        torch.cuda.synchronize()
        got = rows_bytes(out, off, off + cnt)
        for f in FIELDS:
            width = len(solo[f]) // 19
            assert got[f] == solo[f][:width * cnt], f"{f} differs at M={M}"
        assert d[off:off + cnt].cpu().numpy().tobytes() == solo_gate[0][:4 * cnt], f"gate dot M={M}"
        assert s[off:off + cnt].cpu().numpy().tobytes() == solo_gate[1][:4 * cnt], f"gate sigmoid M={M}"
        n += 1
    for M in TAIL_SWEEP:
        off = M - 19                      # the request is the batch's last rows
        X = np.concatenate([pool[:off], req])
        out = route(bi, gu.dev_f32(X), W, k)
        torch.cuda.synchronize()
        got = rows_bytes(out, off, M)
        for f in FIELDS:
            assert got[f] == solo[f], f"{f} differs at M={M} (last rows)"
        n += 1
    assert n == len(M_SWEEP) + len(TAIL_SWEEP) == 52


def test_router_bf16_m_sweep(bi):
    """The bf16-logit router with bf16 inputs (H=2048, E=512, top-10, the
    tie-heavy workload's shape) and the fused shared gate: the 19-token
    request is byte-identical solo and inside batches of every M in the
    sweep, in logits, ids, weights, margins, gate dot and sigmoid."""
    import torch
    H, E, k = 2048, 512, 10
    W = gu.dev_bf16(synth.to_bf16_bits(synth.router_weights(32, 0, E, H)))
    wsg = gu.dev_bf16(synth.to_bf16_bits(synth.shared_gate_weights(32, 0, H)))
    req = synth.to_bf16_bits(synth.tokens(32, 0, 0, 19, H))
    pool = synth.to_bf16_bits(synth.tokens(32, 0, 1, 4096, H))
    keys = FIELDS + ("gate_dot", "gate_sigmoid")

    def call(X):
        o = bi.router_gate_topk(gu.dev_bf16(X), W, wsg, k, "bf16")
        torch.cuda.synchronize()
        return o

    def bytes_of(o, a, b):
        return {f: (o[f][a:b].contiguous().view(torch.int16) if o[f].dtype == torch.bfloat16
                    else o[f][a:b].contiguous()).cpu().numpy().tobytes() for f in keys}

    solo = bytes_of(call(req), 0, 19)
    n = 0
    for M in M_SWEEP + TAIL_SWEEP:
        if M <= 19:
            X, off, cnt = req[:M], 0, M
        else:
            off = (M - 19) // 2 if M in M_SWEEP else M - 19
            X = np.concatenate([pool[:off], req, pool[off:M - 19]])
            cnt = 19
        got = bytes_of(call(X), off, off + cnt)
        for f in keys:
            width = len(solo[f]) // 19
            assert got[f] == solo[f][:width * cnt], f"{f} differs at M={M}"
        n += 1
    assert n == len(M_SWEEP) + len(TAIL_SWEEP) == 52


def test_route_trace_760_decisions(bi):
    """The 19-token request through 40 layers (each with its own gate
    weights and hidden states), solo versus at total M = 75: all 760
    (layer, token) decisions classified as identical / same set in another
    order / different set.  The pages found 422 / 217 / 121; an
    M-invariant router must give 760 / 0 / 0."""
    import torch
    H, E, k = 2048, 256, 8
    same = order_only = different = 0
    for layer in range(40):
        W = gu.dev_f32(synth.router_weights(31, layer, E, H))
        req = synth.tokens(31, layer, 0, 19, H)
        co = synth.tokens(31, layer, 1, 75 - 19, H)
        a = route(bi, gu.dev_f32(req), W, k)["ids"].cpu().numpy()
        X = np.concatenate([co[:20], req, co[20:]])
        b = route(bi, gu.dev_f32(X), W, k)["ids"].cpu().numpy()[20:39]
        torch.cuda.synchronize()
        for t in range(19):
            if np.array_equal(a[t], b[t]):
                same += 1
            elif set(a[t]) == set(b[t]):
                order_only += 1
            else:
                different += 1
    assert same + order_only + different == 760
    assert (same, order_only, different) == (760, 0, 0)


def test_mixed_prefill_prefix_split(bi):
    """16 requests with lengths U[5, 300]; each layer runs the router
    (E=256, top-8), the shared gate and a 2048x2048 bf16 projection.  Every
    request is run batched (all 16 together), solo, as a cache miss (M = N)
    and as a suffix-only cache hit (M = N mod 16, the last full block when
    that is 0).  Per-request route hashes chained over the layers must be
    equal across all runs, and the suffix rows must be byte-identical, at
    all forty layers of the workload."""
    import torch
    H, E, k, L, blk = 2048, 256, 8, 40, 16
    lens = synth.request_lengths(0)
    assert len(lens) == 16 and lens.min() >= 5 and lens.max() <= 300
    offs = np.concatenate([[0], np.cumsum(lens)]).tolist()
    Mtot = offs[-1]
    Ws = [gu.dev_f32(synth.router_weights(40, l, E, H)) for l in range(L)]
    wsg = [gu.dev_f32(synth.shared_gate_weights(40, l, H)) for l in range(L)]
    Bs = [gu.dev_bf16(synth.gemm_b(40, H, H, layer=l)) for l in range(L)]
    # every layer's rows live on the device; a run gathers its rows there
    Xd = [gu.dev_f32(np.concatenate([synth.tokens(40, l, r, int(lens[r]), H) for r in range(16)]))
          for l in range(L)]
    Ad = [gu.dev_bf16(synth.gemm_a(41, Mtot, H, layer=l)) for l in range(L)]

    def run(rows_by_req):
        """rows_by_req: list of (request, row_begin, row_end) packed into one
        batch; returns per-request chained hashes and per-layer outputs."""
        idx = np.concatenate([np.arange(offs[r] + a, offs[r] + b) for r, a, b in rows_by_req])
        idx_d = torch.from_numpy(idx).cuda()
        sub = [0]
        for _, a, b in rows_by_req:
            sub.append(sub[-1] + (b - a))
        h = None
        outs = []
        for l in range(L):
            x = Xd[l].index_select(0, idx_d).contiguous()
            o = route(bi, x, Ws[l], k)
            d, s = bi.shared_gate(x, wsg[l])
            c = bi.gemm_bf16(Ad[l].index_select(0, idx_d).contiguous(), Bs[l])
            h = bi.route_hash(o["ids"], sub, basis=h)
            outs.append((o, d, c, sub))
        torch.cuda.synchronize()
        return h.cpu().numpy().view(np.uint64).copy(), outs

    batched_h, batched = run([(r, 0, int(lens[r])) for r in range(16)])
    cached, _ = bi.prefix_split([int(v) for v in lens], blk)     # the library's cache-hit rule
    compared = 0
    for r in range(16):
        n = int(lens[r])
        solo_h, solo = run([(r, 0, n)])
        assert solo_h[0] == batched_h[r], f"request {r}: hash differs solo vs batched"
        hit = n - cached[r]                         # suffix rows on a cache hit
        assert hit == (n % blk or blk)
        hit_h, hit_o = run([(r, n - hit, n)])
        hb = None
        for l in range(L):                         # the same suffix rows hashed from the batch
            a0 = batched[l][3][r] + n - hit
            hb = bi.route_hash(batched[l][0]["ids"], [a0, a0 + hit], basis=hb)
        torch.cuda.synchronize()
        assert hb.cpu().numpy().view(np.uint64)[0] == hit_h[0], f"request {r}: suffix hash differs"
        for l in range(L):
            bo, bd, bc, bsub = batched[l]
            ho, hd, hc, _ = hit_o[l]
            a0 = bsub[r] + n - hit
            for f in FIELDS:
                assert bo[f][a0:a0 + hit].cpu().numpy().tobytes() == ho[f].cpu().numpy().tobytes()
            assert bd[a0:a0 + hit].cpu().numpy().tobytes() == hd.cpu().numpy().tobytes()
            assert gu.host_bf16_bits(bc[a0:a0 + hit]).tobytes() == gu.host_bf16_bits(hc).tobytes()
            compared += 1
    assert compared == 16 * L
