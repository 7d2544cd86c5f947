"""Pins for the CPU oracle: checks against what the pages and mathematics fix,
never against the oracle itself.

Each function raises AssertionError on a mismatch.  They take the oracle
module as an argument so the mutation tests can run the very same checks
against deliberately broken builds of oracle.c and show that each planted
mistake turns at least one pin red (the method of the mutation proofs in
"diag(MODEL-MM-QWEN4-EXP): the MoE expert selections DIFFER ...", section
"Gates, read literally").
"""
from __future__ import annotations

import itertools
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ helpers
def all_finite_bf16():
    """Every finite bf16 bit pattern and its exact value (via binary32)."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        vals = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    keep = np.isfinite(vals)
    return bits[keep].astype(np.uint16), vals[keep]


def brute_topk(row, k):
    """Enumerate every k-subset; keep the one whose members all rank above
    every non-member under (value descending, index ascending, NaN highest).
    Exactly one subset qualifies; return it in rank order."""
    E = len(row)

    def key(e):
        v = row[e]
        return (0 if np.isnan(v) else 1, 0.0 if np.isnan(v) else -v, e)

    winners = []
    for S in itertools.combinations(range(E), k):
        Sset = set(S)
        if all(key(s) < key(r) for s in S for r in range(E) if r not in Sset):
            winners.append(S)
    assert len(winners) == 1, winners
    return sorted(winners[0], key=key)


def f32_to_bf16_trunc(x):
    """bf16 patterns of float32 values whose low 16 bits are zero."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0)
    return (u >> 16).astype(np.uint16)


# ------------------------------------------------------------------ formats
def pin_bf16_rounding(orc, rng=None):
    """bf16 RNE against brute force over the table of every finite bf16."""
    rng = rng or np.random.default_rng(1234)
    bits, vals = all_finite_bf16()
    # identity on representable values (and -0 stays -0)
    got = orc.round_bf16(vals)
    assert np.array_equal(got, bits), "rounding a bf16 value must return it unchanged"
    # random doubles over a wide range: nearest by search in the sorted table
    order = np.argsort(vals, kind="stable")
    sv, sb = vals[order], bits[order]
    x = np.concatenate([
        rng.standard_normal(4000) * np.exp2(rng.integers(-20, 20, 4000)),
        rng.uniform(-1e-38, 1e-38, 500),
    ])
    got = orc.round_bf16(x)
    for xi, gi in zip(x, got):
        j = np.searchsorted(sv, xi)
        cands = []
        for jj in (j - 1, j):
            if 0 <= jj < len(sv):
                cands.append((abs(sv[jj] - xi), int(sb[jj] & 1), int(sb[jj]), sv[jj]))
        best = min(c[0] for c in cands)
        ties = [c for c in cands if c[0] == best]
        if len(ties) > 1 and ties[0][3] != ties[1][3]:
            want = [c for c in ties if c[1] == 0][0][3]   # even significand
        else:
            want = ties[0][3]
        gv = np.array([gi], dtype=np.uint16).astype(np.uint32) << 16
        gval = float(gv.view(np.float32)[0])
        assert gval == want, (xi, gval, want)
    # exact midpoints between neighbours go to the even pattern
    pos = vals > 0
    pv, pb = vals[pos], bits[pos]
    o = np.argsort(pv)
    pv, pb = pv[o], pb[o]
    idx = rng.integers(0, len(pv) - 2, 2000)
    mids = (pv[idx] + pv[idx + 1]) / 2.0     # exact in double
    got = orc.round_bf16(mids)
    want = np.where((pb[idx] & 1) == 0, pb[idx], pb[idx + 1])
    assert np.array_equal(got, want), "ties must go to the even significand"
    # overflow: the largest finite bf16 plus half a spacing rounds to inf
    mx = float(pv[-1])
    spacing = mx - float(pv[-2])
    assert orc.round_bf16([mx + spacing / 2])[0] == 0x7F80
    assert orc.round_bf16([mx + spacing / 4])[0] == pb[-1]


def pin_f32_rounding(orc, rng=None):
    rng = rng or np.random.default_rng(99)
    x = rng.standard_normal(3000) * np.exp2(rng.integers(-30, 30, 3000))
    got = orc.round_f32(x).astype(np.float64)
    for xi, gi in zip(x, got):
        lo = np.nextafter(np.float32(gi), np.float32(-np.inf)).astype(np.float64)
        hi = np.nextafter(np.float32(gi), np.float32(np.inf)).astype(np.float64)
        assert abs(gi - xi) <= abs(lo - xi) and abs(gi - xi) <= abs(hi - xi), (xi, gi)


def pin_ulp_order(orc):
    """Sign-magnitude order, closed forms and brute-force monotonicity."""
    o = orc.ord_bf16
    assert o([0x0001])[0] - o([0x8001])[0] == 2
    assert o([0x3F80])[0] - o([0xBF80])[0] == 2 * 0x3F80
    assert o([0x0000])[0] == o([0x8000])[0] == 0
    bits, vals = all_finite_bf16()
    ords = orc.ord_bf16(bits)
    order = np.argsort(vals, kind="stable")
    sv, so = vals[order], ords[order]
    d = np.diff(so)
    dv = np.diff(sv)
    assert np.all(d[dv > 0] == 1), "adjacent bf16 values must be exactly 1 apart"
    assert np.all(d[dv == 0] == 0), "only +0/-0 share a value, and they share the ord"
    f = np.array([1.0, -1.0, 1e-40, -1e-40, 0.0, 3.4e38, -3.4e38], dtype=np.float32)
    for v in f:
        up = np.nextafter(v, np.float32(np.inf))
        a = orc.ord_f32(np.array([v], np.float32).view(np.uint32))[0]
        b = orc.ord_f32(np.array([up], np.float32).view(np.uint32))[0]
        assert b - a == 1, (v, a, b)
    assert orc.ord_f32(np.array([0x00000001], np.uint32))[0] - \
        orc.ord_f32(np.array([0x80000001], np.uint32))[0] == 2


# ------------------------------------------------------------------ router
def pin_router_integer_grid(orc, rng=None):
    """Inputs on an integer grid times 2^-4: every product and partial sum
    is exact, so the oracle must equal exact integer arithmetic."""
    rng = rng or np.random.default_rng(7)
    M, H, E = 5, 96, 11
    xi = rng.integers(-7, 8, (M, H))
    wi = rng.integers(-7, 8, (E, H))
    X = (xi * 2.0 ** -4).astype(np.float32)
    W = (wi * 2.0 ** -4).astype(np.float32)
    exact = (xi.astype(np.int64) @ wi.T.astype(np.int64)).astype(np.float64) * 2.0 ** -8
    assert np.array_equal(orc.router_logits(X, W), exact)
    # the same through bf16 inputs (integers <= 7 are exact in bf16)
    assert np.array_equal(orc.router_logits(f32_to_bf16_trunc(X), f32_to_bf16_trunc(W)), exact)


def pin_router_onehot(orc, rng=None):
    """A one-hot gate row picks one input column exactly."""
    rng = rng or np.random.default_rng(8)
    M, H, E = 4, 64, 9
    X = rng.standard_normal((M, H)).astype(np.float32)
    cols = rng.integers(0, H, E)
    W = np.zeros((E, H), np.float32)
    W[np.arange(E), cols] = 1.0
    assert np.array_equal(orc.router_logits(X, W), X[:, cols].astype(np.float64))


def pin_router_vs_matmul(orc, rng=None):
    """General inputs: within a few double roundings of a library matmul."""
    rng = rng or np.random.default_rng(9)
    M, H, E = 6, 256, 20
    X = rng.standard_normal((M, H)).astype(np.float32)
    W = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    ref = X.astype(np.float64) @ W.T.astype(np.float64)
    scale = np.abs(X.astype(np.float64)) @ np.abs(W.T.astype(np.float64))
    got = orc.router_logits(X, W)
    assert np.all(np.abs(got - ref) <= 1e-13 * scale)
    assert np.allclose(orc.router_absdot(X, W), scale, rtol=1e-13, atol=0)


def pin_shared_gate(orc, rng=None):
    from scipy.special import expit
    rng = rng or np.random.default_rng(10)
    M, H = 7, 128
    X = rng.standard_normal((M, H)).astype(np.float32)
    w = (rng.standard_normal(H) * 0.05).astype(np.float32)
    dot, sig = orc.shared_gate(X, w)
    ref = X.astype(np.float64) @ w.astype(np.float64)
    scale = np.abs(X.astype(np.float64)) @ np.abs(w.astype(np.float64))
    assert np.all(np.abs(dot - ref) <= 1e-13 * scale)
    assert np.allclose(sig, expit(dot), rtol=1e-15, atol=1e-16)
    d0, s0 = orc.shared_gate(np.zeros((1, H), np.float32), w)
    assert d0[0] == 0.0 and s0[0] == 0.5
    dn, sn = orc.shared_gate(-X, w)
    assert np.array_equal(dn, -dot)
    assert np.allclose(sn, 1.0 - sig, rtol=0, atol=1e-15)


def pin_shared_gate_onehot(orc, rng=None):
    """A one-hot w_sg picks one input column exactly: dot(X, e_j) = X[:, j],
    for every column j including the first and the last (a dropped term or a
    gate row indexed by token instead of by h gives another value)."""
    rng = rng or np.random.default_rng(21)
    M, H = 5, 48
    X = rng.standard_normal((M, H)).astype(np.float32)
    for j in (0, 1, H // 2, H - 1):
        w = np.zeros(H, np.float32)
        w[j] = 1.0
        dot, _ = orc.shared_gate(X, w)
        assert np.array_equal(dot, X[:, j].astype(np.float64)), j
    # a scaled one-hot: a power of two scales exactly
    w = np.zeros(H, np.float32)
    w[H - 1] = -0.25
    dot, _ = orc.shared_gate(X, w)
    assert np.array_equal(dot, -0.25 * X[:, H - 1].astype(np.float64))


def pin_shared_gate_integer_grid(orc, rng=None):
    """Inputs on an integer grid times 2^-4: every product and partial sum
    is exact in double, so the dot must equal integer arithmetic exactly,
    and the sigmoid at an exact dot of 0 is exactly 1/2."""
    rng = rng or np.random.default_rng(22)
    M, H = 6, 200
    xi = rng.integers(-7, 8, (M, H))
    wi = rng.integers(-7, 8, H)
    wi[-1] = 5                                   # the last term is never zero
    xi[:, -1] = np.arange(1, M + 1)
    X = (xi * 2.0 ** -4).astype(np.float32)
    w = (wi * 2.0 ** -4).astype(np.float32)
    dot, sig = orc.shared_gate(X, w)
    exact = (xi.astype(np.int64) @ wi.astype(np.int64)).astype(np.float64) * 2.0 ** -8
    assert np.array_equal(dot, exact)
    # rows built to cancel: dot exactly 0, sigmoid exactly 1/2
    Xc = np.zeros((2, H), np.float32)
    Xc[0, 0], Xc[0, 1] = 1.0, 1.0
    wc = np.zeros(H, np.float32)
    wc[0], wc[1] = 0.5, -0.5
    Xc[1, H - 2], Xc[1, H - 1] = 3.0, 3.0
    wc[H - 2], wc[H - 1] = 2.0, -2.0
    d, s = orc.shared_gate(Xc, wc)
    assert np.array_equal(d, [0.0, 0.0]) and np.array_equal(s, [0.5, 0.5])
    # sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4 (closed forms), the dot
    # being exactly representable: X = [ln3 as f32], w = [1]
    l3 = np.float32(np.log(3.0))
    d, s = orc.shared_gate(np.array([[l3], [-l3]], np.float32), np.ones(1, np.float32))
    expect = 1.0 / (1.0 + np.array([1.0 / 3.0, 3.0]) * np.exp(np.log(3.0) - float(l3)) ** np.array([1, -1]))
    assert np.allclose(s, expect, rtol=4e-16, atol=0)
    assert abs(s[0] - 0.75) < 1e-7 and abs(s[1] - 0.25) < 1e-7


# ------------------------------------------------------------------ top-k
def pin_topk_bruteforce(orc, rng=None):
    rng = rng or np.random.default_rng(11)
    for trial in range(150):
        E = int(rng.integers(2, 11))
        k = int(rng.integers(1, E))
        row = rng.integers(-2, 3, E).astype(np.float64)   # heavy ties
        if trial % 5 == 0:
            row[rng.integers(0, E)] = np.nan
        if trial % 7 == 0:
            row[rng.integers(0, E)] = -0.0
        want = brute_topk(row, k)
        got = orc.topk(row[None, :], k)[0]
        assert list(got) == list(want), (row, k, got, want)


def pin_topk_special(orc):
    E, k = 64, 8
    eq = np.full((1, E), 0.25)
    assert list(orc.topk(eq, k)[0]) == list(range(k)), "all-equal: lowest indices"
    dec = -np.arange(E, dtype=np.float64)[None, :]
    assert list(orc.topk(dec, k)[0]) == list(range(k))
    inc = np.arange(E, dtype=np.float64)[None, :]
    assert list(orc.topk(inc, k)[0]) == list(range(E - 1, E - 1 - k, -1))
    # +0 and -0 are equal: the lower index wins either way
    z = np.full((1, 4), -1.0)
    z[0, 1], z[0, 3] = -0.0, 0.0
    assert list(orc.topk(z, 1)[0]) == [1]
    z[0, 1], z[0, 3] = 0.0, -0.0
    assert list(orc.topk(z, 1)[0]) == [1]


def pin_topk_permutation(orc, rng=None):
    """Permuting tokens permutes the result rows; relabelling experts maps
    the selected set (values distinct, so no tie-break is involved)."""
    rng = rng or np.random.default_rng(12)
    M, E, k = 9, 40, 6
    L = rng.standard_normal((M, E))
    ids = orc.topk(L, k)
    p = rng.permutation(M)
    assert np.array_equal(orc.topk(L[p], k), ids[p])
    q = rng.permutation(E)               # new expert j is old expert q[j]
    ids2 = orc.topk(L[:, q], k)
    assert np.array_equal(q[ids2], ids)


def pin_planted_ties(orc, rng=None):
    """Duplicated gate rows (j1 < j2) give identical logits; wherever the
    pair straddles the top-k boundary the lower index is the one selected."""
    rng = rng or np.random.default_rng(13)
    M, H, E, k = 64, 32, 24, 5
    X = rng.standard_normal((M, H)).astype(np.float32)
    W = rng.standard_normal((E, H)).astype(np.float32)
    j1, j2 = 3, 17
    W[j2] = W[j1]
    L = orc.router_logits(X, W)
    assert np.array_equal(L[:, j1], L[:, j2])
    ids = orc.topk(L, k)
    straddle = 0
    for m in range(M):
        s = set(ids[m])
        assert not (j2 in s and j1 not in s), "the higher index can never win a tie"
        if j1 in s and j2 not in s:
            straddle += int(L[m, j1] == np.min(L[m, list(s)]))
    typed = L.astype(np.float32)
    mg, ul, smin, rmax = orc.margin(typed, ids)
    zero = np.where(ul == 0)[0]
    assert straddle >= 1
    assert len(zero) == straddle
    for m in zero:
        assert {int(smin[m]), int(rmax[m])} == {j1, j2} and mg[m] == 0.0


# ------------------------------------------------------------------ softmax / margin
def pin_softmax(orc, rng=None):
    from scipy.special import expit
    rng = rng or np.random.default_rng(14)
    L = rng.standard_normal((10, 32)) * 3
    assert np.all(orc.softmax_selected(L, orc.topk(L, 1)) == 1.0)
    eq = np.full((3, 16), 1.5)
    for k in (2, 4, 5):
        w = orc.softmax_selected(eq, orc.topk(eq, k))
        assert np.allclose(w, 1.0 / k, rtol=1e-15)
    ids2 = orc.topk(L, 2)
    w = orc.softmax_selected(L, ids2)
    d = L[np.arange(10), ids2[:, 0]] - L[np.arange(10), ids2[:, 1]]
    assert np.allclose(w[:, 0], expit(d), rtol=1e-14)
    assert np.allclose(w[:, 1], expit(-d), rtol=1e-14)
    ids8 = orc.topk(L, 8)
    w8 = orc.softmax_selected(L, ids8)
    assert np.allclose(w8.sum(1), 1.0, rtol=1e-14)
    assert np.all(np.diff(w8, axis=1) <= 0), "weights follow rank order"
    assert np.allclose(orc.softmax_selected(L + 100.0, ids8), w8, rtol=1e-12)


def pin_margin(orc):
    # bf16: sel_min = 1.0 (0x3F80), rej_max = next below (0x3F7F): one ULP
    row = np.array([[0x3F80, 0x3F7F, 0x4000, 0x3F00]], dtype=np.uint16)
    mg, ul, smin, rmax = orc.margin(row, np.array([[2, 0]], dtype=np.int32))
    assert ul[0] == 1 and smin[0] == 0 and rmax[0] == 1
    assert mg[0] == 1.0 - 0.99609375
    # straddling zero: +min subnormal selected, -min subnormal rejected
    row = np.array([[0x0001, 0x8001, 0xBF80]], dtype=np.uint16)
    mg, ul, _, _ = orc.margin(row, np.array([[0]], np.int32))
    assert ul[0] == 2
    # +1 selected, -1 rejected: 2 * 0x3F80 ULPs apart
    row = np.array([[0xBF80, 0x3F80]], dtype=np.uint16)
    mg, ul, _, _ = orc.margin(row, np.array([[1]], np.int32))
    assert ul[0] == 2 * 0x3F80 and mg[0] == 2.0
    # f32 negative logits: -1.0 selected, nextbelow(-1.0) rejected -> 1 ULP
    a = np.float32(-1.0)
    b = np.nextafter(a, np.float32(-np.inf))
    row = np.array([[b, a, np.float32(-5.0)]], dtype=np.float32)
    mg, ul, _, _ = orc.margin(row, np.array([[1]], np.int32))
    assert ul[0] == 1 and mg[0] == float(a) - float(b)
    # exact tie: zero in both units
    row = np.array([[0.5, 0.5, 0.1]], dtype=np.float32)
    mg, ul, smin, rmax = orc.margin(row, orc.topk(row.astype(np.float64), 1))
    assert ul[0] == 0 and mg[0] == 0.0 and smin[0] == 0 and rmax[0] == 1


# ------------------------------------------------------------------ GEMM
def pin_gemm_identity(orc, rng=None):
    rng = rng or np.random.default_rng(15)
    M, K = 7, 64
    A = (rng.standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    B = np.zeros((K, K), np.uint16)
    B[np.arange(K), np.arange(K)] = 0x3F80          # bf16 1.0
    _, _, Cm = orc.gemm_bf16(A, B)
    assert np.array_equal(orc.bf16_to_double(Cm), orc.bf16_to_double(A))


def pin_gemm_integer_grid(orc, rng=None):
    """Integer inputs times 2^-3 with |C| < 2^8 units: exact in double and
    exactly representable in bf16, so C must equal integer arithmetic."""
    rng = rng or np.random.default_rng(16)
    M, N, K = 9, 24, 64
    ai = rng.integers(-2, 3, (M, K))
    bi = rng.integers(-1, 2, (N, K))
    A = f32_to_bf16_trunc((ai * 2.0 ** -3).astype(np.float32))
    B = f32_to_bf16_trunc((bi * 2.0 ** -3).astype(np.float32))
    exact = (ai @ bi.T).astype(np.float64) * 2.0 ** -6
    assert np.max(np.abs(ai @ bi.T)) < 256
    acc, absacc, Cm = orc.gemm_bf16(A, B)
    assert np.array_equal(acc, exact)
    assert np.array_equal(orc.bf16_to_double(Cm), exact)
    assert np.array_equal(absacc, (np.abs(ai) @ np.abs(bi).T) * 2.0 ** -6)


def pin_gemm_vs_matmul(orc, rng=None):
    rng = rng or np.random.default_rng(17)
    M, N, K = 5, 16, 128
    A = ((rng.standard_normal((M, K)) / 8).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    B = ((rng.standard_normal((N, K)) / 8).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    Ad = orc.bf16_to_double(A)
    Bd = orc.bf16_to_double(B)
    acc, absacc, Cm = orc.gemm_bf16(A, B)
    assert np.all(np.abs(acc - Ad @ Bd.T) <= 1e-13 * (np.abs(Ad) @ np.abs(Bd).T))
    acc2, _, C2 = orc.gemm_bf16(A, B, rows=[4, 1])
    assert np.array_equal(acc2, acc[[4, 1]]) and np.array_equal(C2, Cm[[4, 1]])


# ------------------------------------------------------------------ hash
def load_fnv_vectors():
    out = []
    with open(os.path.join(GOLDEN, "fnv1a64_vectors.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            hexbytes, want = line.split()
            data = bytes.fromhex(hexbytes) if hexbytes != "-" else b""
            out.append((data, int(want, 16)))
    return out


def pin_fnv(orc):
    vecs = load_fnv_vectors()
    assert len(vecs) >= 3
    for data, want in vecs:
        assert orc.fnv1a64(data) == want, (data, hex(orc.fnv1a64(data)), hex(want))
    a, b = b"batch", b"invariant"
    assert orc.fnv1a64(a + b) == orc.fnv1a64(b, orc.fnv1a64(a))


def pin_route_hash(orc, rng=None):
    rng = rng or np.random.default_rng(18)
    M, E, k = 12, 64, 8
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(M)]).astype(np.int32)
    h = orc.route_hash(ids)
    # the selected SET is hashed: any order of ids within a row, same hash
    shuffled = np.stack([rng.permutation(r) for r in ids]).astype(np.int32)
    assert orc.route_hash(shuffled) == h
    other = ids.copy()
    row = set(other[5])
    other[5, 0] = [e for e in range(E) if e not in row][0]
    assert orc.route_hash(other) != h
    for r in (0, 1, 7, M):
        assert orc.route_hash(ids, r, M, orc.route_hash(ids, 0, r)) == h
    assert orc.route_hash(ids, 3, 3) == orc.FNV64_BASIS
    # serialisation: one token {1, 3}, k=2, in either order, is the 8 bytes
    # 01 00 00 00 03 00 00 00 (ascending ids, little-endian int32)
    assert orc.route_hash(np.array([[3, 1]], np.int32)) == orc.fnv1a64(bytes([1, 0, 0, 0, 3, 0, 0, 0]))


ALL_PINS = [
    pin_bf16_rounding, pin_f32_rounding, pin_ulp_order,
    pin_router_integer_grid, pin_router_onehot, pin_router_vs_matmul, pin_shared_gate,
    pin_shared_gate_onehot, pin_shared_gate_integer_grid,
    pin_topk_bruteforce, pin_topk_special, pin_topk_permutation, pin_planted_ties,
    pin_softmax, pin_margin,
    pin_gemm_identity, pin_gemm_integer_grid, pin_gemm_vs_matmul,
    pin_fnv, pin_route_hash,
]
