"""bi_attention_prefill against the attention oracle, and its invariance.

Parity: every output element within the bound derived in `_tol` of the
double-precision oracle (oracle/attention.py), at ragged shapes that span
several query tiles and key blocks with ragged tails, cached prefixes,
empty requests, and MHA, GQA and MQA head groupings; at the full prefill
workload on sampled rows the oracle computes one query at a time.

Invariance (bit-exact, the GPU against itself): a query row's bytes must not
depend on how many of its request's queries are in the call (suffix after a
cached prefix vs full prefill; a chunked prefill), on which query tile it
falls in, or on what other requests share the call.

Source page: "The Illusion of Determinism in Disaggregated Inference",
section "The physics of the cascade"."""
import numpy as np
import pytest

from serving_numerics_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

D = 128
SCALE = 1.0 / np.sqrt(128.0)


def _run(bi, Q, K, V, qo, ko, nh, nkv, scale=SCALE):
    import torch
    o, lse = bi.attention_prefill(gu.dev_bf16(Q), gu.dev_bf16(K), gu.dev_bf16(V), list(qo), list(ko), scale)
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    return gu.host_bf16_bits(o), gu.host(lse)


def _tol(ref_o, V, ko, nh, nkv, q_req):
    """|o - exact| <= 1.05 * 2^-8 * max|v| + 2^-8 * |exact|, per element.

    The weights p_j are rounded to bf16 (relative error <= 2^-9 each) before
    the product with V while the row sum l adds them unrounded, so the kernel
    computes sum_j w_j (1 + d_j) v_j with sum_j w_j = 1 and |d_j| <= 2^-9:
    at most 2^-9 * max|v| over the visible rows of V.  The output's rounding
    to bf16 adds 2^-9 |o|; ex2.approx (relative error about 2^-22), the f32
    scores and the f32 accumulations add terms of order 2^-20.  The bound
    allows twice the weight term (a margin for the reciprocal of l and the
    rescalings) and 2^-8 |o|."""
    Vd = gu_bf16_to_f64(V)
    g = nh // nkv
    tol = np.zeros(ref_o.shape)
    for r in range(len(ko) - 1):
        qs, qe = q_req[r], q_req[r + 1]
        if qe == qs:
            continue
        vmax = np.abs(Vd[ko[r]:ko[r + 1]]).max(axis=(0, 2))          # per kv head
        tol[qs:qe] = 1.05 * 2.0 ** -8 * np.repeat(vmax, g)[None, :, None]
    return tol + 2.0 ** -8 * np.abs(ref_o)


def gu_bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_parity(bi, q_lens, kv_lens, nh, nkv, seed, scale=SCALE):
    from oracle import attention as oatt
    qo, ko = synth.attention_offsets(q_lens, np.asarray(kv_lens) - np.asarray(q_lens))
    Q, K, V = synth.attention_inputs(seed, int(qo[-1]), int(ko[-1]), nh, nkv)
    o, lse = _run(bi, Q, K, V, qo, ko, nh, nkv, scale)
    # the oracle widens each query head's own key/value head
    g = nh // nkv
    ref_o, ref_lse = oatt.attention_prefill(Q, np.repeat(K, g, axis=1), np.repeat(V, g, axis=1), qo, ko, scale)
    got = gu_bf16_to_f64(o)
    tol = _tol(ref_o, V, ko, nh, nkv, qo)
    bad = np.abs(got - ref_o) > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} outputs outside the bound; worst excess " \
                          f"{np.max(np.abs(got - ref_o) - tol):.3g}"
    lse_bad = np.abs(lse - ref_lse) > 2.0 ** -8 + 1e-5 * np.abs(ref_lse)
    assert not lse_bad.any(), f"{lse_bad.sum()} lse values outside the bound"
    return o, lse


# (q_lens, kv_lens, heads, kv heads): a single key; one query after a long
# prefix; a full 128-row tile; several tiles with a ragged tail behind a
# prefix that is not a multiple of 64; an empty request; MHA, GQA 2:1, 3:1
# and 4:1, MQA.  A call bound by its longest tile (all the small ones)
# runs one head per CTA; the last two, bound by their total work on a
# 152-SM GB300, run two heads of a key/value head per CTA.
CASES = [
    ((1, 17, 128, 200, 0, 64), (1, 100, 128, 700, 5, 128), 4, 2),
    ((300,), (300,), 2, 2),
    ((257, 3), (1000, 3), 8, 1),
    ((1, 1, 1), (1, 64, 65), 4, 1),
    ((130, 129, 63), (130, 1153, 200), 4, 4),
    ((100, 50), (300, 50), 6, 2),
    ((1000, 1024, 900, 1100), (1000, 1500, 900, 1300), 16, 2),
    ((700, 600, 650), (1500, 600, 900), 32, 2),
]


@pytest.mark.parametrize("q_lens,kv_lens,nh,nkv", CASES)
def test_attention_parity(bi, q_lens, kv_lens, nh, nkv):
    _check_parity(bi, q_lens, kv_lens, nh, nkv, seed=len(q_lens) * 31 + nh)


@pytest.mark.parametrize("q_lens,kv_lens,nh,nkv", [((150, 40), (400, 40), 2, 1), ((150, 40), (400, 40), 3, 3),
                                                    ((1024,) * 4, (1024,) * 4, 32, 4)])
def test_attention_parity_other_scale(bi, q_lens, kv_lens, nh, nkv):
    """A larger scale (peakier softmax: exponent gaps of tens), so that the
    rows' reference maxima move after the first block and O is rescaled in
    place, for warps where only some rows move; one head per CTA (the first
    two) and two (the last, bound by its total work)."""
    _check_parity(bi, q_lens, kv_lens, nh, nkv, seed=7, scale=0.5)


def _context(seed, n, nh=4, nkv=2):
    return synth.attention_inputs(seed, n, n, nh, nkv)


def test_suffix_equals_full_prefill(bi):
    """The last q_len queries of a 777-token context asked after a cached
    prefix give the bytes the full prefill gives them (tile boundaries fall
    elsewhere each time)."""
    n, nh, nkv = 777, 4, 2
    Q, K, V = _context(11, n, nh, nkv)
    full_o, full_l = _run(bi, Q, K, V, [0, n], [0, n], nh, nkv)
    for ql in (1, 63, 100, 129, 300, n - 64, n - 1):
        o, lse = _run(bi, Q[n - ql:], K, V, [0, ql], [0, n], nh, nkv)
        assert np.array_equal(o, full_o[n - ql:]), ql
        assert np.array_equal(lse.view(np.uint32), full_l[n - ql:].view(np.uint32)), ql


def test_chunked_prefill_equals_full_prefill(bi):
    """The context prefilled in chunks (each chunk's queries against the keys
    so far) gives the full prefill's bytes, for two different chunkings, and
    with all chunks as separate requests of one call."""
    n, nh, nkv = 777, 4, 2
    Q, K, V = _context(12, n, nh, nkv)
    full_o, _ = _run(bi, Q, K, V, [0, n], [0, n], nh, nkv)
    for cuts in ((0, 200, 450, n), (0, 1, 65, 128, 129, 640, n)):
        parts = []
        for a, b in zip(cuts[:-1], cuts[1:]):
            o, _ = _run(bi, Q[a:b], K[:b], V[:b], [0, b - a], [0, b], nh, nkv)
            parts.append(o)
        assert np.array_equal(np.concatenate(parts), full_o), cuts
        # all chunks in one call: request i = chunk i with its own copy of K, V[:b]
        qo = list(cuts)
        ko = [0] + list(np.cumsum(cuts[1:]))
        Kc = np.concatenate([K[:b] for b in cuts[1:]])
        Vc = np.concatenate([V[:b] for b in cuts[1:]])
        o, _ = _run(bi, Q, Kc, Vc, qo, ko, nh, nkv)
        assert np.array_equal(o, full_o), cuts


def test_batch_composition_does_not_matter(bi):
    """A request alone, and the same request between other requests of other
    lengths (so its rows sit at other token indices and other tiles run
    beside it): identical bytes."""
    nh, nkv = 4, 2
    ql, kl = 300, 777
    Q, K, V = synth.attention_inputs(13, ql, kl, nh, nkv)
    alone, alone_l = _run(bi, Q, K, V, [0, ql], [0, kl], nh, nkv)
    before, after = [(5, 90), (128, 128), (1, 2000)], [(77, 300), (200, 201)]
    parts_q, parts_k, parts_v, qo, ko = [], [], [], [0], [0]
    for i, (a, b) in enumerate(before + [(ql, kl)] + after):
        if i == len(before):
            q_, k_, v_ = Q, K, V
        else:
            q_, k_, v_ = synth.attention_inputs(100 + i, a, b, nh, nkv)
        parts_q.append(q_)
        parts_k.append(k_)
        parts_v.append(v_)
        qo.append(qo[-1] + a)
        ko.append(ko[-1] + b)
    o, lse = _run(bi, np.concatenate(parts_q), np.concatenate(parts_k), np.concatenate(parts_v), qo, ko, nh, nkv)
    j = len(before)
    assert np.array_equal(o[qo[j]:qo[j + 1]], alone)
    assert np.array_equal(lse[qo[j]:qo[j + 1]].view(np.uint32), alone_l.view(np.uint32))


def test_repeated_calls_and_graph_replay(bi):
    """Five back-to-back calls and CUDA-graph replays give the same bytes."""
    import torch
    qo, ko = [0, 100, 400], [0, 700, 1000]
    nh, nkv = 4, 2
    Q, K, V = synth.attention_inputs(14, 400, 1000, nh, nkv)
    ref, _ = _run(bi, Q, K, V, qo, ko, nh, nkv)
    q, k, v = gu.dev_bf16(Q), gu.dev_bf16(K), gu.dev_bf16(V)
    outs = [bi.attention_prefill(q, k, v, qo, ko, SCALE)[0] for _ in range(5)]
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(gu.host_bf16_bits(o), ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    o = torch.empty((400, nh, D), dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(s):
        bi.bi_attention_prefill(q, k, v, 2, qo, ko, nh, nkv, D, SCALE, o, None, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        bi.bi_attention_prefill(q, k, v, 2, qo, ko, nh, nkv, D, SCALE, o, None, stream=s)
    for _ in range(3):
        o.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(gu.host_bf16_bits(o), ref)
    assert bi.bi_get_last_device_error() == 0


def test_many_tiles_take_several_launches(bi):
    """More query tiles than one launch's table holds (512): the call is cut
    into several launches; every row still equals its own request run
    alone."""
    nh, nkv = 1, 1
    n_req = 600                      # 600 tiles of one query each... plus one big request
    q_lens = [1] * n_req + [256]
    kv_lens = [3] * n_req + [256]
    qo, ko = synth.attention_offsets(q_lens, np.asarray(kv_lens) - np.asarray(q_lens))
    Q, K, V = synth.attention_inputs(15, int(qo[-1]), int(ko[-1]), nh, nkv)
    o, _ = _run(bi, Q, K, V, qo, ko, nh, nkv)
    for r in (0, 1, 299, 599, 600):
        a, b, c, d = qo[r], qo[r + 1], ko[r], ko[r + 1]
        ro, _ = _run(bi, Q[a:b], K[c:d], V[c:d], [0, b - a], [0, d - c], nh, nkv)
        assert np.array_equal(o[a:b], ro), r


def test_full_workload_sampled_rows(bi):
    """The prefill workload (4096 queries in 8 requests behind cached
    prefixes of up to 3072 tokens, 16 query heads over 2 key/value heads):
    sampled rows of every request against the oracle run one query at a
    time, and the whole output finite."""
    import torch
    from oracle import attention as oatt
    nh, nkv = synth.ATTN_HEADS, synth.ATTN_KV_HEADS
    qo, ko = synth.attention_offsets(synth.ATTN_Q_LENS, synth.ATTN_PREFIX)
    Q, K, V = synth.attention_inputs(16, int(qo[-1]), int(ko[-1]), nh, nkv)
    o, lse = _run(bi, Q, K, V, qo, ko, nh, nkv)
    got = gu_bf16_to_f64(o)
    assert np.isfinite(got).all() and np.isfinite(lse).all()
    g = nh // nkv
    rng = np.random.default_rng(5)
    for r in range(len(qo) - 1):
        ql, kl = qo[r + 1] - qo[r], ko[r + 1] - ko[r]
        for i in sorted(set([0, ql - 1] + list(rng.integers(0, ql, 2)))):
            pos = kl - ql + i
            t = qo[r] + i
            ks = slice(ko[r], ko[r] + pos + 1)
            ref_o, ref_l = oatt.attention_prefill(Q[t:t + 1], np.repeat(K[ks], g, axis=1),
                                                  np.repeat(V[ks], g, axis=1), [0, 1], [0, pos + 1], SCALE)
            vmax = np.abs(gu_bf16_to_f64(V[ks])).max(axis=(0, 2))
            tol = 1.05 * 2.0 ** -8 * np.repeat(vmax, g)[:, None] + 2.0 ** -8 * np.abs(ref_o[0])
            assert (np.abs(got[t] - ref_o[0]) <= tol).all(), (r, i)
            assert (np.abs(lse[t] - ref_l[0]) <= 2.0 ** -8 + 1e-5 * np.abs(ref_l[0])).all(), (r, i)


def test_rejects_bad_calls_on_device(bi):
    """Argument errors come back as status codes and launch nothing."""
    import torch
    q = torch.zeros((4, 4, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((8, 2, D), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((4, 4, D), dtype=torch.bfloat16, device="cuda")
    assert bi.bi_attention_prefill(q, k, k, 1, [0, 4], [0, 8], 4, 2, 64, SCALE, o, check=False) == \
        bi.BI_ERR_UNSUPPORTED_SHAPE
    assert bi.bi_attention_prefill(q, k, k, 1, [0, 4], [0, 3], 4, 2, D, SCALE, o, check=False) == \
        bi.BI_ERR_INVALID_ARG
    assert bi.bi_attention_prefill(q, k, k, 1, [0, 4], [0, 8], 4, 3, D, SCALE, o, check=False) == \
        bi.BI_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0


def test_one_head_and_two_head_ctas_give_the_same_bytes(bi):
    """A 4096-token full prefill (32 tiles x 16 heads, bound by its total
    work) runs two heads of a key/value head per CTA; its last 128 queries,
    a chunk in the middle and its first 300 queries asked alone run one head
    per CTA (each bound by its longest tile).  Same rows, same bytes."""
    n, nh, nkv = 4096, 16, 2
    Q, K, V = synth.attention_inputs(17, n, n, nh, nkv)
    o, lse = _run(bi, Q, K, V, [0, n], [0, n], nh, nkv)
    for a, b in ((n - 128, n), (1000, 1300), (0, 300)):
        ro, rl = _run(bi, Q[a:b], K[:b], V[:b], [0, b - a], [0, b], nh, nkv)
        assert np.array_equal(o[a:b], ro), (a, b)
        assert np.array_equal(lse[a:b].view(np.uint32), rl.view(np.uint32)), (a, b)


def test_max_heads_and_long_context(bi):
    """The largest shapes the call accepts, checked where the oracle can
    afford it: BI_ATTN_MAX_HEADS (256) query heads over 32 key/value heads on
    a small ragged batch, against the oracle element by element; and one
    65536-token context (16 over 2 heads, 512 query tiles: one full table of
    a launch) on sampled rows against the oracle run one query at a time,
    with its last 100 queries asked again after the cached prefix."""
    from oracle import attention as oatt
    assert bi.BI_ATTN_MAX_HEADS == 256
    _check_parity(bi, (130, 7), (300, 7), 256, 32, seed=21)

    n, nh, nkv = 65536, 16, 2
    Q, K, V = synth.attention_inputs(22, n, n, nh, nkv)
    o, lse = _run(bi, Q, K, V, [0, n], [0, n], nh, nkv)
    got = gu_bf16_to_f64(o)
    assert np.isfinite(got).all() and np.isfinite(lse).all()
    g = nh // nkv
    for i in (0, 1, 127, 128, 16383, 16384, 40000, n - 1):
        for h in (0, 5, 8, 15):                      # both key/value heads; one head at a time
            hk = h // g
            ref_o, ref_l = oatt.attention_prefill(Q[i:i + 1, h:h + 1], K[:i + 1, hk:hk + 1], V[:i + 1, hk:hk + 1],
                                                  [0, 1], [0, i + 1], SCALE)
            vmax = np.abs(gu_bf16_to_f64(V[:i + 1, hk])).max()
            tol = 1.05 * 2.0 ** -8 * vmax + 2.0 ** -8 * np.abs(ref_o[0, 0])
            assert (np.abs(got[i, h] - ref_o[0, 0]) <= tol).all(), (i, h)
            assert abs(lse[i, h] - ref_l[0, 0]) <= 2.0 ** -8 + 1e-5 * abs(ref_l[0, 0]), (i, h)
    suf, suf_l = _run(bi, Q[n - 100:], K, V, [0, 100], [0, n], nh, nkv)
    assert np.array_equal(suf, o[n - 100:])
    assert np.array_equal(suf_l.view(np.uint32), lse[n - 100:].view(np.uint32))


def _oracle_rows(Q, K, V, rows_pos, heads, g, scale=SCALE):
    """The oracle one query and head at a time: rows_pos = [(row in Q, position)]."""
    from oracle import attention as oatt
    out = {}
    for r, p in rows_pos:
        for h in heads:
            hk = h // g
            ro, rl = oatt.attention_prefill(Q[r:r + 1, h:h + 1], K[:p + 1, hk:hk + 1], V[:p + 1, hk:hk + 1],
                                            [0, 1], [0, p + 1], scale)
            vmax = np.abs(gu_bf16_to_f64(V[:p + 1, hk])).max()
            out[(r, h)] = (ro[0, 0], rl[0, 0], vmax)
    return out


def _check_rows(o, lse, ref):
    got = gu_bf16_to_f64(o)
    for (r, h), (ro, rl, vmax) in ref.items():
        tol = 1.05 * 2.0 ** -8 * vmax + 2.0 ** -8 * np.abs(ro)
        assert (np.abs(got[r, h] - ro) <= tol).all(), (r, h)
        assert abs(lse[r, h] - rl) <= 2.0 ** -8 + 1e-5 * abs(rl), (r, h)


def test_chunked_context_parity_and_invariance(bi):
    """Past 8192 keys a row's context is computed in 8192-key chunks merged
    in order.  An 8300-token context: rows just below and above the chunk
    boundary against the oracle; the full prefill, two suffixes (one whose
    tile straddles the boundary, one entirely past it) and a prefill chunked
    across the boundary give the same bytes."""
    n, nh, nkv = 8300, 4, 2
    Q, K, V = _context(31, n, nh, nkv)
    full, full_l = _run(bi, Q, K, V, [0, n], [0, n], nh, nkv)
    rows = [0, 8063, 8064, 8191, 8192, 8193, 8255, 8256, n - 1]
    _check_rows(full, full_l, _oracle_rows(Q, K, V, [(r, r) for r in rows], range(nh), nh // nkv))
    for ql in (150, 50):
        o, lse = _run(bi, Q[n - ql:], K, V, [0, ql], [0, n], nh, nkv)
        assert np.array_equal(o, full[n - ql:]), ql
        assert np.array_equal(lse.view(np.uint32), full_l[n - ql:].view(np.uint32)), ql
    parts = []
    for a, b in ((0, 8100), (8100, 8200), (8200, n)):
        o, _ = _run(bi, Q[a:b], K[:b], V[:b], [0, b - a], [0, b], nh, nkv)
        parts.append(o)
    assert np.array_equal(np.concatenate(parts), full)


def test_long_prefix_cache_hit(bi):
    """One request's prefix-cache hit: 128 queries behind 20000 cached tokens
    (three chunks, 16 query heads over 2), against the oracle on sampled rows
    and heads, and the same rows inside a batch with a short request."""
    nh, nkv = 16, 2
    pre, nq = 20000, 128
    Q, K, V = synth.attention_inputs(32, nq, pre + nq, nh, nkv)
    o, lse = _run(bi, Q, K, V, [0, nq], [0, pre + nq], nh, nkv)
    ref = _oracle_rows(Q, K, V, [(r, pre + r) for r in (0, 1, 63, 127)], (0, 7, 8, 15), nh // nkv)
    _check_rows(o, lse, ref)
    Qs, Ks, Vs = synth.attention_inputs(33, 40, 300, nh, nkv)
    ob, lb = _run(bi, np.concatenate([Qs, Q]), np.concatenate([Ks, K]), np.concatenate([Vs, V]),
                  [0, 40, 40 + nq], [0, 300, 300 + pre + nq], nh, nkv)
    assert np.array_equal(ob[40:], o)
    assert np.array_equal(lb[40:].view(np.uint32), lse.view(np.uint32))


def test_walked_and_split_chunks_give_the_same_bytes(bi):
    """A 16384-token prefill (bound by its total work) walks each long tile's
    chunks in one CTA, merging as it goes; its last 200 queries asked alone
    (bound by their longest tile) run each chunk in its own CTA and merge
    them in a second kernel.  Same rows, same bytes; rows on both sides of
    the chunk boundary against the oracle."""
    n, nh, nkv = 16384, 16, 2
    Q, K, V = synth.attention_inputs(34, n, n, nh, nkv)
    o, lse = _run(bi, Q, K, V, [0, n], [0, n], nh, nkv)
    so, sl = _run(bi, Q[n - 200:], K, V, [0, 200], [0, n], nh, nkv)
    assert np.array_equal(so, o[n - 200:])
    assert np.array_equal(sl.view(np.uint32), lse[n - 200:].view(np.uint32))
    ref = _oracle_rows(Q, K, V, [(r, r) for r in (8191, 8192, 12000, n - 1)], (0, 9), nh // nkv)
    _check_rows(o, lse, ref)


def test_walked_tile_across_the_chunk_boundary(bi):
    """A call bound by its total work (5000 queries behind 5000 cached
    tokens, 40 tiles x 8 head pairs) walks its long tiles; tile 24 holds
    positions 8072..8199, across the first chunk boundary, so its rows finish
    at two different chunk ends of one walk.  The same rows asked alone (a
    few tiles: chunk CTAs and the merge kernel) give the same bytes; rows on
    both sides of position 8192 against the oracle."""
    nh, nkv = 16, 2
    ql, kl = 5000, 10000
    Q, K, V = synth.attention_inputs(35, ql, kl, nh, nkv)
    o, lse = _run(bi, Q, K, V, [0, ql], [0, kl], nh, nkv)
    a, b = 3000, 3250                                # positions 8000 .. 8249
    so, sl = _run(bi, Q[a:b], K[:kl - ql + b], V[:kl - ql + b], [0, b - a], [0, kl - ql + b], nh, nkv)
    assert np.array_equal(so, o[a:b])
    assert np.array_equal(sl.view(np.uint32), lse[a:b].view(np.uint32))
    rows = [(r, kl - ql + r) for r in (3191, 3192, 3199, 3200)]     # positions 8191, 8192, 8199, 8200
    _check_rows(o, lse, _oracle_rows(Q, K, V, rows, (0, 15), nh // nkv))
