"""Oracle for batch-invariant prefill attention (TEST INFRASTRUCTURE ONLY:
imported by the test suite alone; it shares no code with the library).

Source: "The Illusion of Determinism in Disaggregated Inference", section
"The physics of the cascade": once a one-ULP difference reaches attention,
the softmax's exponential stretches it and the product with the value
matrix spreads it over every feature, so attention is the next operation on
the cascade path after RMSNorm that must not depend on the batch; the same
page's references list attention among the kernels a batch-invariant engine
rewrites.  The pages fix no attention variant; read here as causal
self-attention over ragged requests, the form a prefill runs:

  request r has q_len[r] queries (the suffix of its context) and kv_len[r]
  keys and values (the whole context, prefix included, q_len <= kv_len);
  query i sits at position kv_len - q_len + i and attends to keys 0 .. that
  position:

      s_ij  = scale * (q_i . k_j)           for j <= pos(i), else -inf
      p_ij  = exp(s_ij - max_j s_ij) / sum_j exp(s_ij - max_j s_ij)
      o_i   = sum_j p_ij v_j

computed exactly in double from the inputs' values (bf16 patterns widened),
head by head.  Nothing in it depends on the other requests or on how many of
a request's queries are asked for at once.
"""
from __future__ import annotations

import numpy as np

from oracle import oracle as orc


def _widen(a):
    a = np.asarray(a)
    return orc.bf16_to_double(a) if a.dtype == np.uint16 else a.astype(np.float64)


def positions(q_len: int, kv_len: int):
    """Context positions of a request's queries: the last q_len of kv_len."""
    return kv_len - q_len + np.arange(q_len)


def visible(q_len: int, kv_len: int):
    """[q_len, kv_len] boolean: key j visible to query i (causal)."""
    return np.arange(kv_len)[None, :] <= positions(q_len, kv_len)[:, None]


def head_attention(q, k, v, scale: float):
    """One request, one head: q [q_len, D], k and v [kv_len, D] (double).
    Returns o [q_len, D] (double) and the log-sum-exp of each row's scores."""
    q_len, kv_len = q.shape[0], k.shape[0]
    s = scale * (q @ k.T)
    s = np.where(visible(q_len, kv_len), s, -np.inf)
    mx = s.max(axis=1, keepdims=True)
    e = np.exp(s - mx)
    den = e.sum(axis=1, keepdims=True)
    return (e / den) @ v, (mx + np.log(den))[:, 0]


def attention_prefill(Q, K, V, q_offsets, kv_offsets, scale: float):
    """Q [Tq, heads, D], K and V [Tkv, heads, D] (float32 or bf16 patterns).
    Request r: queries Q[q_offsets[r]:q_offsets[r+1]], keys and values
    K/V[kv_offsets[r]:kv_offsets[r+1]].  Returns o double [Tq, heads, D] and
    lse double [Tq, heads]."""
    q, k, v = _widen(Q), _widen(K), _widen(V)
    heads = q.shape[1]
    o = np.zeros(q.shape, dtype=np.float64)
    lse = np.zeros(q.shape[:2], dtype=np.float64)
    for r in range(len(q_offsets) - 1):
        qs, qe = int(q_offsets[r]), int(q_offsets[r + 1])
        ks, ke = int(kv_offsets[r]), int(kv_offsets[r + 1])
        if qe == qs:
            continue
        for h in range(heads):
            o[qs:qe, h], lse[qs:qe, h] = head_attention(q[qs:qe, h], k[ks:ke, h], v[ks:ke, h], scale)
    return o, lse


def brute_force_row(q_i, k, v, pos: int, scale: float):
    """One query row by explicit loops (the definition term by term, for tiny
    pins): max over visible keys, exponentials, their sum, weighted values."""
    scores = []
    for j in range(pos + 1):
        acc = 0.0
        for d in range(len(q_i)):
            acc += float(q_i[d]) * float(k[j][d])
        scores.append(scale * acc)
    m = max(scores)
    ex = [np.exp(sv - m) for sv in scores]
    den = sum(ex)
    out = [0.0] * len(q_i)
    for j, e in enumerate(ex):
        for d in range(len(q_i)):
            out[d] += e / den * float(v[j][d])
    return np.array(out)
