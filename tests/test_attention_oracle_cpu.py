"""Pins for the attention oracle (oracle/attention.py): closed forms, brute
force and structural facts that hold for exact attention, each chosen so
that a plausible mistake in the oracle (a dropped scale, an off-by-one in
the causal mask, positions that ignore the prefix, a missing normalisation
or max shift) turns one of them red; the mutants at the end plant exactly
those mistakes.

Source: "The Illusion of Determinism in Disaggregated Inference", section
"The physics of the cascade" (softmax attention is the next amplifier on the
cascade path); the variant is causal prefill attention over ragged
requests, the suffix of each context asking."""
import types

import numpy as np
import pytest

from oracle import attention as att_module

rng = np.random.default_rng(20261202)


def _req(q_len, kv_len, heads=2, D=8, scale=0.3, seed=0):
    g = np.random.default_rng(seed)
    Q = g.standard_normal((q_len, heads, D)).astype(np.float32)
    K = g.standard_normal((kv_len, heads, D)).astype(np.float32)
    V = g.standard_normal((kv_len, heads, D)).astype(np.float32)
    return Q, K, V, np.array([0, q_len]), np.array([0, kv_len]), scale


def pin_single_key(att):
    """One key: every query's output is that key's value row, exactly."""
    Q, K, V, qo, ko, sc = _req(1, 1, seed=1)
    o, lse = att.attention_prefill(Q, K, V, qo, ko, sc)
    assert np.array_equal(o[0], V[0].astype(np.float64))
    for h in range(Q.shape[1]):
        assert lse[0, h] == sc * float(np.dot(Q[0, h].astype(np.float64), K[0, h].astype(np.float64)))


def pin_first_query_of_full_prefill(att):
    """q_len == kv_len: query 0 sees key 0 only."""
    Q, K, V, qo, ko, sc = _req(7, 7, seed=2)
    o, _ = att.attention_prefill(Q, K, V, qo, ko, sc)
    assert np.array_equal(o[0], V[0].astype(np.float64))


def pin_constant_keys_average(att):
    """All keys equal: uniform weights over the visible keys, so query i's
    output is the mean of the visible value rows (the prefix means)."""
    q_len, kv_len = 5, 9
    Q, K, V, qo, ko, sc = _req(q_len, kv_len, seed=3)
    K[:] = K[0:1]
    o, lse = att.attention_prefill(Q, K, V, qo, ko, sc)
    pos = kv_len - q_len + np.arange(q_len)
    for i in range(q_len):
        want = V[:pos[i] + 1].astype(np.float64).mean(axis=0)
        assert np.allclose(o[i], want, rtol=1e-12, atol=1e-14)
        for h in range(Q.shape[1]):
            s = sc * float(np.dot(Q[i, h].astype(np.float64), K[0, h].astype(np.float64)))
            assert abs(lse[i, h] - (s + np.log(pos[i] + 1))) <= 1e-12 * (1 + abs(s))


def pin_zero_scale_average(att):
    """scale = 0: every visible key weighs the same."""
    q_len, kv_len = 4, 6
    Q, K, V, qo, ko, _ = _req(q_len, kv_len, seed=4)
    o, _ = att.attention_prefill(Q, K, V, qo, ko, 0.0)
    pos = kv_len - q_len + np.arange(q_len)
    for i in range(q_len):
        assert np.allclose(o[i], V[:pos[i] + 1].astype(np.float64).mean(axis=0), rtol=1e-12, atol=1e-14)


def pin_dominant_key(att):
    """A key whose score exceeds every other visible score by more than 800
    (exp of the gap underflows to exactly 0 in double): the output is that
    key's value row exactly."""
    D = 4
    Q = np.zeros((1, 1, D), np.float32)
    Q[0, 0, 0] = 1.0
    K = np.zeros((6, 1, D), np.float32)
    K[3, 0, 0] = 1000.0
    V = rng.standard_normal((6, 1, D)).astype(np.float32)
    o, _ = att.attention_prefill(Q, K, V, np.array([0, 1]), np.array([0, 6]), 1.0)
    assert np.array_equal(o[0, 0], V[3, 0].astype(np.float64))


def pin_brute_force(att):
    """Tiny ragged case against the definition term by term."""
    Q, K, V, qo, ko, sc = _req(3, 5, heads=2, D=4, seed=5)
    o, _ = att.attention_prefill(Q, K, V, qo, ko, sc)
    for i in range(3):
        for h in range(2):
            want = att.brute_force_row(Q[i, h], K[:, h], V[:, h], 5 - 3 + i, sc)
            assert np.allclose(o[i, h], want, rtol=1e-12, atol=1e-13)


def pin_suffix_is_full_prefill_tail(att):
    """Asking for the last q_len queries of a context gives the rows the
    full prefill gives them (the queries sit after the prefix)."""
    kv_len, q_len = 11, 4
    Q, K, V, _, ko, sc = _req(kv_len, kv_len, seed=6)
    full, _ = att.attention_prefill(Q, K, V, np.array([0, kv_len]), ko, sc)
    suf, _ = att.attention_prefill(Q[kv_len - q_len:], K, V, np.array([0, q_len]), ko, sc)
    assert np.allclose(suf, full[kv_len - q_len:], rtol=1e-12, atol=1e-14)


def pin_requests_independent(att):
    """Two requests in one call give each request's rows alone."""
    Qa, Ka, Va, qa, ka, sc = _req(3, 6, seed=7)
    Qb, Kb, Vb, qb, kb, _ = _req(2, 2, seed=8)
    oa, _ = att.attention_prefill(Qa, Ka, Va, qa, ka, sc)
    ob, _ = att.attention_prefill(Qb, Kb, Vb, qb, kb, sc)
    o, _ = att.attention_prefill(np.concatenate([Qa, Qb]), np.concatenate([Ka, Kb]), np.concatenate([Va, Vb]),
                                 np.array([0, 3, 5]), np.array([0, 6, 8]), sc)
    assert np.allclose(o[:3], oa, rtol=1e-12, atol=1e-14) and np.allclose(o[3:], ob, rtol=1e-12, atol=1e-14)


PINS = [pin_single_key, pin_first_query_of_full_prefill, pin_constant_keys_average, pin_zero_scale_average,
        pin_dominant_key, pin_brute_force, pin_suffix_is_full_prefill_tail, pin_requests_independent]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(att_module)


# Each mutant plants one plausible mistake in a copy of the oracle's source
# and must turn at least one pin red.
MUTANTS = {
    "diagonal_masked": ("<= positions(q_len, kv_len)[:, None]", "< positions(q_len, kv_len)[:, None]"),
    "positions_ignore_prefix": ("return kv_len - q_len + np.arange(q_len)", "return np.arange(q_len)"),
    "scale_dropped": ("s = scale * (q @ k.T)", "s = q @ k.T"),
    "no_max_shift": ("e = np.exp(s - mx)", "e = np.exp(s)"),
    "not_normalised": ("return (e / den) @ v", "return e @ v"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    import inspect
    src = inspect.getsource(att_module)
    old, new = MUTANTS[name]
    assert src.count(old) == 1, "the planted mistake must apply exactly once"
    mod = types.ModuleType(f"attention_{name}")
    with np.errstate(all="ignore"):
        exec(compile(src.replace(old, new), f"<{name}>", "exec"), mod.__dict__)
        failed = []
        for pin in PINS:
            try:
                pin(mod)
            except (AssertionError, FloatingPointError, ValueError):
                failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
