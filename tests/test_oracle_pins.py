"""The CPU oracle against its pins (closed forms, brute force, exact integer
arithmetic, published FNV vectors).  No GPU."""
import numpy as np
import pytest

from tests import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_tie_heavy_workload_tie_rate(orc):
    """The synthetic tie-heavy workload (E=512, k=10, 48 calls x 5 tokens)
    has about a third of its token-slots at an exact bf16 tie on the
    k-boundary, as measured on the page ("diag(MODEL-MM-QWEN4-EXP) ...",
    intro: 79 of 240).  Self-counting: 48 * 5 = 240 slots are visited."""
    from serving_numerics_gb300 import synth
    slots = ties = 0
    for call in range(48):
        X, W = synth.tie_heavy_call(0, call)
        r = orc.router_full(X, W, synth.TIE512["k"], "bf16")
        slots += len(r["margin_ulps"])
        ties += int(np.sum(r["margin_ulps"] == 0))
        assert np.all((r["margin_ulps"] == 0) == (r["margin"] == 0.0))
    assert slots == 240
    assert ties == 78
