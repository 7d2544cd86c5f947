"""Mutation proofs for the oracle's pins.

Each mutant plants one plausible mistake in a copy of oracle.c (a flipped
tie-break, an unsorted hash, two's-complement instead of sign-magnitude
ULPs, ties-away rounding, a dropped term, a wrong prime ...), is built with
the same compiler command (rc=0 checked, so a broken build cannot pass for a
caught mutant), and must turn at least one pin red.  The substitution is
asserted to apply exactly once: the applied-proof count of the mutation
table in "diag(MODEL-MM-QWEN4-EXP) ...", section "Gates, read literally".
"""
import os
import subprocess

import pytest

from tests import pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "tiebreak_highest_index": ("    return a > b;\n}", "    return a >= b;\n}"),
    "hash_selection_order": ("while (b >= 0 && srt[b] > v)", "while (0 && srt[b] > v)"),
    "ulp_twos_complement": ("return (b & 0x8000u) ? -(int64_t)(b & 0x7FFFu) : (int64_t)b;",
                            "return (int64_t)(int16_t)b;"),
    "round_ties_away": ("(frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))", "(frac >= 0.5)"),
    "router_drop_last_term": (
        "for (int64_t h = 0; h < H; ++h)\n                s += (double)X[m * ldx + h] * (double)W[e * ldw + h];",
        "for (int64_t h = 0; h < H - 1; ++h)\n                s += (double)X[m * ldx + h] * (double)W[e * ldw + h];"),
    "margin_sign": ("margin[m] = row[smin] - row[rmax];\n        ulps[m] = orc_ord_bf16",
                    "margin[m] = row[rmax] - row[smin];\n        ulps[m] = orc_ord_bf16"),
    "softmax_den_start": ("double den = 0.0;", "double den = 1.0;"),
    "gemm_drop_last_k": ("for (int64_t kk = 0; kk < K; ++kk)", "for (int64_t kk = 0; kk < K - 1; ++kk)"),
    "fnv_wrong_prime": ("#define ORC_FNV64_PRIME 0x00000100000001B3ull",
                        "#define ORC_FNV64_PRIME 0x00000100000001B1ull"),
    "gate_sigmoid_sign": ("sig[m] = 1.0 / (1.0 + exp(-s));", "sig[m] = 1.0 / (1.0 + exp(s));"),
    "gate_drop_last_term": (
        "for (int64_t h = 0; h < H; ++h)\n            s += (double)X[m * ldx + h] * (double)w[h];",
        "for (int64_t h = 0; h < H - 1; ++h)\n            s += (double)X[m * ldx + h] * (double)w[h];"),
    "gate_w_indexed_by_row": ("s += (double)X[m * ldx + h] * (double)w[h];",
                              "s += (double)X[m * ldx + h] * (double)w[m];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, orc):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation {name} must apply exactly once"
    mut = tmp_path / "oracle_mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    rc = subprocess.run(["gcc", *orc.CFLAGS, str(mut), "-o", str(so), "-lm"]).returncode
    assert rc == 0, "the mutant must build, or a red test would prove nothing"
    failed = []
    with orc.use(str(so)):
        for pin in pins.ALL_PINS:
            try:
                pin(orc)
            except AssertionError:
                failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
