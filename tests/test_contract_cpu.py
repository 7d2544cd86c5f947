"""bi_get_config and bi_prefix_split: host-only entry points, run without a
GPU.

bi_get_config must report the contract every kernel is compiled with (the
values the header documents, and that the GPU tests hold the kernels to);
bi_prefix_split must give, per request of N tokens and KV block size B, the
rows a prefix-cache hit recomputes: N mod B of them, the last full block when
that is 0, the whole request when N < B ("The Illusion of Determinism in
Disaggregated Inference", "The engineering cost of determinism")."""
import ctypes as C

import numpy as np
import pytest

from serving_numerics_gb300 import binding


@pytest.fixture(scope="module")
def lib():
    from serving_numerics_gb300 import build
    build.build()
    return binding.load()


def test_config_reports_the_contract(lib):
    c = binding.get_config()
    assert c["struct_size"] == C.sizeof(binding.BiConfig)
    assert c["abi_version"] == lib.bi_abi_version() == 2
    assert (c["router_slab"], c["router_block"], c["router_partitions"]) == (128, 8, 16)
    assert c["router_slab"] == c["router_block"] * c["router_partitions"]
    assert c["router_partition_order"] == 1 and c["router_tree"] == binding.BI_TREE_PAIRWISE
    assert c["router_accum"] == binding.BI_F32 and c["gemm_accum"] == binding.BI_F32
    assert (c["gemm_tile_m"], c["gemm_tile_n"], c["gemm_block_k"], c["gemm_mma_k"]) == (128, 256, 64, 16)
    assert c["gemm_split_k"] == 0
    assert c["topk_tie_rule"] == 1 and c["softmax_sum_order"] == 1


def test_config_short_buffer_and_null(lib):
    buf = (C.c_int32 * 4)(-1, -1, -1, -1)
    assert lib.bi_get_config(buf, 8) == binding.BI_OK          # only the first two fields
    assert list(buf) == [C.sizeof(binding.BiConfig), 2, -1, -1]
    assert lib.bi_get_config(buf, 7) == binding.BI_ERR_INVALID_ARG
    assert lib.bi_get_config(None, 64) == binding.BI_ERR_INVALID_ARG


def suffix_rows(n, b):
    """The pages' rule, restated: a miss runs N rows; a hit keeps whole
    blocks and runs the rest, at least one block's worth when N >= B."""
    if n == 0:
        return 0
    r = n % b
    return r if r else b


@pytest.mark.parametrize("block", [1, 16, 64])
def test_prefix_split_matches_the_rule(lib, block):
    g = np.random.default_rng(block)
    lens = [0, 1, block - 1 if block > 1 else 1, block, block + 1, 2 * block, 300] + \
        list(g.integers(0, 1000, 40))
    cached, offs = binding.prefix_split(lens, block)
    assert offs[0] == 0 and len(offs) == len(lens) + 1
    for r, n in enumerate(lens):
        s = suffix_rows(n, block)
        assert cached[r] == n - s, (n, block)
        assert cached[r] % block == 0 and 0 <= cached[r] <= n
        assert offs[r + 1] - offs[r] == s
    assert offs[-1] == sum(suffix_rows(n, block) for n in lens)


def test_prefix_split_worked_example(lib):
    # block 16: 37 tokens keep 32 and recompute 5; 48 keep 32 and recompute
    # the last full block; 7 recompute all 7; 0 recompute nothing
    cached, offs = binding.prefix_split([37, 48, 7, 0], 16)
    assert cached == [32, 32, 0, 0]
    assert offs == [0, 5, 21, 28, 28]


def test_prefix_split_validation(lib):
    arr = (C.c_int32 * 2)(5, -1)
    out = (C.c_int32 * 2)()
    offs = (C.c_int32 * 3)(7, 7, 7)
    assert lib.bi_prefix_split(arr, 2, 16, out, offs) == binding.BI_ERR_INVALID_ARG
    assert list(offs) == [7, 7, 7]                               # outputs untouched
    arr2 = (C.c_int32 * 2)(5, 6)
    assert lib.bi_prefix_split(arr2, 2, 0, out, offs) == binding.BI_ERR_INVALID_ARG
    assert lib.bi_prefix_split(arr2, -1, 16, out, offs) == binding.BI_ERR_INVALID_ARG
    assert lib.bi_prefix_split(None, 2, 16, out, offs) == binding.BI_ERR_INVALID_ARG
    big = (C.c_int32 * 2)(2**31 - 1, 5)
    assert lib.bi_prefix_split(big, 2, 16, out, offs) == binding.BI_ERR_INVALID_ARG
    assert lib.bi_prefix_split(arr2, 0, 16, out, offs) == binding.BI_OK and offs[0] == 0


# ---------------------------------------------------------------------------
# The contract emulator (oracle/contract.c) pinned by hand-worked examples:
# x = 1 everywhere, so every product is exact and each step is one f32
# addition; 2^24 + 1 is a tie that rounds to the even 2^24, so a 1 added to
# 2^24 alone is lost, while 1s summed among themselves first survive.
# ---------------------------------------------------------------------------
BIG = 2.0 ** 24


def _row(H, entries):
    w = np.zeros((1, H), np.float32)
    for h, v in entries.items():
        w[0, h] = v
    return np.ones((1, H), np.float32), w


def test_contract_blocks_of_eight_go_to_partitions():
    """2^24 at h = 0 and 1s at h = 8..15: partition 0 holds 2^24 and
    partition 1 sums the eight 1s to 8, so the tree gives 2^24 + 8 exactly.
    One chain over h would lose every 1 (2^24)."""
    from oracle import contract
    x, w = _row(16, {0: BIG, **{h: 1.0 for h in range(8, 16)}})
    assert contract.router_logits(x, w)[0, 0] == np.float32(BIG + 8)


def test_contract_partition_owns_the_same_block_of_every_slab():
    """2^24 at h = 0 and 1s at h = 128..135 (block 0 of slab 1): both belong
    to partition 0's chain, so each 1 meets 2^24 alone and is lost: 2^24.
    Contiguous ranges of 16 per partition would put the 1s in partition 8
    and give 2^24 + 8."""
    from oracle import contract
    x, w = _row(256, {0: BIG, **{h: 1.0 for h in range(128, 136)}})
    assert contract.router_logits(x, w)[0, 0] == np.float32(BIG)


def test_contract_partials_meet_in_the_pairwise_tree():
    """2^24 in partition 0 and a single 1 in partitions 1, 2, 3: the first
    level gives 2^24 + 1 -> 2^24 and 1 + 1 = 2, the second 2^24 + 2.  A
    sequential sum of the partials would give 2^24, the exact sum rounded to
    f32 gives 2^24 + 4."""
    from oracle import contract
    x, w = _row(32, {0: BIG, 8: 1.0, 16: 1.0, 24: 1.0})
    assert contract.router_logits(x, w)[0, 0] == np.float32(BIG + 2)


def test_contract_exact_on_integer_grid_and_within_f32_bound(orc):
    """On an integer grid every order is exact, so the emulator must equal
    the oracle's double dot; on normal draws it must stay within the f32
    error bound of a chain of H/16 steps and a 4-level tree."""
    from oracle import contract
    g = np.random.default_rng(5)
    for H in (8, 136, 264, 2048):
        X = (g.integers(-8, 9, (6, H)) * 2.0 ** -4).astype(np.float32)
        W = (g.integers(-8, 9, (5, H)) * 2.0 ** -4).astype(np.float32)
        assert np.array_equal(contract.router_logits(X, W).astype(np.float64), orc.router_logits(X, W))
        Xn = g.standard_normal((6, H)).astype(np.float32)
        Wn = (0.02 * g.standard_normal((5, H))).astype(np.float32)
        exact = orc.router_logits(Xn, Wn)
        bound = (H / 16 + 4 + 1) * 2.0 ** -24 * orc.router_absdot(Xn, Wn)
        assert np.all(np.abs(contract.router_logits(Xn, Wn) - exact) <= bound)
