"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and rejects invalid arguments on the host before any CUDA
call (so these calls are safe on a machine with no GPU)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bi.h")


@pytest.fixture(scope="module")
def lib():
    from serving_numerics_gb300 import binding, build
    build.build()
    return binding.load()


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"BI_API\s+[\w\s\*]+?\b(bi_\w+)\s*\(", txt)))


def test_header_declares_the_abi():
    names = declared_symbols()
    for want in ("bi_router_topk", "bi_shared_gate", "bi_gemm_bf16", "bi_route_trace_hash", "bi_selftest_wait_timeout",
                 "bi_status_string", "bi_get_last_device_error", "bi_abi_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    from serving_numerics_gb300 import binding
    for name in declared_symbols():
        assert hasattr(lib, name), f"libbi.so does not export {name}"
        assert name in binding.SIGNATURES, f"binding lacks {name}"
    assert lib.bi_abi_version() == 2


def test_status_strings(lib):
    from serving_numerics_gb300 import binding as b
    for st in range(6):
        assert b.status_string(st).startswith("BI_")


FAKE = 0x10000          # never dereferenced: every call below fails validation first
MIS = FAKE + 4          # not 16-byte aligned


def _router(lib, **kw):
    a = dict(x=FAKE, w=FAKE, ind=0, ld=0, M=4, H=256, E=64, k=4, logits=FAKE, ids=FAKE,
             weights=None, margin=None, ulps=None, ws=None, wsb=0)
    a.update(kw)
    return lib.bi_router_topk(a["x"], a["w"], a["ind"], a["ld"], a["M"], a["H"], a["E"], a["k"],
                              a["logits"], a["ids"], a["weights"], a["margin"], a["ulps"], a["ws"], a["wsb"],
                              None)


@pytest.mark.parametrize("kw,want", [
    (dict(M=-1), 1), (dict(k=0), 1), (dict(k=64), 1), (dict(H=0), 1), (dict(E=0), 1),
    (dict(ind=2), 1), (dict(ld=7), 1),
    (dict(H=260), 2), (dict(E=48), 2), (dict(E=2048), 2), (dict(k=33, E=64), 2), (dict(H=40000), 2),
    (dict(x=None), 1), (dict(ids=None), 1), (dict(logits=None), 1),
    (dict(x=MIS), 3), (dict(w=MIS), 3), (dict(ids=FAKE + 2), 3),
])
def test_router_validation(lib, kw, want):
    assert _router(lib, **kw) == want


def test_router_m0_is_noop(lib):
    assert _router(lib, M=0, x=None, w=None, logits=None, ids=None) == 0


def test_router_workspace_bytes(lib):
    """No workspace for the one-launch cluster router (M <= 112, E <= 512);
    above that the bound of the tiled plans, the same on every GPU."""
    for M, E in ((1, 256), (64, 256), (112, 256), (112, 512), (5, 512)):
        assert lib.bi_router_workspace_bytes(M, E) == 0
    assert lib.bi_router_workspace_bytes(113, 256) == 113 * 256 * 64
    assert lib.bi_router_workspace_bytes(0, 256) == 0
    assert lib.bi_router_workspace_bytes(-3, 256) == 0
    # two-block plan: 8*M*E within its 64 MiB cap, never below the tail
    # plan's min(64*M*E, 16 MiB)
    assert lib.bi_router_workspace_bytes(129, 256) == 129 * 256 * 64
    assert lib.bi_router_workspace_bytes(960, 256) == 64 * 960 * 256   # 120 items: below the persistent plan
    # persistent plan (at least 128 items of 64 x 64 x 8 partitions): epoch
    # and flags (16 KB), 128 KB of hand-off and 2 KB of gate hand-off per CTA
    # for at most 160 CTAs, then the two halves' group sums 8*M*E and the
    # gate's 8*M
    fixed = 16384 + 160 * 128 * 1024 + 160 * 2048
    assert lib.bi_router_workspace_bytes(1024, 256) == fixed + 8 * 1024 * 256 + 8 * 1024
    assert lib.bi_router_workspace_bytes(4096, 256) == fixed + 8 * 4096 * 256 + 8 * 4096
    assert lib.bi_router_workspace_bytes(8192, 512) == fixed + 8 * 8192 * 512 + 8 * 8192
    assert lib.bi_router_workspace_bytes(64, 1024) == 64 * 1024 * 64
    assert lib.bi_router_workspace_bytes(1 << 20, 256) == 16 << 20     # past 64 MiB: the tail plan only


@pytest.mark.parametrize("M,E", [(129, 256), (4096, 256), (64, 1024)])
def test_router_rejects_a_small_workspace(lib, M, E):
    """A workspace below bi_router_workspace_bytes is refused on the host,
    before any CUDA call (so this runs without a GPU)."""
    need = lib.bi_router_workspace_bytes(M, E)
    assert need > 0
    assert _router(lib, M=M, E=E, k=8, ws=0x100000, wsb=need - 1) == 1
    assert _router(lib, M=M, E=E, k=8, ws=None, wsb=need) == 1
    assert _router(lib, M=M, E=E, k=8, ws=0x100008, wsb=need) == 3          # not 16-byte aligned
    assert _router_gate(lib, M=M, E=E, k=8, ws=0x100000, wsb=need - 1) == 1


def _router_gate(lib, wsg=FAKE, dot=FAKE, sig=None, **kw):
    a = dict(x=FAKE, w=FAKE, ind=0, ld=0, M=4, H=256, E=64, k=4, logits=FAKE, ids=FAKE, ws=None, wsb=0)
    a.update(kw)
    return lib.bi_router_gate_topk(a["x"], a["w"], wsg, a["ind"], a["ld"], a["M"], a["H"], a["E"], a["k"],
                                   a["logits"], a["ids"], None, None, None, dot, sig, a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(wsg=None), 1), (dict(dot=None), 1), (dict(M=-1), 1), (dict(k=64), 1), (dict(H=260), 2),
    (dict(wsg=MIS), 3), (dict(dot=FAKE + 2), 3), (dict(sig=FAKE + 1), 3), (dict(x=MIS), 3),
])
def test_router_gate_validation(lib, kw, want):
    assert _router_gate(lib, **kw) == want


def test_router_gate_m0_is_noop(lib):
    assert _router_gate(lib, M=0, x=None, w=None, logits=None, ids=None, wsg=None, dot=None) == 0


@pytest.mark.parametrize("args,want", [
    ((FAKE, FAKE, -1, 256, FAKE, None), 1), ((FAKE, FAKE, 4, 0, FAKE, None), 1),
    ((FAKE, FAKE, 4, 12, FAKE, None), 2), ((None, FAKE, 4, 256, FAKE, None), 1),
    ((MIS, FAKE, 4, 256, FAKE, None), 3), ((FAKE, FAKE, 4, 256, None, None), 1),
    ((None, None, 0, 256, None, None), 0),
])
def test_gate_validation(lib, args, want):
    assert lib.bi_shared_gate(*args, None) == want


@pytest.mark.parametrize("args,want", [
    ((FAKE, FAKE, FAKE, -1, 256, 64, 64, 64, 256), 1),
    ((FAKE, FAKE, FAKE, 4, 256, 96, 96, 96, 256), 2),      # K % 64
    ((FAKE, FAKE, FAKE, 4, 250, 64, 64, 64, 250), 2),      # N % 16
    ((FAKE, FAKE, FAKE, 4, 256, 64, 32, 64, 256), 1),      # lda < K
    ((FAKE, FAKE, FAKE, 4, 256, 64, 68, 64, 256), 3),      # lda % 8
    ((MIS, FAKE, FAKE, 4, 256, 64, 64, 64, 256), 3),
    ((None, FAKE, FAKE, 4, 256, 64, 64, 64, 256), 1),
    ((None, None, None, 0, 256, 64, 64, 64, 256), 0),
])
def test_gemm_validation(lib, args, want):
    assert lib.bi_gemm_bf16(*args, None) == want


def _offs(v):
    arr = (C.c_int32 * len(v))(*v)
    return C.cast(arr, C.c_void_p), arr


@pytest.mark.parametrize("offs,M,k,n,want", [
    ([0, 3, 2], 5, 4, 2, 1),      # decreasing
    ([0, 6], 5, 4, 1, 1),         # past M
    ([0, 5], 5, 0, 1, 1),         # k = 0
    ([0, 5], 5, 33, 1, 2),        # k > max
    ([0, 5], 5, 4, 0, 1),         # no ranges
])
def test_hash_validation(lib, offs, M, k, n, want):
    p, keep = _offs(offs)
    assert lib.bi_route_trace_hash(FAKE, M, k, p, n, None, FAKE, None) == want


def test_hash_too_many_ranges(lib):
    p, keep = _offs([0] * 300)
    assert lib.bi_route_trace_hash(FAKE, 5, 4, p, 299, None, FAKE, None) == 2


def test_selftest_validation(lib):
    assert lib.bi_selftest_wait_timeout(0, None) == 1
    assert lib.bi_selftest_wait_timeout(2000001, None) == 1
    import ctypes as C
    f = C.c_double()
    assert lib.bi_selftest_fma_rate(0, 0, FAKE, None, C.byref(f)) == 1
    assert lib.bi_selftest_fma_rate((1 << 20) + 1, 0, FAKE, None, C.byref(f)) == 1
    assert lib.bi_selftest_fma_rate(10, 2, FAKE, None, C.byref(f)) == 1
    assert lib.bi_selftest_fma_rate(10, 0, None, None, C.byref(f)) == 1
    assert lib.bi_selftest_fma_rate(10, 1, FAKE, None, None) == 1


def _moe(lib, **kw):
    a = dict(X=FAKE, ids=FAKE, w=FAKE, W=FAKE, M=16, k=2, E=8, N=256, K=128, Y=FAKE, out=FAKE,
             ws=0x100000, wsb=1 << 40)
    a.update(kw)
    return lib.bi_moe_expert_gemm(a["X"], a["ids"], a["w"], a["W"], a["M"], a["k"], a["E"], a["N"], a["K"],
                                  a["Y"], a["out"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(M=-1), 1), (dict(k=0), 1), (dict(E=0), 1), (dict(N=0), 1), (dict(K=0), 1),
    (dict(K=100), 2), (dict(N=250), 2), (dict(E=2048), 2), (dict(k=33), 2),
    (dict(X=None), 1), (dict(ids=None), 1), (dict(W=None), 1), (dict(ws=None), 1),
    (dict(Y=None, out=None), 1), (dict(w=None), 1), (dict(wsb=1024), 1),
    (dict(X=MIS), 3), (dict(W=MIS), 3), (dict(ws=0x100010), 3), (dict(Y=FAKE + 2), 3),
])
def test_moe_validation(lib, kw, want):
    assert _moe(lib, **kw) == want


def test_moe_m0_is_noop_and_workspace_size(lib):
    assert _moe(lib, M=0, X=None, ids=None, W=None, ws=None) == 0
    n = lib.bi_moe_workspace_bytes(4096, 8, 256, 1024, 2048)
    cap = ((4096 * 8 + 256 * 127) + 127) // 128 * 128
    assert n >= cap * 2048 * 2 + 4096 * 8 * 1024 * 2          # gathered rows + per-slot outputs
    assert lib.bi_moe_workspace_bytes(-1, 8, 256, 1024, 2048) == 0


@pytest.mark.parametrize("args,want", [
    ((FAKE, FAKE, 0, -1, 256, 1e-6, FAKE, None), 1), ((FAKE, FAKE, 0, 4, 0, 1e-6, FAKE, None), 1),
    ((FAKE, FAKE, 3, 4, 256, 1e-6, FAKE, None), 1), ((FAKE, FAKE, 0, 4, 256, -1.0, FAKE, None), 1),
    ((FAKE, FAKE, 0, 4, 256, float("nan"), FAKE, None), 1), ((FAKE, FAKE, 0, 4, 12, 1e-6, FAKE, None), 2),
    ((None, FAKE, 0, 4, 256, 1e-6, FAKE, None), 1), ((FAKE, FAKE, 0, 4, 256, 1e-6, None, None), 1),
    ((MIS, FAKE, 0, 4, 256, 1e-6, FAKE, None), 3), ((FAKE, FAKE, 0, 4, 256, 1e-6, FAKE, FAKE + 2), 3),
    ((None, None, 0, 0, 256, 1e-6, None, None), 0),
])
def test_rmsnorm_validation(lib, args, want):
    x, w, dt, M, H, eps, y, r = args
    assert lib.bi_rmsnorm(x, w, dt, M, H, C.c_float(eps), y, r, None) == want


def test_router_plan_validation(lib):
    x = C.c_int32()
    assert lib.bi_router_plan(-1, 256, C.byref(x), C.byref(x), C.byref(x)) == 1
    assert lib.bi_router_plan(16, 0, C.byref(x), C.byref(x), C.byref(x)) == 1
    assert lib.bi_router_plan(16, 256, None, C.byref(x), C.byref(x)) == 1


def _attn(lib, q=FAKE, k=FAKE, v=FAKE, qo=(0, 4), ko=(0, 9), nh=4, nkv=2, D=128, scale=0.088, o=FAKE,
          lse=None, ws=None, wsb=0):
    n = len(qo) - 1
    qa = (C.c_int32 * len(qo))(*qo) if qo is not None else None
    ka = (C.c_int32 * len(ko))(*ko) if ko is not None else None
    return lib.bi_attention_prefill(q, k, v, n, qa, ka, nh, nkv, D, C.c_float(scale), o, lse, ws, wsb, None)


@pytest.mark.parametrize("kw,want", [
    (dict(nh=0), 1), (dict(nkv=0), 1), (dict(nh=6, nkv=4), 1), (dict(scale=0.0), 1), (dict(scale=-1.0), 1),
    (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1), (dict(D=64), 2), (dict(D=256), 2),
    (dict(nh=512, nkv=2), 2), (dict(qo=(1, 4), ko=(1, 9)), 1), (dict(qo=(0, 10), ko=(0, 9)), 1),
    (dict(qo=(0, 4, 2), ko=(0, 9, 12)), 1), (dict(qo=(0, 4, 6), ko=(0, 9, 8)), 1),
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(o=None), 1),
    (dict(q=MIS), 3), (dict(k=MIS), 3), (dict(v=MIS), 3), (dict(o=MIS), 3), (dict(lse=FAKE + 2), 3),
])
def test_attention_validation(lib, kw, want):
    assert _attn(lib, **kw) == want


def test_attention_empty_calls_are_noops(lib):
    """No requests, or requests without queries: BI_OK before any CUDA call."""
    assert _attn(lib, q=None, k=None, v=None, o=None, qo=(0,), ko=(0,)) == 0
    assert _attn(lib, q=None, k=None, v=None, o=None, qo=(0, 0, 0), ko=(0, 5, 7)) == 0
    assert lib.bi_attention_prefill(None, None, None, 1, None, None, 4, 2, 128, C.c_float(0.1), None, None,
                                    None, 0, None) == 1


def _wsb(lib, qo, ko, nh):
    return lib.bi_attention_workspace_bytes(len(qo) - 1, (C.c_int32 * len(qo))(*qo), (C.c_int32 * len(ko))(*ko), nh)


def test_attention_workspace_bytes(lib):
    """Contexts within 8192 keys need none; past it, one partial slot per
    8192-key chunk of each query tile that reaches beyond, of 128 rows x
    132 floats per head."""
    slot = 128 * 132 * 4
    cnt = lambda splits, nh: 0
    assert _wsb(lib, (0, 4096), (0, 4096), 16) == 0
    assert _wsb(lib, (0, 128), (0, 8192), 16) == 0                    # positions 8064..8191: one chunk
    assert _wsb(lib, (0, 128), (0, 8193), 16) == 2 * 16 * slot + cnt(1, 16)   # position 8192 opens chunk 1
    assert _wsb(lib, (0, 128, 256), (0, 32896, 65792), 4) == (5 + 5) * 4 * slot + cnt(2, 4)   # 257 blocks each
    assert _wsb(lib, (0, 128, 256), (0, 32896, 33024), 4) == 5 * 4 * slot + cnt(1, 4)         # the second fits
    assert _wsb(lib, (0, 4), (0, 3), 4) == 0                           # invalid offsets: 0
    assert _wsb(lib, (1, 4), (1, 9), 4) == 0


def test_attention_rejects_a_small_workspace(lib):
    qo, ko = (0, 128), (0, 20000)
    n = _wsb(lib, qo, ko, 4)
    assert n > 0
    assert _attn(lib, qo=qo, ko=ko, ws=None, wsb=0) == 1
    assert _attn(lib, qo=qo, ko=ko, ws=FAKE, wsb=n - 1) == 1
    assert _attn(lib, qo=qo, ko=ko, ws=MIS, wsb=n) == 3
