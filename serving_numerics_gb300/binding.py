"""Thin ctypes binding of libbi.so (include/bi.h).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (PyTorch provides device memory
and streams); their data pointers are passed through unchanged.  If the
library has not been built, `load()` raises: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libbi.so")

BI_OK, BI_ERR_INVALID_ARG, BI_ERR_UNSUPPORTED_SHAPE, BI_ERR_MISALIGNED, BI_ERR_CUDA, BI_ERR_TIMEOUT = range(6)
BI_F32, BI_BF16 = 0, 1
BI_MAX_E, BI_MAX_K, BI_MAX_H, BI_MAX_HASH_RANGES = 1024, 32, 32768, 256
BI_NOALLOC_SCRATCH_BYTES = 1 << 20
BI_ATTN_MAX_HEADS = 256
FNV64_BASIS = 0xCBF29CE484222325

# name -> (restype, argtypes), mirroring include/bi.h
_P, _I32, _I64 = C.c_void_p, C.c_int32, C.c_int64
SIGNATURES = {
    "bi_router_topk": (C.c_int, [_P, _P, C.c_int, C.c_int, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P,
                                 C.c_size_t, _P]),
    "bi_router_workspace_bytes": (C.c_size_t, [_I32, _I32]),
    "bi_router_topk_noalloc": (C.c_int, [_P, _P, C.c_int, C.c_int, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P]),
    "bi_shared_gate": (C.c_int, [_P, _P, _I32, _I32, _P, _P, _P]),
    "bi_router_gate_topk": (C.c_int, [_P, _P, _P, C.c_int, C.c_int, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P,
                                      _P, _P, _P, C.c_size_t, _P]),
    "bi_gemm_bf16": (C.c_int, [_P, _P, _P, _I32, _I32, _I32, _I64, _I64, _I64, _P]),
    "bi_route_trace_hash": (C.c_int, [_P, _I32, _I32, _P, _I32, _P, _P, _P]),
    "bi_status_string": (C.c_char_p, [C.c_int]),
    "bi_get_last_device_error": (C.c_int, []),
    "bi_abi_version": (C.c_int32, []),
    "bi_selftest_wait_timeout": (C.c_int, [C.c_uint32, _P]),
    "bi_selftest_fma_rate": (C.c_int, [_I32, _I32, _P, _P, _P]),
    "bi_selftest_dependent_floor": (C.c_int, [_P, _P, _P]),
    "bi_get_config": (C.c_int, [_P, C.c_size_t]),
    "bi_router_plan": (C.c_int, [_I32, _I32, _P, _P, _P]),
    "bi_rmsnorm": (C.c_int, [_P, _P, C.c_int, _I32, _I32, C.c_float, _P, _P, _P]),
    "bi_moe_workspace_bytes": (C.c_size_t, [_I32, _I32, _I32, _I32, _I32]),
    "bi_moe_expert_gemm": (C.c_int, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, C.c_size_t, _P]),
    "bi_prefix_split": (C.c_int, [_P, _I32, _I32, _P, _P]),
    "bi_attention_prefill": (C.c_int, [_P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, C.c_float, _P, _P, _P,
                                       C.c_size_t, _P]),
    "bi_attention_workspace_bytes": (C.c_size_t, [_I32, _P, _P, _I32]),
}

BI_TREE_PAIRWISE = 1


class BiConfig(C.Structure):
    """Mirror of bi_config (include/bi.h), field for field."""
    _fields_ = [(n, C.c_int32) for n in (
        "struct_size", "abi_version", "router_slab", "router_block", "router_partitions",
        "router_partition_order", "router_tree", "router_accum", "gemm_tile_m", "gemm_tile_n",
        "gemm_block_k", "gemm_mma_k", "gemm_accum", "gemm_split_k", "topk_tie_rule", "softmax_sum_order")]

_lib = None


class BiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load(path: str = LIB_PATH):
    """Load libbi.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(st: int) -> str:
    return load().bi_status_string(st).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str):
    if st != BI_OK:
        raise BiError(st, where)


# ------------------------------------------------------------- raw ABI calls
def _workspace(ws):
    """(pointer, bytes) of a router workspace given as None, a torch tensor
    (its whole storage) or a (pointer, bytes) pair."""
    if ws is None:
        return None, 0
    if isinstance(ws, tuple):
        return ws[0], int(ws[1])
    return ws.data_ptr(), ws.numel() * ws.element_size()


def bi_router_topk(x, w_gate, in_dtype, logit_dtype, M, H, E, k, logits_out, ids_out,
                   weights_out=None, margin_out=None, margin_ulps_out=None, workspace=None, stream=None,
                   check=True):
    wp, wn = _workspace(workspace)
    st = load().bi_router_topk(_ptr(x), _ptr(w_gate), in_dtype, logit_dtype, M, H, E, k,
                               _ptr(logits_out), _ptr(ids_out), _ptr(weights_out), _ptr(margin_out),
                               _ptr(margin_ulps_out), wp, wn, _stream(stream))
    if check:
        _check(st, "bi_router_topk")
    return st


def router_workspace_bytes(M: int, E: int) -> int:
    return int(load().bi_router_workspace_bytes(M, E))


def router_workspace(M: int, E: int, device="cuda"):
    """A caller-owned workspace for bi_router_topk / bi_router_gate_topk (a
    torch uint8 tensor of bi_router_workspace_bytes(M, E) bytes; None when
    none is needed).  torch's allocations are 256-byte aligned."""
    import torch
    n = router_workspace_bytes(M, E)
    return torch.empty(n, dtype=torch.uint8, device=device) if n > 0 else None


def bi_router_topk_noalloc(x, w_gate, in_dtype, logit_dtype, M, H, E, k, logits_out, ids_out,
                           weights_out=None, margin_out=None, margin_ulps_out=None, stream=None,
                           check=True):
    st = load().bi_router_topk_noalloc(_ptr(x), _ptr(w_gate), in_dtype, logit_dtype, M, H, E, k,
                                       _ptr(logits_out), _ptr(ids_out), _ptr(weights_out),
                                       _ptr(margin_out), _ptr(margin_ulps_out), _stream(stream))
    if check:
        _check(st, "bi_router_topk_noalloc")
    return st


def bi_router_gate_topk(x, w_gate, w_sg, in_dtype, logit_dtype, M, H, E, k, logits_out, ids_out,
                        weights_out=None, margin_out=None, margin_ulps_out=None, gate_dot_out=None,
                        gate_sigmoid_out=None, workspace=None, stream=None, check=True):
    wp, wn = _workspace(workspace)
    st = load().bi_router_gate_topk(_ptr(x), _ptr(w_gate), _ptr(w_sg), in_dtype, logit_dtype, M, H, E, k,
                                    _ptr(logits_out), _ptr(ids_out), _ptr(weights_out), _ptr(margin_out),
                                    _ptr(margin_ulps_out), _ptr(gate_dot_out), _ptr(gate_sigmoid_out),
                                    wp, wn, _stream(stream))
    if check:
        _check(st, "bi_router_gate_topk")
    return st


def bi_shared_gate(x, w_sg, M, H, dot_out, sigmoid_out=None, stream=None, check=True):
    st = load().bi_shared_gate(_ptr(x), _ptr(w_sg), M, H, _ptr(dot_out), _ptr(sigmoid_out), _stream(stream))
    if check:
        _check(st, "bi_shared_gate")
    return st


def bi_gemm_bf16(A, B, Cout, M, N, K, lda, ldb, ldc, stream=None, check=True):
    st = load().bi_gemm_bf16(_ptr(A), _ptr(B), _ptr(Cout), M, N, K, lda, ldb, ldc, _stream(stream))
    if check:
        _check(st, "bi_gemm_bf16")
    return st


def bi_route_trace_hash(ids, M, k, row_offsets, basis, hash_out, stream=None, check=True):
    """row_offsets: a host sequence of n_ranges + 1 ints."""
    n = len(row_offsets) - 1
    arr = (C.c_int32 * max(1, n + 1))(*[int(v) for v in row_offsets])
    st = load().bi_route_trace_hash(_ptr(ids), M, k, C.cast(arr, C.c_void_p), n, _ptr(basis),
                                    _ptr(hash_out), _stream(stream))
    if check:
        _check(st, "bi_route_trace_hash")
    return st


def bi_get_last_device_error() -> int:
    return load().bi_get_last_device_error()


def bi_abi_version() -> int:
    return load().bi_abi_version()


def bi_rmsnorm(x, w, dtype, M, H, eps, y_out, rstd_out=None, stream=None, check=True):
    st = load().bi_rmsnorm(_ptr(x), _ptr(w), dtype, M, H, C.c_float(eps), _ptr(y_out), _ptr(rstd_out),
                           _stream(stream))
    if check:
        _check(st, "bi_rmsnorm")
    return st


def rmsnorm(x, w, eps: float, stream=None):
    """Allocate outputs with torch and run bi_rmsnorm; x [M, H] and w [H]
    both float32 or both bfloat16.  Returns (y bf16 [M, H], rstd f32 [M])."""
    import torch
    M, H = x.shape
    y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    r = torch.empty((M,), dtype=torch.float32, device=x.device)
    bi_rmsnorm(x, w, BI_F32 if x.dtype == torch.float32 else BI_BF16, M, H, eps, y, r, stream=stream)
    return y, r


def bi_moe_expert_gemm(X, ids, weights, W, M, k, E, N, K, Y_out, out, workspace, workspace_bytes, stream=None,
                       check=True):
    st = load().bi_moe_expert_gemm(_ptr(X), _ptr(ids), _ptr(weights), _ptr(W), M, k, E, N, K, _ptr(Y_out),
                                   _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream))
    if check:
        _check(st, "bi_moe_expert_gemm")
    return st


def moe_workspace(M, k, E, N, K, device="cuda"):
    """A caller-owned workspace for bi_moe_expert_gemm (torch uint8 tensor)."""
    import torch
    n = int(load().bi_moe_workspace_bytes(M, k, E, N, K))
    return torch.empty(n + 256, dtype=torch.uint8, device=device), n


def moe_expert_gemm(X, ids, weights, W, stream=None, want_y=True, want_out=True, workspace=None):
    """Allocate outputs with torch and run bi_moe_expert_gemm.  X [M, K] and
    W [E, N, K] bf16, ids [M, k] int32, weights [M, k] f32 (or None when
    want_out is False).  Returns dict(Y, out)."""
    import torch
    M, K = X.shape
    E, N, _ = W.shape
    k = ids.shape[1]
    if workspace is None:
        workspace = moe_workspace(M, k, E, N, K, X.device)
    buf, n = workspace
    base = (buf.data_ptr() + 255) // 256 * 256           # 256-byte aligned start
    Y = torch.empty((M, k, N), dtype=torch.bfloat16, device=X.device) if want_y else None
    out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if want_out else None
    bi_moe_expert_gemm(X, ids, weights if want_out else None, W, M, k, E, N, K, Y, out, base, n, stream=stream)
    return {"Y": Y, "out": out}


def _host_i32(a):
    """A ctypes int32 array holding the values of a host sequence."""
    vals = [int(v) for v in a]
    return (C.c_int32 * max(len(vals), 1))(*vals)


def bi_attention_prefill(q, k, v, n_req, q_offsets, kv_offsets, n_heads, n_kv_heads, head_dim, scale, o_out,
                         lse_out=None, workspace=None, stream=None, check=True):
    """q_offsets and kv_offsets are host sequences of n_req + 1 ints;
    workspace a torch tensor (its whole storage), a (pointer, bytes) pair or
    None (enough when no context runs past 8192 keys)."""
    wp, wn = _workspace(workspace)
    st = load().bi_attention_prefill(_ptr(q), _ptr(k), _ptr(v), n_req, _host_i32(q_offsets),
                                     _host_i32(kv_offsets), n_heads, n_kv_heads, head_dim, C.c_float(scale),
                                     _ptr(o_out), _ptr(lse_out), wp, wn, _stream(stream))
    if check:
        _check(st, "bi_attention_prefill")
    return st


def attention_workspace_bytes(q_offsets, kv_offsets, n_heads: int) -> int:
    return int(load().bi_attention_workspace_bytes(len(q_offsets) - 1, _host_i32(q_offsets), _host_i32(kv_offsets),
                                                   n_heads))


def attention_workspace(q_offsets, kv_offsets, n_heads: int, device="cuda"):
    """A caller-owned workspace for bi_attention_prefill (torch uint8 tensor,
    or None when the call needs none)."""
    import torch
    n = attention_workspace_bytes(q_offsets, kv_offsets, n_heads)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def attention_prefill(q, k, v, q_offsets, kv_offsets, scale: float, stream=None, want_lse=True, workspace=None):
    """Allocate outputs (and the workspace, unless given) with torch and run
    bi_attention_prefill.  q [Tq, n_heads, 128], k and v [Tkv, n_kv_heads,
    128], all bfloat16; offsets host sequences (0, running sums).  Returns
    (o bf16 [Tq, n_heads, 128], lse f32 [Tq, n_heads] or None)."""
    import torch
    Tq, nh, D = q.shape
    nkv = k.shape[1]
    o = torch.empty((Tq, nh, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((Tq, nh), dtype=torch.float32, device=q.device) if want_lse else None
    if workspace is None:
        workspace = attention_workspace(q_offsets, kv_offsets, nh, q.device)
    bi_attention_prefill(q, k, v, len(q_offsets) - 1, q_offsets, kv_offsets, nh, nkv, D, scale, o, lse,
                         workspace=workspace, stream=stream)
    return o, lse


def selftest_fma_rate(iters: int, sink, packed: bool = False, stream=None) -> float:
    """Launch the FP32 FMA rate probe; returns the FLOPs it performs."""
    f = C.c_double()
    _check(load().bi_selftest_fma_rate(iters, int(packed), _ptr(sink), _stream(stream), C.byref(f)),
           "bi_selftest_fma_rate")
    return f.value


def router_plan(M: int, E: int):
    """bi_router_plan: (m_split, C, launches) for M rows and E experts; C < 0
    means the one-launch cluster router with -C blocks per cluster, m_split <
    0 the persistent projection with -m_split CTAs."""
    ms, c, n = C.c_int32(), C.c_int32(), C.c_int32()
    _check(load().bi_router_plan(M, E, C.byref(ms), C.byref(c), C.byref(n)), "bi_router_plan")
    return ms.value, c.value, n.value


def get_config() -> dict:
    """bi_get_config as a dict of the contract's fields."""
    c = BiConfig()
    _check(load().bi_get_config(C.byref(c), C.sizeof(c)), "bi_get_config")
    return {name: getattr(c, name) for name, _ in BiConfig._fields_}


def prefix_split(lengths, block: int):
    """bi_prefix_split: (cached[n], suffix_offsets[n + 1]) as int lists."""
    n = len(lengths)
    arr = (C.c_int32 * max(n, 1))(*[int(v) for v in lengths])
    cached = (C.c_int32 * max(n, 1))()
    offs = (C.c_int32 * (n + 1))()
    _check(load().bi_prefix_split(arr, n, int(block), cached, offs), "bi_prefix_split")
    return list(cached)[:n], list(offs)


def selftest_dependent_floor(inp, out, stream=None):
    """One launch of the dependent-cluster floor probe (in, out: >= 16 floats)."""
    _check(load().bi_selftest_dependent_floor(_ptr(inp), _ptr(out), _stream(stream)),
           "bi_selftest_dependent_floor")


def bi_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    return load().bi_selftest_wait_timeout(limit_us, _stream(stream))


# ------------------------------------------------------------- tensor helpers
def router_topk(x, w_gate, k: int, logit_dtype: str = "f32", stream=None, out=None, workspace=None):
    """Allocate the outputs (and, for batches that need one, a workspace)
    with torch and run bi_router_topk.

    x [M,H], w_gate [E,H]: both float32 or both bfloat16 CUDA tensors.
    Returns dict(logits, ids, weights, margin, margin_ulps)."""
    import torch
    M, H = x.shape
    E = w_gate.shape[0]
    ind = BI_F32 if x.dtype == torch.float32 else BI_BF16
    ld = BI_F32 if logit_dtype == "f32" else BI_BF16
    if out is None:
        dev = x.device
        out = {
            "logits": torch.empty((M, E), dtype=torch.float32 if ld == BI_F32 else torch.bfloat16, device=dev),
            "ids": torch.empty((M, k), dtype=torch.int32, device=dev),
            "weights": torch.empty((M, k), dtype=torch.float32, device=dev),
            "margin": torch.empty((M,), dtype=torch.float32, device=dev),
            "margin_ulps": torch.empty((M,), dtype=torch.int32, device=dev),
        }
    if workspace is None:
        workspace = router_workspace(M, E, x.device)
    bi_router_topk(x, w_gate, ind, ld, M, H, E, k, out["logits"], out["ids"], out.get("weights"),
                   out.get("margin"), out.get("margin_ulps"), workspace=workspace, stream=stream)
    return out


def router_gate_topk(x, w_gate, w_sg, k: int, logit_dtype: str = "f32", stream=None, workspace=None):
    """Allocate the outputs (and a workspace where needed) with torch and run
    bi_router_gate_topk.  Returns the router_topk dict plus gate_dot and
    gate_sigmoid."""
    import torch
    M, H = x.shape
    E = w_gate.shape[0]
    ind = BI_F32 if x.dtype == torch.float32 else BI_BF16
    ld = BI_F32 if logit_dtype == "f32" else BI_BF16
    dev = x.device
    out = {
        "logits": torch.empty((M, E), dtype=torch.float32 if ld == BI_F32 else torch.bfloat16, device=dev),
        "ids": torch.empty((M, k), dtype=torch.int32, device=dev),
        "weights": torch.empty((M, k), dtype=torch.float32, device=dev),
        "margin": torch.empty((M,), dtype=torch.float32, device=dev),
        "margin_ulps": torch.empty((M,), dtype=torch.int32, device=dev),
        "gate_dot": torch.empty((M,), dtype=torch.float32, device=dev),
        "gate_sigmoid": torch.empty((M,), dtype=torch.float32, device=dev),
    }
    if workspace is None:
        workspace = router_workspace(M, E, dev)
    bi_router_gate_topk(x, w_gate, w_sg, ind, ld, M, H, E, k, out["logits"], out["ids"], out["weights"],
                        out["margin"], out["margin_ulps"], out["gate_dot"], out["gate_sigmoid"],
                        workspace=workspace, stream=stream)
    return out


def shared_gate(x, w_sg, stream=None):
    import torch
    M, H = x.shape
    dot = torch.empty((M,), dtype=torch.float32, device=x.device)
    sig = torch.empty((M,), dtype=torch.float32, device=x.device)
    bi_shared_gate(x, w_sg, M, H, dot, sig, stream=stream)
    return dot, sig


def gemm_bf16(A, B, stream=None, out=None):
    import torch
    M, K = A.shape
    N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    bi_gemm_bf16(A, B, out, M, N, K, A.stride(0), B.stride(0), out.stride(0), stream=stream)
    return out


def route_hash(ids, row_offsets, basis=None, stream=None):
    """Per-range FNV-1a hashes (torch int64 tensor viewed as uint64 bits)."""
    import torch
    M, k = ids.shape
    n = len(row_offsets) - 1
    out = torch.empty((n,), dtype=torch.int64, device=ids.device)
    bi_route_trace_hash(ids, M, k, row_offsets, basis, out, stream=stream)
    return out
