"""Thin ctypes binding of the libddt.so C ABI (include/ddt.h).

Every function here only checks shapes/dtypes of torch CUDA tensors and passes their
device pointers, sizes and the current CUDA stream to the C entry point of the same
name; all of the round's arithmetic runs in the library's CUDA kernels.  There is no
CPU fallback: without the built library (or without a GPU) every call raises.

Outputs are allocated with torch (PyTorch is the device-memory and stream provider);
callers that manage memory themselves can pass `out=` dicts of preallocated tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build_ext

F32, BF16 = 0, 1
_DT = {torch.float32: F32, torch.bfloat16: BF16}
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "capacity", 4: "cuda", 5: "timeout",
          6: "non-finite", 7: "malformed tree"}

_lib = None
_lock = threading.Lock()

_c_int, _c_size, _c_p, _c_float = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float

_SIGS = {
    "ddt_status_string": ([_c_int], ctypes.c_char_p),
    "ddt_version": ([], ctypes.c_char_p),
    "ddt_launch_count": ([], ctypes.c_uint64),
    "ddt_wait_selftest": ([_c_p, _c_p], _c_int),
    "ddt_build_tree_workspace": ([_c_int] * 4, _c_size),
    "ddt_build_tree": ([_c_int] * 6 + [_c_p] * 11 + [_c_p, _c_size, _c_p], _c_int),
    "ddt_build_tree_noalloc": ([_c_int] * 6 + [_c_p] * 11 + [_c_p], _c_int),
    "ddt_tree_attn_workspace": ([_c_int] * 7, _c_size),
    "ddt_tree_attn": ([_c_int] * 9 + [_c_p] * 8 + [_c_float, _c_p, _c_p, _c_p, _c_size, _c_p], _c_int),
    "ddt_tree_gdn_workspace": ([_c_int] * 7, _c_size),
    "ddt_tree_gdn": ([_c_int] * 10 + [_c_p] * 11 + [_c_p, _c_size, _c_p], _c_int),
    "ddt_walk_accept_workspace": ([_c_int] * 3, _c_size),
    "ddt_walk_accept": ([_c_int] * 5 + [_c_p] * 11 + [_c_p, _c_size, _c_p], _c_int),
    "ddt_walk_accept_flat": ([_c_int] * 5 + [_c_p] * 11 + [_c_p, _c_size, _c_p], _c_int),
    "ddt_walk_accept_sample_workspace": ([_c_int] * 3, _c_size),
    "ddt_walk_accept_sample": ([_c_int] * 5 + [_c_float, _c_int] + [_c_p] * 11 + [_c_p, _c_size, _c_p], _c_int),
    "ddt_tree_attn_paged_workspace": ([_c_int] * 8, _c_size),
    "ddt_tree_attn_paged": ([_c_int] * 11 + [_c_p] * 9 + [_c_float, _c_p, _c_p, _c_p, _c_size, _c_p], _c_int),
    "ddt_commit_paged": ([_c_int] * 9 + [_c_p] + [_c_int] + [_c_p] * 4 + [_c_int] * 6 + [_c_int] + [_c_p] * 13,
                         _c_int),
    "ddt_rope_tree": ([_c_int] * 7 + [ctypes.c_double, _c_int] + [_c_p] * 5, _c_int),
    "ddt_tree_attn_rope": ([_c_int] * 9 + [_c_p] * 9 + [_c_int, ctypes.c_double, _c_float, _c_p, _c_p, _c_p, _c_size,
                                                     _c_p], _c_int),
    "ddt_tree_attn_paged_rope": ([_c_int] * 11 + [_c_p] * 10 + [_c_int, ctypes.c_double, _c_float, _c_p, _c_p, _c_p,
                                                                _c_size, _c_p], _c_int),
    "ddt_commit": ([_c_int] * 7 + [_c_int] + [_c_p] * 4 + [_c_int] * 6 + [_c_int] + [_c_p] * 13, _c_int),
}
EXPORTS = tuple(_SIGS)


class DDTError(RuntimeError):
    pass


def lib_path() -> str:
    return build_ext.LIB


def load(build_if_missing: bool = True):
    """Load libddt.so (building it first if it is missing or stale and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = build_ext.LIB
        if build_if_missing and build_ext.is_stale():
            build_ext.build()
        if not os.path.exists(path):
            raise DDTError(f"CUDA library not built: {path} (run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def ddt_launch_count() -> int:
    """Kernel launches the library has issued in this process so far."""
    return int(load().ddt_launch_count())


def ddt_wait_selftest(stream=None) -> int:
    """Runs one bounded device wait that nothing signals and returns the status it wrote
    (DDT_ERR_TIMEOUT = 5 when the wait gave up, as it should); synchronises the stream."""
    lib = _gpu()
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    s = stream or torch.cuda.current_stream()
    _check(lib.ddt_wait_selftest(_ptr(st), ctypes.c_void_p(s.cuda_stream)), "ddt_wait_selftest")
    s.synchronize()
    return int(st.item())


def _gpu():
    if not torch.cuda.is_available():
        raise DDTError("no CUDA device: the DDTree round library runs only on the GPU")
    return load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(rc, what):
    if rc != 0:
        raise DDTError(f"{what}: {STATUS.get(rc, rc)}")


def _need(t, shape, dtype, name):
    if t is None:
        raise DDTError(f"{name} is required")
    if not t.is_cuda or not t.is_contiguous():
        raise DDTError(f"{name} must be a contiguous CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise DDTError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise DDTError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return t


def _ws(nbytes, dev):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=dev)


# --------------------------------------------------------------------------- build
def ddt_build_tree(draft_logits, root_token, prefix_len, top_k: int, budget: int, *, want_score=True,
                   out=None, workspace=None):
    """Best-first draft tree.  draft_logits [B][D][V] (fp32/bf16)."""
    lib = _gpu()
    B, D, V = draft_logits.shape
    dev = draft_logits.device
    _need(draft_logits, (B, D, V), None, "draft_logits")
    _need(root_token, (B,), torch.int32, "root_token")
    _need(prefix_len, (B,), torch.int32, "prefix_len")
    N = budget + 1
    W = (N + 31) // 32
    o = out or {}
    i32 = dict(dtype=torch.int32, device=dev)
    res = {
        "token": o.get("token", torch.empty((B, N), **i32)),
        "parent": o.get("parent", torch.empty((B, N), **i32)),
        "depth": o.get("depth", torch.empty((B, N), **i32)),
        "position": o.get("position", torch.empty((B, N), **i32)),
        "n_nodes": o.get("n_nodes", torch.empty((B,), **i32)),
        "anc": o.get("anc", torch.empty((B, N, W), dtype=torch.int32, device=dev)),
        "score": o.get("score", torch.empty((B, N), dtype=torch.float64, device=dev)) if want_score else None,
        "status": o.get("status", torch.empty((B,), **i32)),
    }
    need = lib.ddt_build_tree_workspace(B, D, V, top_k)
    ws = workspace if workspace is not None else _ws(need, dev)
    rc = lib.ddt_build_tree(B, D, V, int(top_k), int(budget), _DT[draft_logits.dtype], _ptr(draft_logits),
                            _ptr(root_token), _ptr(prefix_len), _ptr(res["token"]), _ptr(res["parent"]),
                            _ptr(res["depth"]), _ptr(res["position"]), _ptr(res["n_nodes"]), _ptr(res["anc"]),
                            _ptr(res["score"]), _ptr(res["status"]), _ptr(ws), ws.numel(), _stream())
    _check(rc, "ddt_build_tree")
    return res


def ddt_build_tree_noalloc(draft_logits, root_token, prefix_len, top_k: int, budget: int, *, out):
    """ddt_build_tree for callers that cannot allocate device memory: the scratch is the
    library's fixed 4 MiB device array, so `out` must hold every preallocated output
    (token, parent, depth, position, n_nodes, anc, score or None, status).  Calls whose
    kernels overlap on the GPU share that array and must be ordered by the caller."""
    lib = _gpu()
    B, D, V = draft_logits.shape
    _need(draft_logits, (B, D, V), None, "draft_logits")
    _need(root_token, (B,), torch.int32, "root_token")
    _need(prefix_len, (B,), torch.int32, "prefix_len")
    N = budget + 1
    for name, shape in (("token", (B, N)), ("parent", (B, N)), ("depth", (B, N)), ("position", (B, N)),
                        ("n_nodes", (B,)), ("anc", (B, N, (N + 31) // 32)), ("status", (B,))):
        _need(out.get(name), shape, None, name)
    if out.get("score") is not None:
        _need(out["score"], (B, N), torch.float64, "score")
    rc = lib.ddt_build_tree_noalloc(B, D, V, int(top_k), int(budget), _DT[draft_logits.dtype], _ptr(draft_logits),
                                    _ptr(root_token), _ptr(prefix_len), _ptr(out["token"]), _ptr(out["parent"]),
                                    _ptr(out["depth"]), _ptr(out["position"]), _ptr(out["n_nodes"]),
                                    _ptr(out["anc"]), _ptr(out.get("score")), _ptr(out["status"]), _stream())
    _check(rc, "ddt_build_tree_noalloc")
    return out


# ----------------------------------------------------------------------- attention
def ddt_tree_attn(q, k_tree, v_tree, k_cache, v_cache, prefix_len, n_nodes, anc, *, scale: float,
                  out_dtype=None, out=None, status=None, workspace=None):
    """q [L][B][N][Hq][d]; k/v_tree [L][B][N][Hkv][d]; k/v_cache [L][B][Hkv][Pcap][d];
    scale: the softmax scale, passed through as given (1/sqrt(d) for standard attention)."""
    lib = _gpu()
    L, B, N, Hq, d = q.shape
    Hkv = k_tree.shape[3]
    Pcap = k_cache.shape[3]
    dt = q.dtype
    _need(q, (L, B, N, Hq, d), dt, "q")
    _need(k_tree, (L, B, N, Hkv, d), dt, "k_tree")
    _need(v_tree, (L, B, N, Hkv, d), dt, "v_tree")
    _need(k_cache, (L, B, Hkv, Pcap, d), dt, "k_cache")
    _need(v_cache, (L, B, Hkv, Pcap, d), dt, "v_cache")
    _need(prefix_len, (B,), torch.int32, "prefix_len")
    _need(n_nodes, (B,), torch.int32, "n_nodes")
    _need(anc, (B, N, (N + 31) // 32), None, "anc")
    out_dtype = out_dtype or dt
    o = out if out is not None else torch.empty((L, B, N, Hq, d), dtype=out_dtype, device=q.device)
    _need(o, (L, B, N, Hq, d), out_dtype, "o")
    st = status if status is not None else torch.empty((B,), dtype=torch.int32, device=q.device)
    scale = float(scale)
    need = lib.ddt_tree_attn_workspace(L, B, N, Hq, Hkv, d, Pcap)
    ws = workspace if workspace is not None else _ws(need, q.device)
    rc = lib.ddt_tree_attn(L, B, N, Hq, Hkv, d, Pcap, _DT[dt], _DT[out_dtype], _ptr(q), _ptr(k_tree), _ptr(v_tree),
                           _ptr(k_cache), _ptr(v_cache), _ptr(prefix_len), _ptr(n_nodes), _ptr(anc), scale, _ptr(o),
                           _ptr(st), _ptr(ws), ws.numel(), _stream())
    _check(rc, "ddt_tree_attn")
    return {"o": o, "status": st}


def ddt_tree_attn_paged(q, k_tree, v_tree, k_pages, v_pages, block_table, prefix_len, n_nodes, anc, *,
                        scale: float, out_dtype=None, out=None, status=None, workspace=None):
    """q [L][B][N][Hq][d]; k/v_tree [L][B][N][Hkv][d]; k/v_pages [L][num_pages][Hkv][page_size][d] (bf16);
    block_table [B][max_pages] int32; scale as in ddt_tree_attn."""
    lib = _gpu()
    L, B, N, Hq, d = q.shape
    Hkv = k_tree.shape[3]
    num_pages, page = k_pages.shape[1], k_pages.shape[3]
    max_pages = block_table.shape[1]
    dt = q.dtype
    _need(q, (L, B, N, Hq, d), dt, "q")
    _need(k_tree, (L, B, N, Hkv, d), dt, "k_tree")
    _need(v_tree, (L, B, N, Hkv, d), dt, "v_tree")
    _need(k_pages, (L, num_pages, Hkv, page, d), dt, "k_pages")
    _need(v_pages, (L, num_pages, Hkv, page, d), dt, "v_pages")
    _need(block_table, (B, max_pages), torch.int32, "block_table")
    _need(prefix_len, (B,), torch.int32, "prefix_len")
    _need(n_nodes, (B,), torch.int32, "n_nodes")
    _need(anc, (B, N, (N + 31) // 32), None, "anc")
    out_dtype = out_dtype or dt
    o = out if out is not None else torch.empty((L, B, N, Hq, d), dtype=out_dtype, device=q.device)
    _need(o, (L, B, N, Hq, d), out_dtype, "o")
    st = status if status is not None else torch.empty((B,), dtype=torch.int32, device=q.device)
    scale = float(scale)
    need = lib.ddt_tree_attn_paged_workspace(L, B, N, Hq, Hkv, d, page, max_pages)
    ws = workspace if workspace is not None else _ws(need, q.device)
    rc = lib.ddt_tree_attn_paged(L, B, N, Hq, Hkv, d, page, num_pages, max_pages, _DT[dt], _DT[out_dtype], _ptr(q),
                                 _ptr(k_tree), _ptr(v_tree), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                 _ptr(prefix_len), _ptr(n_nodes), _ptr(anc), scale, _ptr(o), _ptr(st), _ptr(ws),
                                 ws.numel(), _stream())
    _check(rc, "ddt_tree_attn_paged")
    return {"o": o, "status": st}


def ddt_rope_tree(q, k_tree, position, n_nodes, *, rot_dim=None, theta=10000.0, Hq=None):
    """In place: q [L][B][N][Hq][d], k_tree [L][B][N][Hkv][d] rotated at position [B][N].
    q may be None (keys only; then Hq is not needed)."""
    lib = _gpu()
    L, B, N, Hkv, d = k_tree.shape
    _need(k_tree, (L, B, N, Hkv, d), k_tree.dtype, "k_tree")
    if q is not None:
        Hq = q.shape[3]
        _need(q, (L, B, N, Hq, d), k_tree.dtype, "q")
    _need(position, (B, N), torch.int32, "position")
    _need(n_nodes, (B,), torch.int32, "n_nodes")
    rot = int(rot_dim or d)
    rc = lib.ddt_rope_tree(L, B, N, int(Hq or 1), Hkv, d, rot, float(theta), _DT[k_tree.dtype], _ptr(position),
                           _ptr(n_nodes), _ptr(q), _ptr(k_tree), _stream())
    _check(rc, "ddt_rope_tree")
    return q, k_tree


def rope_workspace_bytes(base_bytes, B, N, rot_dim):
    """Workspace of the rotary attention calls: the plain call's bytes rounded up to 256,
    then the per-row cos/sin table."""
    return ((int(base_bytes) + 255) // 256) * 256 + 4 * B * N * int(rot_dim)


def ddt_tree_attn_rope(q, k_tree, v_tree, k_cache, v_cache, prefix_len, n_nodes, anc, position, *, scale: float,
                       rot_dim=None, theta=10000.0, out_dtype=None, out=None, status=None, workspace=None):
    """ddt_tree_attn with q BEFORE rotary embedding (rotated inside the kernel at position [B][N])."""
    lib = _gpu()
    L, B, N, Hq, d = q.shape
    Hkv = k_tree.shape[3]
    Pcap = k_cache.shape[3]
    dt = q.dtype
    _need(q, (L, B, N, Hq, d), dt, "q")
    _need(k_tree, (L, B, N, Hkv, d), dt, "k_tree")
    _need(v_tree, (L, B, N, Hkv, d), dt, "v_tree")
    _need(k_cache, (L, B, Hkv, Pcap, d), dt, "k_cache")
    _need(v_cache, (L, B, Hkv, Pcap, d), dt, "v_cache")
    _need(prefix_len, (B,), torch.int32, "prefix_len")
    _need(n_nodes, (B,), torch.int32, "n_nodes")
    _need(anc, (B, N, (N + 31) // 32), None, "anc")
    _need(position, (B, N), torch.int32, "position")
    out_dtype = out_dtype or dt
    o = out if out is not None else torch.empty((L, B, N, Hq, d), dtype=out_dtype, device=q.device)
    _need(o, (L, B, N, Hq, d), out_dtype, "o")
    st = status if status is not None else torch.empty((B,), dtype=torch.int32, device=q.device)
    rot = int(rot_dim or d)
    need = rope_workspace_bytes(lib.ddt_tree_attn_workspace(L, B, N, Hq, Hkv, d, Pcap), B, N, rot)
    ws = workspace if workspace is not None else _ws(need, q.device)
    rc = lib.ddt_tree_attn_rope(L, B, N, Hq, Hkv, d, Pcap, _DT[dt], _DT[out_dtype], _ptr(q), _ptr(k_tree),
                                _ptr(v_tree), _ptr(k_cache), _ptr(v_cache), _ptr(prefix_len), _ptr(n_nodes), _ptr(anc),
                                _ptr(position), rot, float(theta), float(scale), _ptr(o), _ptr(st), _ptr(ws),
                                ws.numel(), _stream())
    _check(rc, "ddt_tree_attn_rope")
    return {"o": o, "status": st}


def ddt_tree_attn_paged_rope(q, k_tree, v_tree, k_pages, v_pages, block_table, prefix_len, n_nodes, anc, position, *,
                             scale: float, rot_dim=None, theta=10000.0, out_dtype=None, out=None, status=None,
                             workspace=None):
    """ddt_tree_attn_paged with q BEFORE rotary embedding (rotated inside the kernel)."""
    lib = _gpu()
    L, B, N, Hq, d = q.shape
    Hkv = k_tree.shape[3]
    num_pages, page = k_pages.shape[1], k_pages.shape[3]
    max_pages = block_table.shape[1]
    dt = q.dtype
    _need(q, (L, B, N, Hq, d), dt, "q")
    _need(k_tree, (L, B, N, Hkv, d), dt, "k_tree")
    _need(v_tree, (L, B, N, Hkv, d), dt, "v_tree")
    _need(k_pages, (L, num_pages, Hkv, page, d), dt, "k_pages")
    _need(v_pages, (L, num_pages, Hkv, page, d), dt, "v_pages")
    _need(block_table, (B, max_pages), torch.int32, "block_table")
    _need(prefix_len, (B,), torch.int32, "prefix_len")
    _need(n_nodes, (B,), torch.int32, "n_nodes")
    _need(anc, (B, N, (N + 31) // 32), None, "anc")
    _need(position, (B, N), torch.int32, "position")
    out_dtype = out_dtype or dt
    o = out if out is not None else torch.empty((L, B, N, Hq, d), dtype=out_dtype, device=q.device)
    _need(o, (L, B, N, Hq, d), out_dtype, "o")
    st = status if status is not None else torch.empty((B,), dtype=torch.int32, device=q.device)
    rot = int(rot_dim or d)
    need = rope_workspace_bytes(lib.ddt_tree_attn_paged_workspace(L, B, N, Hq, Hkv, d, page, max_pages), B, N, rot)
    ws = workspace if workspace is not None else _ws(need, q.device)
    rc = lib.ddt_tree_attn_paged_rope(L, B, N, Hq, Hkv, d, page, num_pages, max_pages, _DT[dt], _DT[out_dtype], _ptr(q),
                                      _ptr(k_tree), _ptr(v_tree), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                      _ptr(prefix_len), _ptr(n_nodes), _ptr(anc), _ptr(position), rot, float(theta),
                                      float(scale), _ptr(o), _ptr(st), _ptr(ws), ws.numel(), _stream())
    _check(rc, "ddt_tree_attn_paged_rope")
    return {"o": o, "status": st}


# ----------------------------------------------------------------------------- GDN
def ddt_tree_gdn(x, conv_w, conv_state, beta, decay, S, parent, n_nodes, *, Hk: int, out_dtype=None, out=None,
                 status=None, workspace=None, S_node_debug=None):
    """x [L][B][N][C]; conv_w [L][C][K]; conv_state [L][B][K-1][C]; beta/decay [L][B][N][Hv] fp32;
    S [L][B][Hv][dv][dk] fp32; parent [B][N]; n_nodes [B].  S_node_debug: optional
    [L][B][N][Hv][dv][dk] fp32 tensor that receives every node's own state (small trees)."""
    lib = _gpu()
    L, B, N, C = x.shape
    Hv, dv, dk = S.shape[2], S.shape[3], S.shape[4]
    K = conv_w.shape[2]
    dt = x.dtype
    _need(x, (L, B, N, C), dt, "x")
    if C != 2 * Hk * dk + Hv * dv:
        raise DDTError("x channels must be 2*Hk*dk + Hv*dv")
    _need(conv_w, (L, C, K), dt, "conv_w")
    _need(conv_state, (L, B, K - 1, C), dt, "conv_state")
    _need(beta, (L, B, N, Hv), torch.float32, "beta")
    _need(decay, (L, B, N, Hv), torch.float32, "decay")
    _need(S, (L, B, Hv, dv, dk), torch.float32, "S")
    _need(parent, (B, N), torch.int32, "parent")
    _need(n_nodes, (B,), torch.int32, "n_nodes")
    out_dtype = out_dtype or dt
    o = out if out is not None else torch.empty((L, B, N, Hv, dv), dtype=out_dtype, device=x.device)
    _need(o, (L, B, N, Hv, dv), out_dtype, "o")
    st = status if status is not None else torch.empty((B,), dtype=torch.int32, device=x.device)
    if S_node_debug is not None:
        _need(S_node_debug, (L, B, N, Hv, dv, dk), torch.float32, "S_node_debug")
    need = lib.ddt_tree_gdn_workspace(L, B, N, Hk, Hv, dk, dv)
    ws = workspace if workspace is not None else _ws(need, x.device)
    rc = lib.ddt_tree_gdn(L, B, N, Hk, Hv, dk, dv, K, _DT[dt], _DT[out_dtype], _ptr(x), _ptr(conv_w),
                          _ptr(conv_state), _ptr(beta), _ptr(decay), _ptr(S), _ptr(parent), _ptr(n_nodes), _ptr(o),
                          _ptr(S_node_debug), _ptr(st), _ptr(ws), ws.numel(), _stream())
    _check(rc, "ddt_tree_gdn")
    return {"o": o, "status": st}


# ---------------------------------------------------------------------------- walk
def ddt_walk_accept(token, parent, n_nodes, max_accept: int, *, target_logits=None, target_argmax=None, out=None,
                    workspace=None, flat=False):
    """Greedy walk.  target_logits [B][N][V] (or target_argmax [B][N] int32).  flat: the
    safe mode that only descends into first (rank-0) children (ddt_walk_accept_flat)."""
    lib = _gpu()
    B, N = token.shape
    dev = token.device
    _need(token, (B, N), torch.int32, "token")
    _need(parent, (B, N), torch.int32, "parent")
    _need(n_nodes, (B,), torch.int32, "n_nodes")
    A = max_accept + 1
    o = out or {}
    i32 = dict(dtype=torch.int32, device=dev)
    if target_logits is not None:
        V = target_logits.shape[2]
        _need(target_logits, (B, N, V), None, "target_logits")
        targ = o.get("target_argmax", torch.empty((B, N), **i32))
        dt = _DT[target_logits.dtype]
    else:
        V = 1
        targ = _need(target_argmax, (B, N), torch.int32, "target_argmax")
        dt = F32
    res = {"target_argmax": targ,
           "acc_nodes": o.get("acc_nodes", torch.empty((B, A), **i32)),
           "acc_len": o.get("acc_len", torch.empty((B,), **i32)),
           "bonus": o.get("bonus", torch.empty((B,), **i32)),
           "emitted": o.get("emitted", torch.empty((B, A), **i32)),
           "n_emitted": o.get("n_emitted", torch.empty((B,), **i32)),
           "status": o.get("status", torch.empty((B,), **i32))}
    need = lib.ddt_walk_accept_workspace(B, N, V)
    ws = workspace if workspace is not None else _ws(need, dev)
    fn = lib.ddt_walk_accept_flat if flat else lib.ddt_walk_accept
    rc = fn(B, N, V, int(max_accept), dt, _ptr(target_logits), _ptr(targ), _ptr(token),
            _ptr(parent), _ptr(n_nodes), _ptr(res["acc_nodes"]), _ptr(res["acc_len"]),
            _ptr(res["bonus"]), _ptr(res["emitted"]), _ptr(res["n_emitted"]), _ptr(res["status"]),
            _ptr(ws), ws.numel(), _stream())
    _check(rc, "ddt_walk_accept_flat" if flat else "ddt_walk_accept")
    return res


def ddt_walk_accept_sample(token, parent, n_nodes, max_accept: int, *, target_logits, uniforms, temperature: float,
                           out=None, workspace=None):
    """Tree-walk rejection sampling at `temperature`.  uniforms [B][max_accept + 1][C + 1]
    fp32 in [0, 1); C (the most children a node may have) is read from its last dimension."""
    lib = _gpu()
    B, N = token.shape
    dev = token.device
    _need(token, (B, N), torch.int32, "token")
    _need(parent, (B, N), torch.int32, "parent")
    _need(n_nodes, (B,), torch.int32, "n_nodes")
    A = max_accept + 1
    V = target_logits.shape[2]
    _need(target_logits, (B, N, V), None, "target_logits")
    C = uniforms.shape[-1] - 1
    _need(uniforms, (B, A, C + 1), torch.float32, "uniforms")
    o = out or {}
    i32 = dict(dtype=torch.int32, device=dev)
    res = {"acc_nodes": o.get("acc_nodes", torch.empty((B, A), **i32)),
           "acc_len": o.get("acc_len", torch.empty((B,), **i32)),
           "bonus": o.get("bonus", torch.empty((B,), **i32)),
           "emitted": o.get("emitted", torch.empty((B, A), **i32)),
           "n_emitted": o.get("n_emitted", torch.empty((B,), **i32)),
           "status": o.get("status", torch.empty((B,), **i32))}
    need = lib.ddt_walk_accept_sample_workspace(B, N, V)
    ws = workspace if workspace is not None else _ws(need, dev)
    rc = lib.ddt_walk_accept_sample(B, N, V, int(max_accept), int(C), float(temperature), _DT[target_logits.dtype],
                                    _ptr(target_logits), _ptr(uniforms), _ptr(token), _ptr(parent), _ptr(n_nodes),
                                    _ptr(res["acc_nodes"]), _ptr(res["acc_len"]), _ptr(res["bonus"]),
                                    _ptr(res["emitted"]), _ptr(res["n_emitted"]), _ptr(res["status"]), _ptr(ws),
                                    ws.numel(), _stream())
    _check(rc, "ddt_walk_accept_sample")
    return res


# -------------------------------------------------------------------------- commit
def ddt_commit(acc_nodes, acc_len, prefix_len, *, k_tree=None, v_tree=None, k_cache=None, v_cache=None, x=None,
               conv_w=None, beta=None, decay=None, S=None, conv_state=None, Hk: int = 1, out=None):
    """In-place commit of the accepted path into the caches / GDN state / conv state."""
    lib = _gpu()
    B, A = acc_nodes.shape
    dev = acc_nodes.device
    _need(acc_nodes, (B, A), torch.int32, "acc_nodes")
    _need(acc_len, (B,), torch.int32, "acc_len")
    _need(prefix_len, (B,), torch.int32, "prefix_len")
    N = None
    if k_cache is not None:
        La, _, N, Hkv, d = k_tree.shape
        Pcap = k_cache.shape[3]
        kdt = k_tree.dtype
        _need(k_tree, (La, B, N, Hkv, d), kdt, "k_tree")
        _need(v_tree, (La, B, N, Hkv, d), kdt, "v_tree")
        _need(k_cache, (La, B, Hkv, Pcap, d), kdt, "k_cache")
        _need(v_cache, (La, B, Hkv, Pcap, d), kdt, "v_cache")
        kvd = _DT[kdt]
    else:
        La, Hkv, d, Pcap, kvd = 0, 1, 1, 0, F32
    if S is not None:
        Lg, _, N2, C = x.shape
        N = N2 if N is None else N
        if N2 != N:
            raise DDTError("tree rows differ between the attention and GDN parts")
        Hv, dv, dk = S.shape[2], S.shape[3], S.shape[4]
        K = conv_w.shape[2]
        _need(x, (Lg, B, N, C), x.dtype, "x")
        _need(conv_w, (Lg, C, K), x.dtype, "conv_w")
        _need(conv_state, (Lg, B, K - 1, C), x.dtype, "conv_state")
        _need(beta, (Lg, B, N, Hv), torch.float32, "beta")
        _need(decay, (Lg, B, N, Hv), torch.float32, "decay")
        _need(S, (Lg, B, Hv, dv, dk), torch.float32, "S")
        xd = _DT[x.dtype]
    else:
        Lg, Hv, dk, dv, K, xd = 0, 1, 1, 1, 1, F32
    if N is None:
        raise DDTError("ddt_commit needs the attention part, the GDN part, or both")
    o = out or {}
    i32 = dict(dtype=torch.int32, device=dev)
    res = {"src_row": o.get("src_row", torch.empty((B, A), **i32)),
           "dst_pos": o.get("dst_pos", torch.empty((B, A), **i32)),
           "status": o.get("status", torch.empty((B,), **i32))}
    rc = lib.ddt_commit(B, N, A, La, Hkv, d, Pcap, kvd, _ptr(k_tree), _ptr(v_tree), _ptr(k_cache), _ptr(v_cache),
                        Lg, Hk, Hv, dk, dv, K, xd, _ptr(x), _ptr(conv_w), _ptr(beta), _ptr(decay), _ptr(S),
                        _ptr(conv_state), _ptr(acc_nodes), _ptr(acc_len), _ptr(prefix_len), _ptr(res["src_row"]),
                        _ptr(res["dst_pos"]), _ptr(res["status"]), _stream())
    _check(rc, "ddt_commit")
    return res


def ddt_commit_paged(acc_nodes, acc_len, prefix_len, block_table, *, k_tree, v_tree, k_pages, v_pages, x=None,
                     conv_w=None, beta=None, decay=None, S=None, conv_state=None, Hk: int = 1, out=None):
    """ddt_commit with the KV part written through a block table into k/v_pages
    [L][num_pages][Hkv][page_size][d]."""
    lib = _gpu()
    B, A = acc_nodes.shape
    dev = acc_nodes.device
    _need(acc_nodes, (B, A), torch.int32, "acc_nodes")
    _need(acc_len, (B,), torch.int32, "acc_len")
    _need(prefix_len, (B,), torch.int32, "prefix_len")
    La, _, N, Hkv, d = k_tree.shape
    num_pages, page = k_pages.shape[1], k_pages.shape[3]
    max_pages = block_table.shape[1]
    kdt = k_tree.dtype
    _need(k_tree, (La, B, N, Hkv, d), kdt, "k_tree")
    _need(v_tree, (La, B, N, Hkv, d), kdt, "v_tree")
    _need(k_pages, (La, num_pages, Hkv, page, d), kdt, "k_pages")
    _need(v_pages, (La, num_pages, Hkv, page, d), kdt, "v_pages")
    _need(block_table, (B, max_pages), torch.int32, "block_table")
    if S is not None:
        Lg, _, N2, C = x.shape
        if N2 != N:
            raise DDTError("tree rows differ between the attention and GDN parts")
        Hv, dv, dk = S.shape[2], S.shape[3], S.shape[4]
        K = conv_w.shape[2]
        _need(x, (Lg, B, N, C), x.dtype, "x")
        _need(conv_w, (Lg, C, K), x.dtype, "conv_w")
        _need(conv_state, (Lg, B, K - 1, C), x.dtype, "conv_state")
        _need(beta, (Lg, B, N, Hv), torch.float32, "beta")
        _need(decay, (Lg, B, N, Hv), torch.float32, "decay")
        _need(S, (Lg, B, Hv, dv, dk), torch.float32, "S")
        xd = _DT[x.dtype]
    else:
        Lg, Hv, dk, dv, K, xd = 0, 1, 1, 1, 1, F32
    o = out or {}
    i32 = dict(dtype=torch.int32, device=dev)
    res = {"src_row": o.get("src_row", torch.empty((B, A), **i32)),
           "dst_pos": o.get("dst_pos", torch.empty((B, A), **i32)),
           "status": o.get("status", torch.empty((B,), **i32))}
    rc = lib.ddt_commit_paged(B, N, A, La, Hkv, d, page, num_pages, max_pages, _ptr(block_table), _DT[kdt],
                              _ptr(k_tree), _ptr(v_tree), _ptr(k_pages), _ptr(v_pages), Lg, Hk, Hv, dk, dv, K, xd,
                              _ptr(x), _ptr(conv_w), _ptr(beta), _ptr(decay), _ptr(S), _ptr(conv_state),
                              _ptr(acc_nodes), _ptr(acc_len), _ptr(prefix_len), _ptr(res["src_row"]),
                              _ptr(res["dst_pos"]), _ptr(res["status"]), _stream())
    _check(rc, "ddt_commit_paged")
    return res
