"""Plain fp64 CPU oracle of one DDTree verification round -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  It wraps ``ddt_oracle.c`` (plain C, fp64) through ctypes and
shares no code with the CUDA library of ``tree_speculative_decoding_02_gb300``.

Inputs are numpy arrays (any float dtype is converted exactly to float64; bf16 data
should be passed as float32/float64 arrays holding the bf16 values).  Each function
returns a dict of numpy arrays.  The C functions cite the pages they follow.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ddt_oracle.c")
_HDR = os.path.join(_HERE, "ddt_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libddt_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C99, OpenMP over independent units)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB_PATH) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fopenmp", "-Wall",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            for name in ("ddto_build_tree", "ddto_attn_row", "ddto_tree_attn", "ddto_gdn_unit",
                         "ddto_tree_gdn", "ddto_walk", "ddto_commit", "ddto_gather_pages",
                         "ddto_scatter_pages", "ddto_rope_tree", "ddto_walk_flat", "ddto_walk_sample"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _u32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint32))


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def set_threads(n: int) -> None:
    """Number of OpenMP threads the oracle uses (spreads independent units only)."""
    os.environ["OMP_NUM_THREADS"] = str(int(n))
    try:
        lib = ctypes.CDLL("libgomp.so.1")
        lib.omp_set_num_threads(ctypes.c_int(int(n)))
    except OSError:
        pass


def build_tree(logits, root_token, prefix_len, top_k: int, budget: int):
    """Best-first tree build.  logits [B][D][V]."""
    lib = _load()
    logits = _f64(logits)
    B, D, V = logits.shape
    N = budget + 1
    W = (N + 31) // 32
    out = {name: np.zeros((B, N), np.int32) for name in ("token", "parent", "depth", "position", "rank")}
    out["n_nodes"] = np.zeros(B, np.int32)
    out["anc"] = np.zeros((B, N, W), np.uint32)
    out["score"] = np.zeros((B, N), np.float64)
    out["lse"] = np.zeros((B, D), np.float64)
    out["margin"] = np.zeros(B, np.float64)
    out["margin_depth"] = np.zeros((B, 2), np.int32)
    rc = lib.ddto_build_tree(
        B, D, V, int(top_k), int(budget), _p(logits), _p(_i32(root_token)), _p(_i32(prefix_len)),
        _p(out["token"]), _p(out["parent"]), _p(out["depth"]), _p(out["position"]), _p(out["rank"]),
        _p(out["n_nodes"]), _p(out["anc"]), _p(out["score"]), _p(out["lse"]), _p(out["margin"]),
        _p(out["margin_depth"]))
    _check(rc, "build_tree")
    return out


def attn_row(q, k_prefix, v_prefix, k_tree, v_tree, anc_row, n_nodes: int, scale: float):
    """One query row: q [d], k/v_prefix [P][d], k/v_tree [n][d], anc_row [W]."""
    lib = _load()
    q = _f64(q)
    kp, vp = _f64(k_prefix), _f64(v_prefix)
    kt, vt = _f64(k_tree), _f64(v_tree)
    d = q.shape[0]
    P = kp.shape[0]
    out = np.zeros(d, np.float64)
    rc = lib.ddto_attn_row(P, int(n_nodes), d, _p(q), _p(kp), _p(vp), ctypes.c_long(d), _p(kt), _p(vt),
                           ctypes.c_long(d), _p(_u32(anc_row)), ctypes.c_double(scale), _p(out))
    _check(rc, "attn_row")
    return out


def gather_pages(pages, block_table, prefix_len, Pcap: int):
    """pages [L][num_pages][Hkv][page][d], block_table [B][max_pages] -> the contiguous
    cache [L][B][Hkv][Pcap][d] (rows >= prefix_len zero)."""
    lib = _load()
    pages = _f64(pages)
    L, num_pages, Hkv, page, d = pages.shape
    bt = _i32(block_table)
    B, max_pages = bt.shape
    cache = np.zeros((L, B, Hkv, Pcap, d))
    rc = lib.ddto_gather_pages(L, B, Hkv, d, page, num_pages, max_pages, _p(pages), _p(bt), _p(_i32(prefix_len)),
                               Pcap, _p(cache))
    _check(rc, "gather_pages")
    return cache


def scatter_pages(cache, block_table, n_rows, pages):
    """Rows [0, n_rows[b]) of the contiguous cache [L][B][Hkv][Pcap][d] into (a copy of)
    pages [L][num_pages][Hkv][page][d]."""
    lib = _load()
    cache = _f64(cache)
    L, B, Hkv, Pcap, d = cache.shape
    out = _f64(pages).copy()
    num_pages, page = out.shape[1], out.shape[3]
    bt = _i32(block_table)
    max_pages = bt.shape[1]
    rc = lib.ddto_scatter_pages(L, B, Hkv, d, page, num_pages, max_pages, _p(cache), Pcap, _p(bt), _p(_i32(n_rows)),
                                _p(out))
    _check(rc, "scatter_pages")
    return out


def rope_tree(x, position, n_nodes, rot: int, theta: float = 10000.0):
    """Rotary embedding of x [L][B][N][H][d] at position [B][N] (a copy is returned)."""
    lib = _load()
    x = _f64(x).copy()
    L, B, N, H, d = x.shape
    rc = lib.ddto_rope_tree(L, B, N, H, d, int(rot), ctypes.c_double(theta), _p(_i32(position)),
                            _p(_i32(n_nodes)), _p(x))
    _check(rc, "rope_tree")
    return x


def tree_attn(q, k_tree, v_tree, k_cache, v_cache, prefix_len, n_nodes, anc, scale: float):
    """q [L][B][N][Hq][d]; k/v_tree [L][B][N][Hkv][d]; k/v_cache [L][B][Hkv][Pcap][d]."""
    lib = _load()
    q = _f64(q)
    L, B, N, Hq, d = q.shape
    k_cache = _f64(k_cache)
    Hkv, Pcap = k_cache.shape[2], k_cache.shape[3]
    o = np.zeros_like(q)
    rc = lib.ddto_tree_attn(L, B, N, Hq, Hkv, d, Pcap, _p(q), _p(_f64(k_tree)), _p(_f64(v_tree)),
                            _p(k_cache), _p(_f64(v_cache)), _p(_i32(prefix_len)), _p(_i32(n_nodes)),
                            _p(_u32(anc)), ctypes.c_double(scale), _p(o))
    _check(rc, "tree_attn")
    return {"o": o}


def gdn_unit(x, conv_w, conv_state, beta, decay, S0, parent, n_nodes: int, Hk: int, Hv: int, h: int,
             want_states: bool = False):
    """One (layer, request, value head): x [N][C], conv_w [C][K], conv_state [K-1][C],
    beta/decay [N][Hv], S0 [dk][dv], parent [N]."""
    lib = _load()
    x = _f64(x)
    N, C = x.shape
    S0 = _f64(S0)
    dk, dv = S0.shape
    conv_w = _f64(conv_w)
    K = conv_w.shape[1]
    o = np.zeros((N, dv), np.float64)
    sn = np.zeros((N, dk, dv), np.float64) if want_states else None
    rc = lib.ddto_gdn_unit(N, int(n_nodes), Hk, Hv, dk, dv, K, int(h), _p(x), _p(conv_w),
                           _p(_f64(conv_state)), _p(_f64(beta)), _p(_f64(decay)), _p(S0),
                           _p(_i32(parent)), _p(o), _p(sn))
    _check(rc, "gdn_unit")
    return {"o": o, "S_node": sn}


def tree_gdn(x, conv_w, conv_state, beta, decay, S, parent, n_nodes, Hk: int, want_states: bool = False):
    """x [L][B][N][C]; conv_w [L][C][K]; conv_state [L][B][K-1][C]; beta/decay [L][B][N][Hv];
    S [L][B][Hv][dk][dv]; parent [B][N]; n_nodes [B]."""
    lib = _load()
    x = _f64(x)
    L, B, N, C = x.shape
    S = _f64(S)
    Hv, dk, dv = S.shape[2], S.shape[3], S.shape[4]
    conv_w = _f64(conv_w)
    K = conv_w.shape[2]
    o = np.zeros((L, B, N, Hv, dv), np.float64)
    sn = np.zeros((L, B, N, Hv, dk, dv), np.float64) if want_states else None
    rc = lib.ddto_tree_gdn(L, B, N, Hk, Hv, dk, dv, K, _p(x), _p(conv_w), _p(_f64(conv_state)),
                           _p(_f64(beta)), _p(_f64(decay)), _p(S), _p(_i32(parent)), _p(_i32(n_nodes)),
                           _p(o), _p(sn))
    _check(rc, "tree_gdn")
    return {"o": o, "S_node": sn}


def walk(token, parent, n_nodes, D: int, target_logits=None, target_argmax=None, flat: bool = False):
    """Greedy tree walk.  target_logits [B][N][V] or target_argmax [B][N].  flat: the safe
    mode that only descends into first (rank-0) children."""
    lib = _load()
    token, parent = _i32(token), _i32(parent)
    B, N = token.shape
    A = D + 1
    if target_logits is not None:
        tl = _f64(target_logits)
        V = tl.shape[2]
        ta_in = None
    else:
        tl = None
        ta_in = _i32(target_argmax)
        V = 1
    out = {"target_argmax": np.zeros((B, N), np.int32), "acc_nodes": np.zeros((B, A), np.int32),
           "acc_len": np.zeros(B, np.int32), "bonus": np.zeros(B, np.int32),
           "emitted": np.zeros((B, A), np.int32), "n_emitted": np.zeros(B, np.int32)}
    fn = lib.ddto_walk_flat if flat else lib.ddto_walk
    rc = fn(B, N, V, D, _p(tl), _p(ta_in), _p(token), _p(parent), _p(_i32(n_nodes)),
            _p(out["target_argmax"]), _p(out["acc_nodes"]), _p(out["acc_len"]), _p(out["bonus"]),
            _p(out["emitted"]), _p(out["n_emitted"]))
    _check(rc, "walk")
    return out


def walk_sample(token, parent, n_nodes, D: int, target_logits, uniforms, temperature: float, C: int):
    """Tree-walk rejection sampling.  target_logits [B][N][V]; uniforms [B][D+1][C+1];
    C = the most children a node may have.  Adds status [B] and margin [B] (the smallest
    distance between a uniform's target and its threshold over the request's decisions)."""
    lib = _load()
    token, parent = _i32(token), _i32(parent)
    B, N = token.shape
    A = D + 1
    tl = _f64(target_logits)
    V = tl.shape[2]
    U = _f64(uniforms)
    if U.shape != (B, A, C + 1):
        raise ValueError(f"uniforms must be [B][D+1][C+1] = {(B, A, C + 1)}, got {U.shape}")
    out = {"acc_nodes": np.zeros((B, A), np.int32), "acc_len": np.zeros(B, np.int32),
           "bonus": np.zeros(B, np.int32), "emitted": np.zeros((B, A), np.int32),
           "n_emitted": np.zeros(B, np.int32), "margin": np.zeros(B, np.float64),
           "status": np.zeros(B, np.int32)}
    rc = lib.ddto_walk_sample(B, N, V, D, C, ctypes.c_double(float(temperature)), _p(tl), _p(U), _p(token),
                              _p(parent), _p(_i32(n_nodes)), _p(out["acc_nodes"]), _p(out["acc_len"]),
                              _p(out["bonus"]), _p(out["emitted"]), _p(out["n_emitted"]), _p(out["margin"]),
                              _p(out["status"]))
    _check(rc, "walk_sample")
    return out


def commit(acc_nodes, acc_len, prefix_len, *, k_tree=None, v_tree=None, k_cache=None, v_cache=None,
           x=None, conv_w=None, beta=None, decay=None, S=None, conv_state=None, Hk: int = 1):
    """Commit the accepted path.  Returns updated copies (inputs are not modified)."""
    lib = _load()
    acc_nodes = _i32(acc_nodes)
    B, A = acc_nodes.shape
    prefix_len = _i32(prefix_len).copy()
    if k_cache is not None:
        k_tree, v_tree = _f64(k_tree), _f64(v_tree)
        k_cache, v_cache = _f64(k_cache).copy(), _f64(v_cache).copy()
        La, _, N, Hkv, d = k_tree.shape
        Pcap = k_cache.shape[3]
    else:
        La, Hkv, d, Pcap = 0, 1, 1, 0
        N = None
    if S is not None:
        x = _f64(x)
        Lg, _, N2, C = x.shape
        N = N2 if N is None else N
        S = _f64(S).copy()
        conv_state = _f64(conv_state).copy()
        Hv, dk, dv = S.shape[2], S.shape[3], S.shape[4]
        conv_w = _f64(conv_w)
        K = conv_w.shape[2]
        beta, decay = _f64(beta), _f64(decay)
    else:
        Lg, Hv, dk, dv, K = 0, 1, 1, 1, 1
    if N is None:
        raise ValueError("commit needs the attention part, the GDN part, or both")
    out = {"src_row": np.zeros((B, A), np.int32), "dst_pos": np.zeros((B, A), np.int32),
           "status": np.zeros(B, np.int32)}
    rc = lib.ddto_commit(La, B, N, Hkv, d, Pcap, _p(k_tree), _p(v_tree), _p(k_cache), _p(v_cache),
                         Lg, Hk, Hv, dk, dv, K, _p(x), _p(conv_w), _p(beta), _p(decay), _p(S),
                         _p(conv_state), _p(acc_nodes), _p(_i32(acc_len)), A, _p(prefix_len),
                         _p(out["src_row"]), _p(out["dst_pos"]), _p(out["status"]))
    _check(rc, "commit")
    out.update({"prefix_len": prefix_len, "k_cache": k_cache, "v_cache": v_cache, "S": S,
                "conv_state": conv_state})
    return out
