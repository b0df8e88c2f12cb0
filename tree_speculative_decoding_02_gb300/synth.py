"""Seeded synthetic inputs for one DDTree verification round.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can be fed from it.
Seeds: workload c, tensor t -> ``1000 * c + t``.  Small tensors are drawn on the CPU
(bit-identical everywhere); the big prefix caches of the batched workload are drawn
on the device with a seeded CUDA generator.

The workloads follow the shapes of the pages' Qwen3.6-style hybrid target (full
attention + Gated DeltaNet layers) and of a DFlash drafter (depth 15, vocabulary
151936).  No dataset or trained weight is used; every value is synthetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# Workloads (sizes as named in the project's scope table).
WORKLOADS = {
    1: dict(name="tiny-round-fp32", B=1, P=256, D=8, V=1024, top_k=8, budget=16,
            Lf=1, Hq=4, Hkv=1, d=64, Lg=1, Hk=2, Hv=2, dk=32, dv=32, conv_k=4,
            dtype=torch.float32, logit_std=2.0, boost=0.0),
    2: dict(name="build-walk-bf16", B=1, D=15, V=151936, top_k=8, budgets=(32, 64),
            dtype=torch.bfloat16, logit_std=3.0, boost=6.0),
    3: dict(name="tree-attn-bf16", B=1, P=4096, Lf=16, Hq=24, Hkv=4, d=256, budget=64,
            D=15, V=151936, top_k=8, dtype=torch.bfloat16, logit_std=3.0, boost=6.0),
    4: dict(name="tree-gdn-bf16", B=1, P=0, Lg=48, Hk=16, Hv=48, dk=128, dv=128, conv_k=4, budget=64,
            D=15, V=151936, top_k=8, dtype=torch.bfloat16, logit_std=3.0, boost=6.0),
    5: dict(name="batched-round-bf16", B=32, P_lo=1024, P_hi=32768, D=15, V=151936, top_k=8, budget=64,
            Lf=16, Hq=24, Hkv=4, d=256, Lg=48, Hk=16, Hv=48, dk=128, dv=128, conv_k=4,
            dtype=torch.bfloat16, logit_std=3.0, boost=6.0),
}


def gen(workload: int, tensor: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(1000 * int(workload) + int(tensor))
    return g


def normal(shape, std=1.0, *, g, dtype=torch.float32, device="cpu"):
    t = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def draft_logits(B, D, V, *, std, boost, g, dtype, device="cpu"):
    """[B][D][V] logits ~ N(0, std), plus `boost` on one uniformly drawn token per
    (request, depth) -- a peaked, confident drafter."""
    t = torch.randn((B, D, V), generator=g, dtype=torch.float32, device=device) * std
    if boost:
        idx = torch.randint(0, V, (B, D, 1), generator=g, device=device)
        t.scatter_add_(2, idx, torch.full((B, D, 1), float(boost), device=device))
    return t.to(dtype)


def target_logits(B, N, V, *, g, dtype, device="cpu"):
    """[B][N][V] target logits ~ N(0, 1)."""
    return torch.randn((B, N, V), generator=g, dtype=torch.float32, device=device).to(dtype)


def plant_path(target, token, parent, n_nodes, path_len, *, boost=8.0):
    """Boost, along one root-to-node path of each request's tree, the target logit of
    the child token at each node, so that the walk accepts `path_len[b]` nodes (or
    stops where the tree ends).  Returns the planted node list per request.
    The path takes the first child in row order at each step (a seeded choice is made
    by the caller through `path_len`)."""
    B = target.shape[0]
    paths = []
    for b in range(B):
        cur, path = 0, [0]
        for _ in range(int(path_len[b])):
            kids = [c for c in range(1, int(n_nodes[b])) if int(parent[b][c]) == cur]
            if not kids:
                break
            nxt = kids[0]
            target[b, cur, int(token[b][nxt])] += boost
            cur = nxt
            path.append(cur)
        paths.append(path)
    return paths


def add_peaks(target, n_peaks, height, *, g):
    """Raise `n_peaks` seeded tokens of every row by height, height - 1, ...: a peaked
    target in which a few tokens hold much of each row's mass (in place, fp32)."""
    B, N, V = target.shape
    idx = torch.randint(0, V, (B, N, n_peaks), generator=g)
    bump = float(height) - torch.arange(n_peaks, dtype=torch.float32)
    target.scatter_add_(2, idx, bump.expand(B, N, n_peaks).contiguous())
    return target


def uniforms(B, A, C, *, g, device="cpu"):
    """[B][A][C + 1] fp32 uniforms in [0, 1): the random numbers of a sampling walk."""
    return torch.rand((B, A, C + 1), generator=g, dtype=torch.float32, device=device)


def prefix_lengths(B, lo, hi, *, g):
    """Committed prefix lengths ~ U{lo..hi}."""
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int32)


@dataclass
class AttnInputs:
    q: torch.Tensor
    k_tree: torch.Tensor
    v_tree: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    prefix_len: torch.Tensor
    extra: dict = field(default_factory=dict)


def attn_inputs(L, B, N, Hq, Hkv, d, Pcap, prefix_len, *, workload, dtype, device="cpu", poison=True):
    """Q / tree K,V / prefix caches ~ N(0,1).  Cache rows at or beyond a request's
    prefix length are NaN-poisoned, so any read past the prefix shows up."""
    q = normal((L, B, N, Hq, d), g=gen(workload, 10, device), dtype=dtype, device=device)
    k_tree = normal((L, B, N, Hkv, d), g=gen(workload, 11, device), dtype=dtype, device=device)
    v_tree = normal((L, B, N, Hkv, d), g=gen(workload, 12, device), dtype=dtype, device=device)
    k_cache = torch.empty((L, B, Hkv, Pcap, d), dtype=dtype, device=device)
    v_cache = torch.empty_like(k_cache)
    gk, gv = gen(workload, 13, device), gen(workload, 14, device)
    for l in range(L):  # per layer keeps the fp32 staging buffer small
        k_cache[l] = torch.randn((B, Hkv, Pcap, d), generator=gk, device=device).to(dtype)
        v_cache[l] = torch.randn((B, Hkv, Pcap, d), generator=gv, device=device).to(dtype)
    if poison:
        for b in range(B):
            p = int(prefix_len[b])
            k_cache[:, b, :, p:, :] = float("nan")
            v_cache[:, b, :, p:, :] = float("nan")
    return AttnInputs(q, k_tree, v_tree, k_cache, v_cache,
                      torch.as_tensor(prefix_len, dtype=torch.int32).to(device))


@dataclass
class GdnInputs:
    x: torch.Tensor
    conv_w: torch.Tensor
    conv_state: torch.Tensor
    beta: torch.Tensor
    decay: torch.Tensor
    S: torch.Tensor


def gdn_inputs(L, B, N, Hk, Hv, dk, dv, K, *, workload, dtype, device="cpu"):
    """Pre-conv channels x ~ N(0,1) (q | k | v), conv weights ~ 0.5 N(0,1), conv state
    ~ N(0,1), beta = sigmoid(N(0,1)), decay = exp(-softplus(N(0,1))) (fp32), committed
    state S ~ N(0,1) (fp32)."""
    C = 2 * Hk * dk + Hv * dv
    x = normal((L, B, N, C), g=gen(workload, 20, device), dtype=dtype, device=device)
    conv_w = normal((L, C, K), std=0.5, g=gen(workload, 21, device), dtype=dtype, device=device)
    conv_state = normal((L, B, K - 1, C), g=gen(workload, 22, device), dtype=dtype, device=device)
    zb = torch.randn((L, B, N, Hv), generator=gen(workload, 23, device), device=device)
    za = torch.randn((L, B, N, Hv), generator=gen(workload, 24, device), device=device)
    beta = torch.sigmoid(zb)
    decay = torch.exp(-torch.nn.functional.softplus(za))
    S = torch.randn((L, B, Hv, dk, dv), generator=gen(workload, 25, device), device=device)
    return GdnInputs(x, conv_w, conv_state, beta, decay, S)
