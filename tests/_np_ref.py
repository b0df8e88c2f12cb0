"""Independent numpy restatements used to pin the oracle (test-only).

Each helper computes a quantity by a different route than the oracle does -- brute
force over every candidate tree, causal attention over a stand-alone sequence, the
delta rule written in its projection form along a single path -- so that a mistake
in the oracle's bookkeeping or formulas shows up as a mismatch.
"""
from __future__ import annotations

import itertools
import math

import numpy as np


# ---------------------------------------------------------------------------- build
def rank_order(row):
    """Token ids of one depth sorted by (logit desc, id asc)."""
    row = np.asarray(row, dtype=np.float64)
    return np.lexsort((np.arange(row.shape[0]), -row))


def lse_exact(row):
    """log-sum-exp with an exactly rounded sum (math.fsum)."""
    row = np.asarray(row, dtype=np.float64)
    m = float(row.max())
    return m + math.log(math.fsum(np.exp(row - m).tolist()))


def brute_force_tree(logits, k, budget):
    """Every path of length 1..D whose depth-d token is among depth d's top-k, scored by
    the log of the product of its drafter probabilities; the first `budget` under
    (score desc, token sequence asc).  Returns (list of (score, seq)), sorted."""
    logits = np.asarray(logits, dtype=np.float64)
    D = logits.shape[0]
    tops = [rank_order(logits[d])[:k] for d in range(D)]
    lses = [lse_exact(logits[d]) for d in range(D)]
    cands = []
    for n in range(1, D + 1):
        for seq in itertools.product(*[tops[d] for d in range(n)]):
            logp = math.fsum(float(logits[d, t]) - lses[d] for d, t in enumerate(seq))
            cands.append((logp, tuple(int(t) for t in seq)))
    cands.sort(key=lambda c: (-c[0], c[1]))
    return cands[:budget], cands[budget:]


def tree_sequences(token, parent, n_nodes):
    """Token sequence (root excluded) of every row 1..n_nodes-1."""
    seqs = {}
    for i in range(1, int(n_nodes)):
        path = []
        j = i
        while j > 0:
            path.append(int(token[j]))
            j = int(parent[j])
        seqs[i] = tuple(reversed(path))
    return seqs


def anc_from_parent(parent, n_nodes, N):
    W = (N + 31) // 32
    anc = np.zeros((N, W), np.uint32)
    for i in range(int(n_nodes)):
        j = i
        while j >= 0:
            anc[i, j // 32] |= np.uint32(1 << (j % 32))
            j = int(parent[j]) if j > 0 else -1
    return anc


def path_rows(parent, i):
    """Rows root..i along the ancestor chain."""
    p = []
    j = i
    while j >= 0:
        p.append(j)
        j = int(parent[j]) if j > 0 else -1
    return list(reversed(p))


# ------------------------------------------------------------------------ attention
def causal_attention(q, k, v, scale):
    """Plain causal self-attention of a stand-alone sequence: q, k, v [T][d]."""
    q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
    T = q.shape[0]
    s = scale * (q @ k.T)
    s = np.where(np.tril(np.ones((T, T), bool)), s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


# ------------------------------------------------------------------------------ GDN
def silu(z):
    return z / (1.0 + np.exp(-z))


def gdn_sequence(xs, conv_w, conv_state, betas, decays, S0, Hk, Hv, h):
    """Gated delta rule over one stand-alone token sequence, written in projection form
        S_t = a_t (I - b_t k k^T) S_{t-1} + b_t k v^T,   o_t = S_t^T q,
    after a causal depthwise conv of width K over [conv_state ; xs] and SiLU, with q, k
    L2-normalised (eps 1e-6) and q scaled by dk^-1/2.  Returns (o [n][dv], S [n][dk][dv])."""
    xs = np.asarray(xs, np.float64)
    conv_w = np.asarray(conv_w, np.float64)
    S = np.asarray(S0, np.float64).copy()
    dk, dv = S.shape
    K = conv_w.shape[1]
    seq = np.concatenate([np.asarray(conv_state, np.float64).reshape(K - 1, -1), xs], axis=0)
    g = h // (Hv // Hk)
    qs = slice(g * dk, (g + 1) * dk)
    ks = slice(Hk * dk + g * dk, Hk * dk + (g + 1) * dk)
    vs = slice(2 * Hk * dk + h * dv, 2 * Hk * dk + (h + 1) * dv)
    outs, states = [], []
    for t in range(xs.shape[0]):
        window = seq[t:t + K]                     # oldest first, current last
        y = silu(np.einsum("kc,ck->c", window, conv_w))
        q = y[qs] / math.sqrt(float(y[qs] @ y[qs]) + 1e-6) / math.sqrt(dk)
        k = y[ks] / math.sqrt(float(y[ks] @ y[ks]) + 1e-6)
        v = y[vs]
        a, b = float(decays[t]), float(betas[t])
        S = a * (np.eye(dk) - b * np.outer(k, k)) @ S + b * np.outer(k, v)
        outs.append(S.T @ q)
        states.append(S.copy())
    return np.array(outs), np.array(states)


# ----------------------------------------------------------------------------- walk
def walk_bruteforce(token, parent, n_nodes, argmax):
    """Deepest node whose every edge matches the target argmax of its parent row."""
    best, best_depth = 0, 0
    for i in range(1, int(n_nodes)):
        path = path_rows(parent, i)
        ok = all(int(token[path[j + 1]]) == int(argmax[path[j]]) for j in range(len(path) - 1))
        if ok and len(path) - 1 > best_depth:
            best, best_depth = i, len(path) - 1
    return best, path_rows(parent, best)
