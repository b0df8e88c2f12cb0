"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerance (2e-3 max relative error with fp32 accumulation, read normwise): for every output
vector (one (layer, request, row, head) attention or GDN output, one (layer, request,
head) GDN state matrix) max|gpu - oracle| / max|oracle| <= 2e-3, with the GPU writing
fp32 outputs.  Integer outputs (tree arrays, masks, accepted rows, commit indices) must
match exactly.  Near-ties of the tree build across depths are handled by NEAR_TIE.
"""
from __future__ import annotations

import numpy as np

TOL = 2e-3
# Two paths at different depths whose log-probabilities differ by less than this are a
# near-tie: the GPU's per-depth log-sum-exp (fp32 exp, fp64 sums) and the oracle's (fp64)
# may order them differently.
NEAR_TIE = 1e-5


def normwise(got, want, axes):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    num = np.abs(got - want).max(axis=axes)
    den = np.abs(want).max(axis=axes)
    return num / np.maximum(den, 1e-30)


def tree_sequences(token, parent, n):
    seqs = {}
    for i in range(1, int(n)):
        path, j = [], i
        while j > 0:
            path.append(int(token[j]))
            j = int(parent[j])
        seqs[i] = tuple(reversed(path))
    return seqs


def assert_tree_equal(gpu, orc, b, check_scores=True):
    """Bit-exact tree arrays; on a flagged near-tie, only the cut may differ."""
    n_g, n_o = int(gpu["n_nodes"][b]), int(orc["n_nodes"][b])
    assert n_g == n_o, f"request {b}: n_nodes {n_g} vs {n_o}"
    same = all(np.array_equal(np.asarray(gpu[k][b]), np.asarray(orc[k][b]))
               for k in ("token", "parent", "depth", "position"))
    same = same and np.array_equal(np.asarray(gpu["anc"][b]).view(np.uint32), np.asarray(orc["anc"][b]))
    if not same:
        md = orc["margin_depth"][b]
        near = orc["margin"][b] < NEAR_TIE and md[0] != md[1]
        assert near, f"request {b}: tree differs from the oracle (margin {orc['margin'][b]:.3g})"
        # near-tie: the node sets may differ only by swaps within the tie window, on both
        # sides: every oracle node the GPU left out scores within NEAR_TIE of the cut (the
        # oracle's lowest selected score), and so does every GPU node the oracle left out
        # (by the GPU's own score, which differs from the exact one by ~1e-7)
        sg = tree_sequences(gpu["token"][b], gpu["parent"][b], n_g)
        so = tree_sequences(orc["token"][b], orc["parent"][b], n_o)
        cut = min(orc["score"][b][1:n_o])
        set_g, set_o = set(sg.values()), set(so.values())
        for i, s in so.items():
            if s not in set_g:
                assert orc["score"][b][i] - cut < NEAR_TIE, f"request {b}: oracle node {s} left out"
        extra = [i for i, s in sg.items() if s not in set_o]
        assert len(extra) == sum(1 for s in so.values() if s not in set_g)
        if extra:
            assert gpu.get("score") is not None, "a near-tie swap can only be checked with the GPU's scores"
            for i in extra:
                assert abs(float(gpu["score"][b][i]) - cut) < NEAR_TIE, f"request {b}: GPU node {sg[i]} outside the tie window"
        return
    if check_scores and gpu.get("score") is not None:
        sg = np.asarray(gpu["score"][b][:n_g])
        np.testing.assert_allclose(sg, orc["score"][b][:n_o], rtol=0, atol=1e-5)
