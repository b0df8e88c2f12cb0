"""ddt_build_tree_noalloc: the tree build for callers that cannot allocate device memory
(its scratch is the library's fixed 4 MiB device array).  Its results must equal those
of ddt_build_tree with a caller-supplied workspace, on two calls in a row (different
sizes, so stale contents of the shared array would show), and sizes whose scratch
would not fit must be refused before anything runs.  This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

from tests import _cases as C
from tests._parity import assert_tree_equal
from tree_speculative_decoding_02_gb300 import ddt, synth

pytestmark = pytest.mark.gpu

KEYS = ("token", "parent", "depth", "position", "n_nodes", "anc", "score", "status")


def _outs(B, N, dev):
    i32 = dict(dtype=torch.int32, device=dev)
    return {"token": torch.full((B, N), -7, **i32), "parent": torch.full((B, N), -7, **i32),
            "depth": torch.full((B, N), -7, **i32), "position": torch.full((B, N), -7, **i32),
            "n_nodes": torch.zeros((B,), **i32), "anc": torch.zeros((B, N, (N + 31) // 32), **i32),
            "score": torch.zeros((B, N), dtype=torch.float64, device=dev), "status": torch.full((B,), -1, **i32)}


def _host(d):
    return {k: v.cpu().numpy() for k, v in d.items()}


def test_noalloc_build_matches_workspace_build_twice():
    dev = torch.device("cuda")
    cases = [(4, 15, 151936, 8, 64, 51), (2, 9, 5000, 5, 37, 52)]   # different partial layouts
    for (B, D, V, k, budget, wl) in cases:
        logits = synth.draft_logits(B, D, V, std=3.0, boost=6.0, g=synth.gen(wl, 1), dtype=torch.bfloat16).to(dev)
        root = torch.arange(B, dtype=torch.int32, device=dev)
        pl = torch.arange(B, dtype=torch.int32, device=dev) * 100
        want = ddt.ddt_build_tree(logits, root, pl, k, budget)
        got = ddt.ddt_build_tree_noalloc(logits, root, pl, k, budget, out=_outs(B, budget + 1, dev))
        torch.cuda.synchronize()
        w, g = _host(want), _host(got)
        for key in KEYS:
            np.testing.assert_array_equal(g[key], w[key], err_msg=key)
        assert (g["status"] == 0).all()
        # and both equal the oracle's tree
        orc = C.oracle_tree(logits.cpu(), root.cpu().numpy(), pl.cpu().numpy(), k, budget)
        for b in range(B):
            assert_tree_equal(g, orc, b)


def test_noalloc_refuses_oversized_scratch():
    dev = torch.device("cuda")
    lib = ddt.load()
    B, D, V, k = 2048, 64, 1000, 32   # needs ~35 MiB of per-row results
    assert lib.ddt_build_tree_workspace(B, D, V, k) > (4 << 20)
    p = ctypes.c_void_p(torch.empty(16, device=dev).data_ptr())
    rc = lib.ddt_build_tree_noalloc(B, D, V, k, 64, 1, *([p] * 11), None)
    assert rc == 3
