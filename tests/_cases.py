"""Seeded test cases shared by the GPU parity tests (inputs from the synth module; trees
from the oracle's own build, so that no oracle input comes from the CUDA path)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tree_speculative_decoding_02_gb300 import synth


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_tree(logits_cpu, root, prefix, top_k, budget):
    return oracle.build_tree(f64(logits_cpu), np.asarray(root), np.asarray(prefix), top_k, budget)


def tree_to_dev(tree, dev="cuda"):
    """Oracle tree arrays as int32 device tensors (the mask words keep their bits)."""
    out = {k: torch.as_tensor(np.ascontiguousarray(tree[k], dtype=np.int32)).to(dev)
           for k in ("token", "parent", "depth", "position", "n_nodes")}
    out["anc"] = torch.as_tensor(np.ascontiguousarray(tree["anc"]).view(np.int32)).to(dev)
    return out


def tree_from_logits(workload, B, D, V, top_k, budget, *, std=3.0, boost=6.0, prefix=None, tensor=1):
    g = synth.gen(workload, tensor)
    logits = synth.draft_logits(B, D, V, std=std, boost=boost, g=g, dtype=torch.bfloat16)
    prefix = np.zeros(B, np.int32) if prefix is None else np.asarray(prefix, np.int32)
    root = np.arange(B, dtype=np.int32) + 7
    return oracle_tree(logits, root, prefix, top_k, budget), logits


def s_to_oracle(S_dev):
    """GPU state layout [..][dv][dk] -> oracle layout [..][dk][dv] (fp64)."""
    return np.swapaxes(f64(S_dev), -1, -2)
