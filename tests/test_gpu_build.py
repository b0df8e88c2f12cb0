"""GPU parity of ddt_build_tree against the oracle (bit-exact tree arrays)."""
import numpy as np
import pytest
import torch

from tests import _cases as C
from tests._parity import assert_tree_equal
from tree_speculative_decoding_02_gb300 import ddt, synth

pytestmark = pytest.mark.gpu


def _run(logits, root, prefix, k, budget):
    dev = torch.device("cuda")
    g = ddt.ddt_build_tree(logits.to(dev), torch.as_tensor(root, dtype=torch.int32, device=dev),
                           torch.as_tensor(prefix, dtype=torch.int32, device=dev), k, budget)
    torch.cuda.synchronize()
    return {k_: (v.cpu().numpy() if v is not None else None) for k_, v in g.items()}


def _compare(logits, root, prefix, k, budget):
    o = C.oracle_tree(logits, root, prefix, k, budget)
    g = _run(logits, root, prefix, k, budget)
    assert (g["status"] == 0).all()
    for b in range(logits.shape[0]):
        assert_tree_equal(g, o, b)
    return g, o


def test_build_tiny_round_fp32():
    """B=1, depth 8, V=1024, N(0,2) logits, budget 16, top-k 8, fp32."""
    g = synth.gen(1, 1)
    logits = synth.draft_logits(1, 8, 1024, std=2.0, boost=0.0, g=g, dtype=torch.float32)
    _compare(logits, [11], [256], 8, 16)


@pytest.mark.parametrize("budget", [32, 64])
def test_build_drafter_vocab_bf16(budget):
    """B=1, depth 15, V=151936, N(0,3) + 6 on one token per depth, top-k 8, bf16."""
    g = synth.gen(2, 1)
    logits = synth.draft_logits(1, 15, 151936, std=3.0, boost=6.0, g=g, dtype=torch.bfloat16)
    gpu, orc = _compare(logits, [3], [100], 8, budget)
    assert gpu["n_nodes"][0] == budget + 1


def test_build_batched_ragged_prefix():
    g = synth.gen(5, 1)
    logits = synth.draft_logits(4, 15, 151936, std=3.0, boost=6.0, g=g, dtype=torch.bfloat16)
    pl = synth.prefix_lengths(4, 1024, 32768, g=synth.gen(5, 2)).numpy()
    _compare(logits, [1, 2, 3, 4], pl, 8, 64)


@pytest.mark.parametrize("seed", range(24))
def test_build_random_small(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    V = int(rng.integers(2, 70))
    D = int(rng.integers(1, 9))
    k = int(rng.integers(1, min(8, V) + 1))
    budget = int(rng.integers(0, 65))
    if seed % 3 == 0:   # integer-valued logits: exact ties everywhere
        logits = torch.as_tensor(rng.integers(-3, 4, size=(B, D, V)).astype(np.float32))
    else:
        logits = torch.as_tensor(rng.normal(0, 2, size=(B, D, V)).astype(np.float32))
    if seed % 2:
        logits = logits.to(torch.bfloat16)
    _compare(logits, rng.integers(0, V, B), rng.integers(0, 1000, B), k, budget)


def test_build_k1_chain_and_empty_budget():
    g = synth.gen(1, 3)
    logits = synth.draft_logits(2, 6, 300, std=2.0, boost=0.0, g=g, dtype=torch.float32)
    gpu, _ = _compare(logits, [0, 1], [5, 6], 1, 10)
    assert (gpu["n_nodes"] == 7).all()
    gpu, _ = _compare(logits, [0, 1], [5, 6], 4, 0)
    assert (gpu["n_nodes"] == 1).all()


def test_build_max_sizes():
    """budget 1023 (N = 1024 rows, 32 mask words), top-k 32, depth 40."""
    rng = np.random.default_rng(5)
    logits = torch.as_tensor(rng.normal(0, 1.5, size=(1, 40, 700)).astype(np.float32))
    _compare(logits, [9], [0], 32, 1023)


def test_build_nonfinite_logits_flagged():
    g = synth.gen(1, 4)
    logits = synth.draft_logits(2, 4, 5000, std=2.0, boost=0.0, g=g, dtype=torch.float32)
    logits[1, 2, 77] = float("nan")
    out = _run(logits, [0, 0], [0, 0], 4, 8)
    assert out["status"][0] == 0 and out["status"][1] == 6
    assert out["n_nodes"][1] == 1


@pytest.mark.parametrize("k", [1, 8, 32])
def test_build_many_ties_wide_vocab(k):
    """Integer-valued logits over a 20000-token vocabulary (three chunks, the last one
    ragged): thousands of exact ties in every chunk, so the lowest-id rule decides which
    entries make each top k."""
    rng = np.random.default_rng(40 + k)
    logits = torch.as_tensor(rng.integers(-2, 3, size=(2, 5, 20000)).astype(np.float32)).to(torch.bfloat16)
    _compare(logits, [1, 2], [10, 20], k, 40)
