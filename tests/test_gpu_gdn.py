"""GPU parity of ddt_tree_gdn against the oracle (normwise <= 2e-3 per output row)."""
import numpy as np
import pytest
import torch

import oracle
from tests import _cases as C
from tests._parity import TOL, normwise
from tree_speculative_decoding_02_gb300 import ddt, synth

pytestmark = pytest.mark.gpu


def _gpu(tree, gi, Hk, out_dtype=torch.float32):
    t = C.tree_to_dev(tree)
    S_dev = gi.S.transpose(-1, -2).contiguous().cuda()   # [dk][dv] draw -> [dv][dk] layout
    r = ddt.ddt_tree_gdn(gi.x.cuda(), gi.conv_w.cuda(), gi.conv_state.cuda(), gi.beta.cuda(), gi.decay.cuda(),
                         S_dev, t["parent"], t["n_nodes"], Hk=Hk, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return r


def _check(got, want, tree):
    got = got.cpu().double().numpy()
    assert np.isfinite(got).all()
    for b in range(got.shape[1]):
        n = int(tree["n_nodes"][b])
        err = normwise(got[:, b, :n], want[:, b, :n], axes=-1)
        assert err.max() <= TOL, f"request {b}: max normwise error {err.max():.3g}"
        assert (got[:, b, n:] == 0).all()


def _oracle(tree, gi, Hk):
    return oracle.tree_gdn(C.f64(gi.x), C.f64(gi.conv_w), C.f64(gi.conv_state), C.f64(gi.beta), C.f64(gi.decay),
                           C.f64(gi.S), tree["parent"], tree["n_nodes"], Hk)["o"]


def test_gdn_tiny_round_fp32():
    """One GDN layer, Hk=Hv=2, dk=dv=32, conv 4, fp32; budget 16 tree of the tiny round."""
    tree, _ = C.tree_from_logits(1, 1, 8, 1024, 8, 16, std=2.0, boost=0.0)
    gi = synth.gdn_inputs(1, 1, 17, 2, 2, 32, 32, 4, workload=1, dtype=torch.float32)
    r = _gpu(tree, gi, 2)
    _check(r["o"], _oracle(tree, gi, 2), tree)


@pytest.mark.parametrize("dims", [(128, 128), (64, 64), (64, 128)])
def test_gdn_bf16_multi(dims):
    dk, dv = dims
    tree, _ = C.tree_from_logits(4, 2, 15, 3000, 8, 64)
    gi = synth.gdn_inputs(2, 2, 65, 2, 6, dk, dv, 4, workload=4, dtype=torch.bfloat16)
    r = _gpu(tree, gi, 2)
    _check(r["o"], _oracle(tree, gi, 2), tree)


def test_gdn_small_trees_and_root_only():
    tree, _ = C.tree_from_logits(4, 3, 3, 50, 2, 5, std=2.0, boost=0.0)
    tree0, _ = C.tree_from_logits(4, 3, 3, 50, 2, 0, std=2.0, boost=0.0)
    for tr in (tree, tree0):
        N = tr["token"].shape[1]
        gi = synth.gdn_inputs(1, 3, N, 1, 2, 32, 32, 4, workload=4, dtype=torch.float32)
        r = _gpu(tr, gi, 1)
        _check(r["o"], _oracle(tr, gi, 1), tr)


def test_gdn_malformed_tree_flagged():
    tree, _ = C.tree_from_logits(4, 2, 3, 50, 2, 5, std=2.0, boost=0.0)
    tree["parent"][1][3] = 5   # parent after child
    gi = synth.gdn_inputs(1, 2, 6, 1, 1, 32, 32, 4, workload=4, dtype=torch.float32)
    r = _gpu(tree, gi, 1)
    assert r["status"].cpu().tolist() == [0, 7]
    assert (r["o"][:, 1] == 0).all()


def test_gdn_tree_workload_full():
    """48 layers, Hk=16, Hv=48, dk=dv=128, budget-64 tree from a drafter-vocab build: every
    (layer, node, value head) output against the oracle, with fp32 and with bf16 outputs."""
    tree, _ = C.tree_from_logits(4, 1, 15, 151936, 8, 64)
    gi = synth.gdn_inputs(48, 1, 65, 16, 48, 128, 128, 4, workload=4, dtype=torch.bfloat16)
    r = _gpu(tree, gi, 16)
    _check(r["o"], _oracle(tree, gi, 16), tree)
    assert int(r["status"][0]) == 0
    _assert_rounded(_gpu(tree, gi, 16, out_dtype=torch.bfloat16)["o"], r["o"])


def _assert_rounded(o16, o32):
    """bf16 outputs are the fp32 outputs rounded: within one bf16 ulp, element by element."""
    assert o16.dtype == torch.bfloat16
    a, bq = o32.float(), o16.float()
    ulp = torch.clamp(a.abs(), min=1e-30) * 2.0 ** -7
    assert ((a - bq).abs() <= ulp).all()


@pytest.mark.parametrize("Hk,Hv,dtype,budget", [(2, 2, torch.bfloat16, 16), (1, 4, torch.float32, 64),
                                                 (2, 4, torch.float32, 32), (3, 6, torch.bfloat16, 0),
                                                 (1, 3, torch.bfloat16, 65), (1, 2, torch.float32, 62)])
def test_gdn_head128_variants(Hk, Hv, dtype, budget):
    """Head size 128: one or several value heads per key head, fp32 or bf16 inputs, root-only
    trees, and the largest trees the tensor-core path stages (66 rows for bf16, 63 for
    fp32); larger fp32 trees take the CUDA-core path."""
    tree, _ = C.tree_from_logits(4, 2, 15, 3000, 8, budget)
    gi = synth.gdn_inputs(2, 2, budget + 1, Hk, Hv, 128, 128, 4, workload=4, dtype=dtype)
    r = _gpu(tree, gi, Hk)
    _check(r["o"], _oracle(tree, gi, Hk), tree)
    assert (r["status"].cpu() == 0).all()


def test_gdn_head128_deep_chain():
    """A 17-node chain (depth 16, the head-128 path's limit) runs; a 20-node chain (depth
    19) is refused for that request."""
    for n in (17, 20):
        parent = np.array([[-1] + list(range(n - 1))], np.int32)
        tree = {"parent": parent, "n_nodes": np.array([n], np.int32), "token": np.zeros((1, n), np.int32),
                "depth": np.arange(n, dtype=np.int32)[None], "position": np.arange(n, dtype=np.int32)[None],
                "anc": np.zeros((1, n, (n + 31) // 32), np.uint32)}
        gi = synth.gdn_inputs(1, 1, n, 1, 2, 128, 128, 4, workload=4, dtype=torch.bfloat16)
        r = _gpu(tree, gi, 1)
        if n <= 17:
            _check(r["o"], _oracle(tree, gi, 1), tree)
            assert int(r["status"][0]) == 0
        else:
            assert int(r["status"][0]) == 2   # deeper than this path supports: refused per request


@pytest.mark.parametrize("K", [1, 2, 6])
def test_gdn_head128_conv_widths(K):
    """Conv widths other than 4 (the generic tensor-core instance), including no conv state."""
    tree, _ = C.tree_from_logits(4, 2, 15, 3000, 8, 24)
    gi = synth.gdn_inputs(1, 2, 25, 2, 4, 128, 128, K, workload=4, dtype=torch.bfloat16)
    r = _gpu(tree, gi, 2)
    _check(r["o"], _oracle(tree, gi, 2), tree)
    assert (r["status"].cpu() == 0).all()


@pytest.mark.parametrize("Hk,Hv,L", [(2, 6, 2), (16, 48, 1)])
def test_gdn_bf16_output_instance(Hk, Hv, L):
    """The instance the batched round runs (bf16 inputs and outputs, head 128, conv 4,
    budget-64 tree): each bf16 output within one bf16 rounding of the same call's fp32
    output, which is within the tolerance of the oracle."""
    tree, _ = C.tree_from_logits(4, 2, 15, 3000, 8, 64)
    gi = synth.gdn_inputs(L, 2, 65, Hk, Hv, 128, 128, 4, workload=4, dtype=torch.bfloat16)
    r32 = _gpu(tree, gi, Hk)
    _check(r32["o"], _oracle(tree, gi, Hk), tree)
    r16 = _gpu(tree, gi, Hk, out_dtype=torch.bfloat16)
    _assert_rounded(r16["o"], r32["o"])
    assert (r16["o"].float()[:, :, 65:] == 0).all()
    assert (r16["status"].cpu() == 0).all()


@pytest.mark.parametrize("case", ["tiny_fp32", "head128_bf16", "dk64_dv128"])
def test_gdn_node_states_match_oracle(case):
    """The optional per-node state output: every node's own branch-local state S_n, formed
    by reading its parent's state and writing its own scratch copy, against the oracle's
    per-node states (normwise per (layer, request, node, head) matrix); padding rows stay
    zero, and the outputs o (the normal path) still match."""
    if case == "tiny_fp32":
        tree, _ = C.tree_from_logits(1, 1, 8, 1024, 8, 16, std=2.0, boost=0.0)
        L, B, Hk, Hv, dk, dv, dt = 1, 1, 2, 2, 32, 32, torch.float32
    elif case == "head128_bf16":
        tree, _ = C.tree_from_logits(4, 2, 15, 3000, 8, 12)
        L, B, Hk, Hv, dk, dv, dt = 2, 2, 1, 3, 128, 128, torch.bfloat16
    else:
        tree, _ = C.tree_from_logits(4, 2, 6, 300, 3, 10, std=2.0, boost=0.0)
        L, B, Hk, Hv, dk, dv, dt = 1, 2, 2, 4, 64, 128, torch.float32
    N = tree["token"].shape[1]
    gi = synth.gdn_inputs(L, B, N, Hk, Hv, dk, dv, 4, workload=4, dtype=dt)
    t = C.tree_to_dev(tree)
    S_dev = gi.S.transpose(-1, -2).contiguous().cuda()
    sn = torch.full((L, B, N, Hv, dv, dk), float("nan"), device="cuda")
    r = ddt.ddt_tree_gdn(gi.x.cuda(), gi.conv_w.cuda(), gi.conv_state.cuda(), gi.beta.cuda(), gi.decay.cuda(),
                         S_dev, t["parent"], t["n_nodes"], Hk=Hk, out_dtype=torch.float32, S_node_debug=sn)
    torch.cuda.synchronize()
    want = oracle.tree_gdn(C.f64(gi.x), C.f64(gi.conv_w), C.f64(gi.conv_state), C.f64(gi.beta), C.f64(gi.decay),
                           C.f64(gi.S), tree["parent"], tree["n_nodes"], Hk, want_states=True)
    got = np.swapaxes(sn.cpu().double().numpy(), -1, -2)      # -> [..][dk][dv] like the oracle
    for b in range(B):
        n = int(tree["n_nodes"][b])
        err = normwise(got[:, b, :n], want["S_node"][:, b, :n], axes=(-2, -1))
        assert err.max() <= TOL, f"request {b}: node-state error {err.max():.3g}"
        assert (got[:, b, n:] == 0).all()
    _check(r["o"], want["o"], tree)
