"""GPU parity of ddt_tree_attn against the oracle (normwise <= 2e-3 per output row)."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import _cases as C
from tests._parity import TOL, normwise
from tree_speculative_decoding_02_gb300 import ddt, synth

pytestmark = pytest.mark.gpu


def _case(workload, L, B, Hq, Hkv, d, prefix, budget, dtype, Pcap=None, D=6, V=300, k=4):
    tree, _ = C.tree_from_logits(workload, B, D, V, k, budget, std=2.0, boost=0.0, prefix=prefix)
    N = budget + 1
    Pcap = Pcap or (max(prefix) + N + 5)
    inp = synth.attn_inputs(L, B, N, Hq, Hkv, d, Pcap, np.asarray(prefix), workload=workload, dtype=dtype)
    return tree, inp, N


def _gpu(tree, inp, out_dtype=torch.float32):
    t = C.tree_to_dev(tree)
    r = ddt.ddt_tree_attn(inp.q.cuda(), inp.k_tree.cuda(), inp.v_tree.cuda(), inp.k_cache.cuda(),
                          inp.v_cache.cuda(), inp.prefix_len.cuda(), t["n_nodes"], t["anc"],
                          scale=1.0 / math.sqrt(inp.q.shape[-1]), out_dtype=out_dtype)
    torch.cuda.synchronize()
    return r


def _oracle(tree, inp, d):
    return oracle.tree_attn(C.f64(inp.q), C.f64(inp.k_tree), C.f64(inp.v_tree),
                            np.nan_to_num(C.f64(inp.k_cache)), np.nan_to_num(C.f64(inp.v_cache)),
                            inp.prefix_len.numpy(), tree["n_nodes"], tree["anc"], 1 / math.sqrt(d))["o"]


def _check(got, want, tree):
    got = got.cpu().double().numpy()
    assert np.isfinite(got).all()
    for b in range(got.shape[1]):
        n = int(tree["n_nodes"][b])
        err = normwise(got[:, b, :n], want[:, b, :n], axes=-1)
        assert err.max() <= TOL, f"request {b}: max normwise error {err.max():.3g}"
        assert (got[:, b, n:] == 0).all()


def test_attn_tiny_round_fp32():
    """One layer, Hq=4, Hkv=1, d=64, prefix 256, budget 16, fp32."""
    tree, inp, N = _case(1, 1, 1, 4, 1, 64, [256], 16, torch.float32, D=8, V=1024, k=8)
    r = _gpu(tree, inp)
    _check(r["o"], _oracle(tree, inp, 64), tree)
    assert int(r["status"][0]) == 0


@pytest.mark.parametrize("d", [64, 128, 256])
def test_attn_bf16_ragged(d):
    """bf16, GQA group 6, ragged prefixes (0, 1, 300 rows), NaN-poisoned cache tails."""
    tree, inp, N = _case(3, 2, 3, 24, 4, d, [0, 1, 300], 64, torch.bfloat16)
    r = _gpu(tree, inp)
    _check(r["o"], _oracle(tree, inp, d), tree)
    rb = _gpu(tree, inp, out_dtype=torch.bfloat16)
    # bf16 output = fp32 output rounded (within one bf16 ulp)
    a = r["o"].float()
    bq = rb["o"].float()
    ulp = torch.clamp(a.abs(), min=1e-30) * 2.0 ** -7
    assert ((a - bq).abs() <= ulp).all()


def test_attn_no_gqa_and_single_row():
    tree, inp, N = _case(3, 1, 2, 2, 2, 128, [129, 7], 0, torch.bfloat16)
    r = _gpu(tree, inp)
    _check(r["o"], _oracle(tree, inp, 128), tree)


def test_attn_bad_prefix_flagged():
    tree, inp, N = _case(3, 1, 2, 4, 1, 64, [10, 10], 8, torch.float32)
    inp.prefix_len[1] = inp.k_cache.shape[3] + 1
    r = _gpu(tree, inp)
    assert r["status"].cpu().tolist() == [0, 3]
    assert (r["o"][:, 1] == 0).all()


def test_attn_tree_verify_workload_full():
    """Prefix 4096, 16 layers, Hq=24, Hkv=4, d=256, tree of budget 64 from a drafter-vocab
    build: every one of the 16 x 65 x 24 output rows against the oracle."""
    tree, _ = C.tree_from_logits(3, 1, 15, 151936, 8, 64, prefix=[4096])
    N = 65
    inp = synth.attn_inputs(16, 1, N, 24, 4, 256, 4096 + 16, [4096], workload=3, dtype=torch.bfloat16)
    r = _gpu(tree, inp)
    assert int(r["status"][0]) == 0
    _check(r["o"], _oracle(tree, inp, 256), tree)


def test_attn_bf16_split_kv_and_big_tree():
    """Long prefix with few work units (split-KV partials + merge) and a 201-row tree
    (several tree tiles and M-tiles); ragged prefix lengths incl. one shorter than a tile."""
    tree, inp, N = _case(6, 1, 2, 8, 2, 128, [2000, 37], 200, torch.bfloat16, D=12, V=400, k=6)
    r = _gpu(tree, inp)
    _check(r["o"], _oracle(tree, inp, 128), tree)
    assert r["status"].cpu().tolist() == [0, 0]


def test_attn_bf16_values_past_fp16_range():
    """V values far past fp16's range (prefix keys, the last row of a shifted prefix
    tile, a tree key) are applied at bf16 precision like any other."""
    tree, inp, N = _case(3, 2, 2, 24, 4, 256, [300, 130], 64, torch.bfloat16)
    vc = inp.v_cache.float()
    vc[0, 0, 1, 70:72] *= 3e5      # one prefix tile of request 0, kv head 1
    vc[1, 1, 2, 129] = 7e4         # the last prefix row of request 1 (a shifted tile)
    inp.v_cache = vc.to(torch.bfloat16)
    vt = inp.v_tree.float()
    vt[1, 0, 3, 0] = -2e5          # a tree key of request 0, kv head 0
    inp.v_tree = vt.to(torch.bfloat16)
    r = _gpu(tree, inp)
    _check(r["o"], _oracle(tree, inp, 256), tree)
    assert r["status"].cpu().tolist() == [0, 0]


def test_attn_bf16_values_far_past_fp16_range():
    """V values of 1e5 to 5e8 (prefix tiles of both requests, a tree key) among N(0, 1)
    values in the same rows: bf16 V is applied as it is, whatever its range."""
    tree, inp, N = _case(3, 2, 2, 24, 4, 256, [300, 700], 64, torch.bfloat16)
    vc = inp.v_cache.float()
    vc[0, 0, 1, 5] *= 3e7          # tile 0 of request 0, kv head 1: bf16 path
    vc[1, 1, 3, 650] = -5e8        # a later tile of request 1: bf16 path
    vc[1, 1, 0, 200] = 1e5         # scaled fp16 (s = 3)
    inp.v_cache = vc.to(torch.bfloat16)
    vt = inp.v_tree.float()
    vt[0, 1, 10, 2] = 2e7          # the tree tile of request 1: bf16 path
    inp.v_tree = vt.to(torch.bfloat16)
    for d in (256,):
        r = _gpu(tree, inp)
        _check(r["o"], _oracle(tree, inp, d), tree)
        assert r["status"].cpu().tolist() == [0, 0]
