"""GPU parity of ddt_walk_accept_sample (tree-walk rejection sampling) against the oracle.

Both sides take the same uniforms.  A request whose oracle margin (the smallest distance
between a uniform's target and the threshold it met) is at least 1e-5 must match the
oracle exactly; the GPU's normaliser carries an error of about 1e-6, so a request below
that margin may take the other side of one decision, and is then checked as a valid walk
of the same rule within 1e-5 (every decision replayed against fp64 probabilities)."""
import numpy as np
import pytest
import torch

import oracle
from tests import _cases as C
from tree_speculative_decoding_02_gb300 import ddt, synth

pytestmark = pytest.mark.gpu

_KEYS = ("acc_nodes", "acc_len", "bonus", "emitted", "n_emitted", "status")
EXACT_MARGIN = 1e-5


def _softmax(x, T):
    z = np.exp((x - x.max()) / T)
    return z / z.sum()


def _gpu(tree, D, tl, U, T):
    t = C.tree_to_dev(tree)
    r = ddt.ddt_walk_accept_sample(t["token"], t["parent"], t["n_nodes"], D, target_logits=tl.cuda(),
                                   uniforms=U.cuda(), temperature=T)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in r.items()}


def _replay_ok(tok, par, n, tl, U, T, C_, g, eps=EXACT_MARGIN):
    """The GPU walk of one request is a walk of the rule: each decision on the far side of
    its threshold by less than eps at most (fp64 probabilities)."""
    A = U.shape[0]
    a = int(g["acc_len"])
    path = [int(x) for x in g["acc_nodes"][:a + 1]]
    assert path[0] == 0 and (g["acc_nodes"][a + 1:] == -1).all()
    for s, u in enumerate(path):
        p = _softmax(tl[u], T)
        kids = [c for c in range(1, n) if par[c] == u]
        nxt = path[s + 1] if s + 1 < len(path) else None
        if nxt is not None:
            assert nxt in kids
            tried = kids[:kids.index(nxt) + 1]
        else:
            tried = kids if s + 1 < A else []
        R, rejected = 0.0, []
        for i, c in enumerate(tried):
            thr = p[tok[c]] / (1.0 - R)
            if c == nxt:
                assert U[s][i] < thr + eps, (s, i, U[s][i], thr)
            else:
                assert U[s][i] >= thr - eps, (s, i, U[s][i], thr)
                R += p[tok[c]]
                rejected.append(tok[c])
        if nxt is None:
            t = int(g["bonus"])
            assert 0 <= t < len(p) and t not in rejected
            q = p.copy()
            q[rejected] = 0.0
            cs = np.cumsum(q)
            target = U[s][C_] * (1.0 - R)
            assert cs[t] - q[t] - eps <= target <= cs[t] + eps, (t, target, cs[t] - q[t], cs[t])
    em = [int(tok[r]) for r in path[1:]] + [int(g["bonus"])]
    assert g["emitted"][:a + 1].tolist() == em and (g["emitted"][a + 1:] == -1).all()
    assert g["n_emitted"] == a + 1 and g["status"] == 0


def _compare(tree, D, tl, U, T, C_, g, o, min_exact=0.5):
    """Exact where the oracle's margin allows it, a valid walk elsewhere; returns the
    number of requests compared exactly."""
    B = tree["token"].shape[0]
    tl64, U64 = C.f64(tl), U.double().numpy()
    exact = 0
    for b in range(B):
        if o["status"][b] != 0 or o["margin"][b] >= EXACT_MARGIN:
            for k in _KEYS:
                np.testing.assert_array_equal(g[k][b], o[k][b], err_msg=f"{k} of request {b}")
            exact += 1
        else:
            _replay_ok(tree["token"][b], tree["parent"][b], int(tree["n_nodes"][b]), tl64[b], U64[b], T, C_,
                       {k: g[k][b] for k in _KEYS})
    assert exact >= min_exact * B, f"only {exact} of {B} requests had a margin for an exact comparison"
    return exact


def _peaked_target(tree, V, workload, lens, *, boost, peaks=3, height=12.0, dtype=torch.bfloat16):
    B, N = tree["token"].shape
    tl = synth.target_logits(B, N, V, g=synth.gen(workload, 30), dtype=torch.float32)
    synth.add_peaks(tl, peaks, height, g=synth.gen(workload, 31))
    synth.plant_path(tl, tree["token"], tree["parent"], tree["n_nodes"], lens, boost=boost)
    return tl.to(dtype)


@pytest.mark.parametrize("T", [1.0, 0.6, 1.7])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sample_small_trees(T, dtype):
    """V = 1000 (one chunk, a ragged vector tail), trees of budget 24, top-k 4."""
    B, D, V, k = 24, 6, 1000, 4
    tree, _ = C.tree_from_logits(41, B, D, V, k, 24, std=2.0, boost=3.0)
    lens = np.random.default_rng(41).integers(0, D + 1, B)
    tl = _peaked_target(tree, V, 41, lens, boost=6.0, height=6.0, dtype=dtype)
    U = synth.uniforms(B, D + 1, k, g=synth.gen(41, 32))
    g = _gpu(tree, D, tl, U, T)
    o = oracle.walk_sample(tree["token"], tree["parent"], tree["n_nodes"], D, C.f64(tl), U.double().numpy(), T, k)
    _compare(tree, D, tl, U, T, k, g, o, min_exact=0.8)
    assert g["acc_len"].max() > 0 and (g["acc_len"] == 0).any()


@pytest.mark.parametrize("V", [6, 16384, 16385, 50001])
def test_sample_vocab_sizes(V):
    """One entry, exactly one chunk, one entry past a chunk, several chunks with an odd tail
    (scalar loads), fp32 logits."""
    B, D, k = 8, 4, 3
    tree, _ = C.tree_from_logits(42, B, D, V, k, 12, std=2.0, boost=2.0)
    lens = np.random.default_rng(42).integers(0, D + 1, B)
    tl = _peaked_target(tree, V, 42, lens, boost=4.0, height=5.0, dtype=torch.float32)
    U = synth.uniforms(B, D + 1, k, g=synth.gen(42, 32))
    g = _gpu(tree, D, tl, U, 1.0)
    o = oracle.walk_sample(tree["token"], tree["parent"], tree["n_nodes"], D, C.f64(tl), U.double().numpy(), 1.0, k)
    _compare(tree, D, tl, U, 1.0, k, g, o, min_exact=0.5)


def test_sample_drafter_vocab_full_batch():
    """The batched round's shape: 32 requests, budget 64 from drafter logits of depth 15,
    V = 151936 bf16, peaked target with planted paths.  The GPU runs all 32 requests in one
    call; the oracle replays eight of them one request at a time."""
    B, D, V, k = 32, 15, 151936, 8
    tree, _ = C.tree_from_logits(5, B, D, V, k, 64)
    lens = np.random.default_rng(5).integers(0, 5, B)
    tl = _peaked_target(tree, V, 5, lens, boost=13.0)
    U = synth.uniforms(B, D + 1, k, g=synth.gen(5, 32))
    g = _gpu(tree, D, tl, U, 1.0)
    assert (g["status"] == 0).all()
    sample = [0, 3, 7, 12, 18, 22, 27, 31]
    exact = 0
    for b in sample:
        sub = {key: tree[key][b:b + 1] for key in ("token", "parent", "n_nodes")}
        o = oracle.walk_sample(sub["token"], sub["parent"], sub["n_nodes"], D, C.f64(tl[b:b + 1]),
                               U[b:b + 1].double().numpy(), 1.0, k)
        gb = {key: g[key][b:b + 1] for key in _KEYS}
        exact += _compare(sub, D, tl[b:b + 1], U[b:b + 1], 1.0, k, gb, o, min_exact=0.0)
    assert exact >= len(sample) // 2
    assert g["acc_len"].max() >= 2


def test_sample_cold_limit_equals_greedy_walk():
    """T = 1e-3 on logits with gaps of at least 0.1: the sampler takes the greedy walk."""
    B, D, V, k = 6, 6, 512, 4
    tree, _ = C.tree_from_logits(43, B, D, V, k, 30, std=2.0, boost=3.0)
    N = tree["token"].shape[1]
    rng = np.random.default_rng(43)
    tl = np.stack([[rng.permutation(V) * 0.1 for _ in range(N)] for _ in range(B)]).astype(np.float32)
    tl = torch.as_tensor(tl)
    lens = rng.integers(1, D + 1, B)
    synth.plant_path(tl, tree["token"], tree["parent"], tree["n_nodes"], lens, boost=60.0)
    U = synth.uniforms(B, D + 1, k, g=synth.gen(43, 32)) * 0.99
    g = _gpu(tree, D, tl, U, 1e-3)
    t = C.tree_to_dev(tree)
    gr = ddt.ddt_walk_accept(t["token"], t["parent"], t["n_nodes"], D, target_logits=tl.cuda())
    torch.cuda.synchronize()
    for key in ("acc_nodes", "acc_len", "bonus", "emitted", "n_emitted", "status"):
        np.testing.assert_array_equal(g[key], gr[key].cpu().numpy(), err_msg=key)
    assert g["acc_len"].max() > 0


def test_sample_max_accept_cut():
    """max_accept below the tree depth: the walk stops there and draws the bonus from the
    whole p of the last node (no child tried)."""
    B, D, V, k = 6, 8, 700, 2
    tree, _ = C.tree_from_logits(44, B, D, V, k, 20, std=2.0, boost=4.0)
    lens = np.full(B, D)
    tl = _peaked_target(tree, V, 44, lens, boost=30.0, height=5.0, dtype=torch.float32)
    A_cut = 2
    U = synth.uniforms(B, A_cut + 1, k, g=synth.gen(44, 32))
    g = _gpu(tree, A_cut, tl, U, 1.0)
    o = oracle.walk_sample(tree["token"], tree["parent"], tree["n_nodes"], A_cut, C.f64(tl), U.double().numpy(),
                           1.0, k)
    _compare(tree, A_cut, tl, U, 1.0, k, g, o, min_exact=0.5)
    assert (g["acc_len"] <= A_cut).all() and (g["acc_len"] == A_cut).any()


def test_sample_statuses():
    """Malformed trees and non-finite logits: the same status as the oracle, empty walks."""
    B, D, V, k = 6, 3, 64, 3
    tree, _ = C.tree_from_logits(45, B, D, V, k, 9, std=2.0, boost=2.0)
    tree = {key: np.array(val) for key, val in tree.items()}
    tl = synth.target_logits(B, tree["token"].shape[1], V, g=synth.gen(45, 30), dtype=torch.float32)
    N = tree["token"].shape[1]
    kids1 = [c for c in range(1, tree["n_nodes"][1]) if tree["parent"][1][c] == 0]
    assert len(kids1) >= 2
    tree["n_nodes"][5] = N - 2                               # the last rows (leaves) dropped
    tree["token"][1][kids1[1]] = tree["token"][1][kids1[0]]  # a token twice among siblings
    tree["token"][2][1] = V + 5                              # token outside the vocabulary
    tree["parent"][3][2] = 5                                  # a parent after its child
    tl[4, 1, 7] = float("nan")                                # non-finite logit in a tree row
    tl[5, tree["n_nodes"][5], 3] = float("inf")               # ... but past the tree: ignored
    U = synth.uniforms(B, D + 1, 2, g=synth.gen(45, 32))     # C = 2 < 3 children at the root
    g = _gpu(tree, D, tl, U, 1.0)
    o = oracle.walk_sample(tree["token"], tree["parent"], tree["n_nodes"], D, C.f64(tl), U.double().numpy(), 1.0, 2)
    np.testing.assert_array_equal(g["status"], o["status"])
    for b in range(B):
        if o["status"][b] != 0:
            assert g["n_emitted"][b] == 0 and g["bonus"][b] == -1 and (g["emitted"][b] == -1).all()
    assert (o["status"][1:5] != 0).all()
    U3 = synth.uniforms(B, D + 1, 3, g=synth.gen(45, 33))
    g3 = _gpu({key: tree[key] for key in tree}, D, tl, U3, 1.0)
    o3 = oracle.walk_sample(tree["token"], tree["parent"], tree["n_nodes"], D, C.f64(tl), U3.double().numpy(), 1.0, 3)
    np.testing.assert_array_equal(g3["status"], o3["status"])
    assert o3["status"][0] == 0 and o3["status"][5] == 0


def test_sample_bf16_nonfinite_in_packed_units():
    """Full 2048-entry bf16 units take their max and finiteness check on packed pairs:
    +inf, -inf and NaN in either half of a pair, in a full unit and in the ragged last
    unit, flag the request as the oracle does; a non-finite entry in a row past the tree
    and the largest finite bf16 do not."""
    B, D, V = 8, 3, 3 * 2048 + 613
    tree, _ = C.tree_from_logits(47, B, D, 300, 3, 8, std=2.0, boost=2.0)
    tree = {k: np.array(v) for k, v in tree.items()}
    N = tree["token"].shape[1]
    tree["n_nodes"][4] = N - 2                                  # the last rows (leaves) dropped
    tl = synth.target_logits(B, N, V, g=synth.gen(47, 30), dtype=torch.float32)
    tl[0, 0, 2 * 2048 + 10] = float("inf")                       # low half of a pair, full unit
    tl[1, 1, 2048 + 7] = float("-inf")                           # high half of a pair
    tl[2, 0, V - 3] = float("nan")                               # ragged last unit
    tl[3, 0, 1] = float("nan")                                   # first unit, high half
    tl[4, N - 1, 100] = float("inf")                             # a row past the tree: ignored
    tl[6, 2, 0] = float("-inf")                                  # the very first entry of a row
    tl[7, 1, 99] = 3.3895313892515355e38                         # the largest finite bf16
    tl = tl.to(torch.bfloat16)
    U = synth.uniforms(B, D + 1, 4, g=synth.gen(47, 32))
    g = _gpu(tree, D, tl, U, 1.0)
    o = oracle.walk_sample(tree["token"], tree["parent"], tree["n_nodes"], D, C.f64(tl), U.double().numpy(), 1.0, 4)
    np.testing.assert_array_equal(g["status"], o["status"])
    assert g["status"].tolist() == [6, 6, 6, 6, 0, 0, 6, 0]
    for b in range(B):
        if o["status"][b] != 0:
            assert g["n_emitted"][b] == 0 and g["bonus"][b] == -1 and (g["emitted"][b] == -1).all()


def test_sample_deterministic_and_graph_safe():
    """Same inputs, same outputs, call after call (no atomics decide anything)."""
    B, D, V, k = 16, 15, 151936, 8
    tree, _ = C.tree_from_logits(46, B, D, V, k, 64)
    lens = np.random.default_rng(46).integers(0, 4, B)
    tl = _peaked_target(tree, V, 46, lens, boost=13.0)
    U = synth.uniforms(B, D + 1, k, g=synth.gen(46, 32))
    first = _gpu(tree, D, tl, U, 0.8)
    for _ in range(3):
        again = _gpu(tree, D, tl, U, 0.8)
        for key in _KEYS:
            np.testing.assert_array_equal(first[key], again[key])


def test_sample_rejects_bad_arguments():
    tree, _ = C.tree_from_logits(47, 1, 3, 64, 2, 6, std=2.0, boost=2.0)
    t = C.tree_to_dev(tree)
    tl = torch.zeros((1, 7, 64), device="cuda")
    U = torch.zeros((1, 4, 3), device="cuda")
    for T in (0.0, -1.0, float("inf"), float("nan"), 1e-40):
        with pytest.raises(ddt.DDTError):
            ddt.ddt_walk_accept_sample(t["token"], t["parent"], t["n_nodes"], 3, target_logits=tl, uniforms=U,
                                       temperature=T)
