"""GPU parity of ddt_walk_accept and ddt_commit against the oracle (bit-exact indices,
normwise <= 2e-3 for the committed GDN state)."""
import numpy as np
import pytest
import torch

import oracle
from tests import _cases as C
from tests._parity import TOL, normwise
from tree_speculative_decoding_02_gb300 import ddt, synth

pytestmark = pytest.mark.gpu

_WALK_KEYS = ("acc_nodes", "acc_len", "bonus", "emitted", "n_emitted")


def _planted_logits(tree, V, workload, dtype, lens):
    B, N = tree["token"].shape
    tl = synth.target_logits(B, N, V, g=synth.gen(workload, 30), dtype=torch.float32)
    synth.plant_path(tl, tree["token"], tree["parent"], tree["n_nodes"], lens, boost=8.0)
    return tl.to(dtype)


def _walk_gpu(tree, D, tl=None, targ=None):
    t = C.tree_to_dev(tree)
    r = ddt.ddt_walk_accept(t["token"], t["parent"], t["n_nodes"], D,
                            target_logits=None if tl is None else tl.cuda(),
                            target_argmax=None if targ is None else torch.as_tensor(targ, dtype=torch.int32).cuda())
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in r.items()}


def _check_walk(g, o, tree):
    for k in _WALK_KEYS:
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)
    for b in range(tree["token"].shape[0]):
        n = tree["n_nodes"][b]
        np.testing.assert_array_equal(g["target_argmax"][b][:n], o["target_argmax"][b][:n])
    assert (g["status"] == 0).all()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_walk_tiny_and_drafter_vocab(dtype):
    for (B, D, V, budget, wl) in [(1, 8, 1024, 16, 1), (3, 15, 151936, 64, 2)]:
        tree, _ = C.tree_from_logits(wl, B, D, V, 8, budget)
        lens = np.random.default_rng(wl).integers(0, D + 1, B)
        tl = _planted_logits(tree, V, wl, dtype, lens)
        g = _walk_gpu(tree, D, tl=tl)
        o = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], D, target_logits=C.f64(tl))
        _check_walk(g, o, tree)
        assert g["acc_len"].max() > 0


def test_walk_argmax_input_and_ties():
    tree, _ = C.tree_from_logits(2, 2, 6, 40, 3, 20, std=2.0, boost=0.0)
    rng = np.random.default_rng(3)
    tl = torch.as_tensor(rng.integers(0, 3, size=(2, 21, 40)).astype(np.float32))  # many argmax ties
    g = _walk_gpu(tree, 6, tl=tl)
    o = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], 6, target_logits=C.f64(tl))
    _check_walk(g, o, tree)
    g2 = _walk_gpu(tree, 6, targ=o["target_argmax"])
    for k in _WALK_KEYS:
        np.testing.assert_array_equal(g2[k], o[k])


def test_flat_walk_matches_oracle():
    """Safe mode: only first (rank-0) children are taken.  Targets agree with a random child
    (often not the first) at 70 % of the rows, so the flat and the ordinary walks differ."""
    tree, _ = C.tree_from_logits(2, 4, 8, 3000, 4, 64)
    rng = np.random.default_rng(9)
    N = tree["token"].shape[1]
    targ = np.full((4, N), 5, np.int32)
    for b in range(4):
        for i in range(int(tree["n_nodes"][b])):
            kids = [c for c in range(1, int(tree["n_nodes"][b])) if tree["parent"][b][c] == i]
            if kids and rng.random() < 0.7:
                targ[b, i] = tree["token"][b][kids[0] if rng.random() < 0.6 else kids[-1]]
    t = C.tree_to_dev(tree)
    r = ddt.ddt_walk_accept(t["token"], t["parent"], t["n_nodes"], 8,
                            target_argmax=torch.as_tensor(targ).cuda(), flat=True)
    torch.cuda.synchronize()
    o = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], 8, target_argmax=targ, flat=True)
    for k in _WALK_KEYS:
        np.testing.assert_array_equal(r[k].cpu().numpy(), o[k], err_msg=k)
    full = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], 8, target_argmax=targ)
    assert (o["acc_len"] <= full["acc_len"]).all() and (o["acc_len"] < full["acc_len"]).any()
    # with target logits: planted along the first-child spine, flat and ordinary agree
    tl = _planted_logits(tree, 3000, 2, torch.bfloat16, np.array([8, 3, 0, 5]))
    g = _walk_gpu(tree, 8, tl=tl)
    r2 = ddt.ddt_walk_accept(t["token"], t["parent"], t["n_nodes"], 8, target_logits=tl.cuda(), flat=True)
    torch.cuda.synchronize()
    for k in _WALK_KEYS:
        np.testing.assert_array_equal(r2[k].cpu().numpy(), g[k], err_msg=k)


def test_walk_nonfinite_flagged():
    tree, _ = C.tree_from_logits(2, 2, 4, 40, 2, 6, std=2.0, boost=0.0)
    tl = torch.randn(2, 7, 40)
    tl[0, 0, 3] = float("inf")
    g = _walk_gpu(tree, 4, tl=tl)
    assert g["status"].tolist() == [6, 0]


def test_walk_bf16_nonfinite_in_packed_rows():
    """bf16 rows take the packed argmax (two entries a step, and the exponent field's max for
    the finiteness check): +inf, -inf and NaN in either half of a packed pair, in a full
    16384-entry chunk and in the ragged last chunk, flag the request; a non-finite entry
    in a row past the tree and the largest finite bf16 do not, and the clean requests walk
    as the oracle does."""
    B, D, V = 8, 3, 16384 + 6181
    tree, _ = C.tree_from_logits(46, B, D, 300, 3, 8, std=2.0, boost=2.0)
    tree = {k: np.array(v) for k, v in tree.items()}
    N = tree["token"].shape[1]
    tree["n_nodes"][4] = N - 2                                  # the last rows (leaves) dropped
    tl = synth.target_logits(B, N, V, g=synth.gen(46, 30), dtype=torch.float32)
    tl[0, 0, 1234] = float("inf")                                # low half of a pair, full chunk
    tl[1, 1, 4321] = float("-inf")                               # high half of a pair
    tl[2, 0, V - 5] = float("nan")                               # ragged last chunk
    tl[3, 2, 16383] = float("nan")                               # last entry of the first chunk
    tl[4, N - 1, 100] = float("inf")                             # a row past the tree: ignored
    tl[6, 0, 0] = float("-inf")                                  # the very first entry
    tl[7, 1, 777] = 3.3895313892515355e38                        # the largest finite bf16
    tl = tl.to(torch.bfloat16)
    assert float(tl[7, 1, 777]) == 3.3895313892515355e38
    g = _walk_gpu(tree, D, tl=tl)
    assert g["status"].tolist() == [6, 6, 6, 6, 0, 0, 6, 0]
    clean = [4, 5, 7]
    sub = {k: v[clean] for k, v in tree.items()}
    o = oracle.walk(sub["token"], sub["parent"], sub["n_nodes"], D, target_logits=C.f64(tl[clean]))
    for k in _WALK_KEYS:
        np.testing.assert_array_equal(g[k][clean], o[k], err_msg=k)
    assert g["target_argmax"][7][1] == 777


def _commit_case(La, Lg, B, budget, D, wl, Pcap_extra=8, dtype=torch.bfloat16, dims=(32, 32, 1, 2)):
    dk, dv, Hk, Hv = dims
    tree, _ = C.tree_from_logits(wl, B, D, 200, 3, budget, std=2.0, boost=0.0)
    N = budget + 1
    lens = np.random.default_rng(wl + 1).integers(1, D + 1, B)
    tl = _planted_logits(tree, 200, wl, torch.float32, lens)
    wk = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], D, target_logits=C.f64(tl))
    pl = np.random.default_rng(wl).integers(0, 50, B).astype(np.int32)
    Pcap = int(pl.max()) + D + 1 + Pcap_extra
    ai = synth.attn_inputs(La, B, N, 4, 2, 64, Pcap, pl, workload=wl, dtype=dtype, poison=False)
    gi = synth.gdn_inputs(Lg, B, N, Hk, Hv, dk, dv, 4, workload=wl, dtype=dtype)
    return tree, wk, pl, Pcap, ai, gi


def _commit_gpu(wk, pl, ai, gi, Hk):
    kc, vc = ai.k_cache.cuda(), ai.v_cache.cuda()
    S = gi.S.transpose(-1, -2).contiguous().cuda()
    cs = gi.conv_state.cuda()
    pld = torch.as_tensor(pl).cuda()
    r = ddt.ddt_commit(torch.as_tensor(wk["acc_nodes"]).cuda(), torch.as_tensor(wk["acc_len"]).cuda(), pld,
                       k_tree=ai.k_tree.cuda(), v_tree=ai.v_tree.cuda(), k_cache=kc, v_cache=vc, x=gi.x.cuda(),
                       conv_w=gi.conv_w.cuda(), beta=gi.beta.cuda(), decay=gi.decay.cuda(), S=S, conv_state=cs, Hk=Hk)
    torch.cuda.synchronize()
    return r, kc, vc, S, cs, pld


def _oracle_commit(wk, pl, ai, gi, Hk):
    return oracle.commit(wk["acc_nodes"], wk["acc_len"], pl, k_tree=C.f64(ai.k_tree), v_tree=C.f64(ai.v_tree),
                         k_cache=C.f64(ai.k_cache), v_cache=C.f64(ai.v_cache), x=C.f64(gi.x),
                         conv_w=C.f64(gi.conv_w), beta=C.f64(gi.beta), decay=C.f64(gi.decay), S=C.f64(gi.S),
                         conv_state=C.f64(gi.conv_state), Hk=Hk)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_commit_kv_gdn_conv(dtype):
    tree, wk, pl, Pcap, ai, gi = _commit_case(2, 2, 3, 24, 6, 11, dtype=dtype)
    r, kc, vc, S, cs, pld = _commit_gpu(wk, pl, ai, gi, 1)
    o = _oracle_commit(wk, pl, ai, gi, 1)
    assert r["status"].cpu().tolist() == o["status"].tolist() == [0, 0, 0]
    np.testing.assert_array_equal(pld.cpu().numpy(), o["prefix_len"])
    np.testing.assert_array_equal(r["src_row"].cpu().numpy(), o["src_row"])
    np.testing.assert_array_equal(r["dst_pos"].cpu().numpy(), o["dst_pos"])
    np.testing.assert_array_equal(C.f64(kc), o["k_cache"])
    np.testing.assert_array_equal(C.f64(vc), o["v_cache"])
    np.testing.assert_array_equal(C.f64(cs), o["conv_state"])
    err = normwise(C.s_to_oracle(S), o["S"], axes=(-2, -1))
    assert err.max() <= TOL, err.max()


def test_commit_capacity_refused():
    tree, wk, pl, Pcap, ai, gi = _commit_case(1, 1, 2, 10, 4, 12, Pcap_extra=0)
    wk["acc_len"][1] = 0
    wk["acc_nodes"][1][1:] = -1
    pl[0] = Pcap - int(wk["acc_len"][0])  # root + accepted rows no longer fit
    r, kc, vc, S, cs, pld = _commit_gpu(wk, pl, ai, gi, 1)
    o = _oracle_commit(wk, pl, ai, gi, 1)
    assert r["status"].cpu().tolist() == o["status"].tolist() == [3, 0]
    np.testing.assert_array_equal(pld.cpu().numpy(), o["prefix_len"])
    np.testing.assert_array_equal(C.f64(kc), o["k_cache"])
    err = normwise(C.s_to_oracle(S), o["S"], axes=(-2, -1))
    assert err.max() <= TOL


def test_commit_gdn_workload_forced_path():
    """48 GDN layers, Hk=16, Hv=48, dk=dv=128: commit of a seeded root-to-leaf path; every
    (layer, value head) state and every layer's conv state against the oracle."""
    tree, _ = C.tree_from_logits(4, 1, 15, 151936, 8, 64)
    rng = np.random.default_rng(4)
    path = [0]
    while True:
        kids = [c for c in range(1, tree["n_nodes"][0]) if tree["parent"][0][c] == path[-1]]
        if not kids:
            break
        path.append(kids[int(rng.integers(len(kids)))])
    A = 16
    acc = np.full((1, A), -1, np.int32)
    acc[0, :len(path)] = path
    al = np.array([len(path) - 1], np.int32)
    gi = synth.gdn_inputs(48, 1, 65, 16, 48, 128, 128, 4, workload=4, dtype=torch.bfloat16)
    S = gi.S.transpose(-1, -2).contiguous().cuda()
    cs = gi.conv_state.cuda()
    pld = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = ddt.ddt_commit(torch.as_tensor(acc).cuda(), torch.as_tensor(al).cuda(), pld, x=gi.x.cuda(),
                       conv_w=gi.conv_w.cuda(), beta=gi.beta.cuda(), decay=gi.decay.cuda(), S=S, conv_state=cs,
                       Hk=16)
    torch.cuda.synchronize()
    assert int(r["status"][0]) == 0 and int(pld[0]) == len(path)
    o = oracle.commit(acc, al, [0], x=C.f64(gi.x), conv_w=C.f64(gi.conv_w), beta=C.f64(gi.beta),
                      decay=C.f64(gi.decay), S=C.f64(gi.S), conv_state=C.f64(gi.conv_state), Hk=16)
    err = normwise(C.s_to_oracle(S), o["S"], axes=(-2, -1))
    assert err.max() <= TOL, err.max()
    np.testing.assert_array_equal(C.f64(cs), o["conv_state"])
