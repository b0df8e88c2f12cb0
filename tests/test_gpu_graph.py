"""A whole verification round captures into one CUDA graph: the library launches only
stream-ordered kernels (no allocation, no host synchronisation), so replaying the graph
gives bit-identical trees, outputs, accepted paths and committed state to eager calls."""
import pytest
import torch

from tree_speculative_decoding_02_gb300 import ddt, synth
from tree_speculative_decoding_02_gb300.round import Round

pytestmark = pytest.mark.gpu

# a small batched round with the production head shapes (2 attention + 2 GDN layers)
CFG = dict(synth.WORKLOADS[5], name="graph-round", B=3, P_lo=100, P_hi=3000, Lf=2, Lg=2)


def _outputs(r):
    out = {k: v.clone() for k, v in r.tree.items()}
    out.update({"walk_" + k: v.clone() for k, v in r.walk.items()})
    out.update({"commit_" + k: v.clone() for k, v in r.commit.items()})
    out.update(attn_o=r.attn_o.clone(), gdn_o=r.gdn_o.clone(), prefix_len=r.prefix_len.clone(),
               S=r.gdn.S.clone(), conv_state=r.gdn.conv_state.clone(), k_cache=r.attn.k_cache.clone(),
               v_cache=r.attn.v_cache.clone())
    return out


def test_round_replays_from_a_cuda_graph_bit_exact():
    r = Round(CFG, device="cuda", workload=5)
    state0 = {"S": r.gdn.S.clone(), "cs": r.gdn.conv_state.clone(), "k": r.attn.k_cache.clone(),
              "v": r.attn.v_cache.clone()}

    def restore():
        r.gdn.S.copy_(state0["S"])
        r.gdn.conv_state.copy_(state0["cs"])
        r.attn.k_cache.copy_(state0["k"])
        r.attn.v_cache.copy_(state0["v"])
        r.restore_prefix()

    restore()
    r.step()
    torch.cuda.synchronize()
    eager = _outputs(r)
    assert (r.tree["status"] == 0).all() and (r.commit["status"] == 0).all()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            restore()
            r.step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    launches = ddt.ddt_launch_count()
    with torch.cuda.graph(g):
        r.restore_prefix()
        r.step()
    assert ddt.ddt_launch_count() - launches >= 9   # the round's kernels went into the graph
    for _ in range(2):
        restore()
        g.replay()
        torch.cuda.synchronize()
        got = _outputs(r)
        for k, v in eager.items():
            assert torch.equal(got[k], v) or (v.is_floating_point() and torch.equal(got[k].nan_to_num(7.0),
                                                                                   v.nan_to_num(7.0))), k


@pytest.mark.parametrize("temperature", [0.0, 0.8])
def test_graph_round_matches_oracle(temperature):
    """The graph-replayed round against the oracle, every output of the small round: the
    trees, all attention rows and GDN units (fp32 outputs, <= 2e-3 normwise), the walk
    (greedy; or rejection sampling with the round's uniforms, exact where the oracle's
    margin allows), and the commit (KV rows bit-exact, states <= 2e-3)."""
    import math

    import numpy as np

    import oracle
    from tests import _cases as C
    from tests._parity import TOL, assert_tree_equal, normwise

    cfg = dict(CFG, temperature=temperature)
    r = Round(cfg, device="cuda", workload=5, attn_out_dtype=torch.float32, gdn_out_dtype=torch.float32)
    B, D, k = cfg["B"], cfg["D"], cfg["top_k"]
    # the tree is a function of the drafter logits: build it once to plant acceptances
    ddt.ddt_build_tree(r.draft_logits, r.root_token, r.prefix_len, k, cfg["budget"], out=r.tree, workspace=r.build_ws)
    torch.cuda.synchronize()
    tok, par = r.tree["token"].cpu().numpy(), r.tree["parent"].cpu().numpy()
    nn = r.tree["n_nodes"].cpu().numpy()
    tl = r.target_logits.float().cpu()
    if temperature > 0:                # a peaked target, so that most draws have a margin
        synth.add_peaks(tl, 3, 12.0, g=synth.gen(5, 31))
    synth.plant_path(tl, tok, par, nn, [2, 1, 3], boost=14.0)
    r.target_logits.copy_(tl.to(r.target_logits.dtype))
    kc0, vc0 = C.f64(r.attn.k_cache), C.f64(r.attn.v_cache)
    S0, cs0 = C.s_to_oracle(r.gdn.S), C.f64(r.gdn.conv_state)
    P0 = r.prefix0.cpu().numpy()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        r.restore_prefix()
        r.walk_step()                 # warm the walk's own allocations outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        r.restore_prefix()
        r.step()
    g.replay()                         # the capture itself ran nothing: this is the round
    torch.cuda.synchronize()
    for st in (r.tree["status"], r.attn_status, r.gdn_status, r.commit["status"]):
        assert (st == 0).all()

    orc = oracle.build_tree(C.f64(r.draft_logits), r.root_token.cpu().numpy(), P0, k, cfg["budget"])
    gpu = {key: v.cpu().numpy() for key, v in r.tree.items()}
    for b in range(B):
        assert_tree_equal(gpu, orc, b)

    a = r.attn
    want = oracle.tree_attn(C.f64(a.q), C.f64(a.k_tree), C.f64(a.v_tree), np.nan_to_num(kc0), np.nan_to_num(vc0), P0,
                            nn, gpu["anc"].view(np.uint32), 1.0 / math.sqrt(cfg["d"]))["o"]
    got = C.f64(r.attn_o)
    for b in range(B):
        assert normwise(got[:, b, :nn[b]], want[:, b, :nn[b]], axes=-1).max() <= TOL

    gi = r.gdn
    want = oracle.tree_gdn(C.f64(gi.x), C.f64(gi.conv_w), cs0, C.f64(gi.beta), C.f64(gi.decay), S0, par, nn,
                           cfg["Hk"])["o"]
    got = C.f64(r.gdn_o)
    for b in range(B):
        assert normwise(got[:, b, :nn[b]], want[:, b, :nn[b]], axes=-1).max() <= TOL

    if temperature > 0:
        from tests.test_gpu_walk_sample import _KEYS, _replay_ok

        U = r.uniforms.double().cpu().numpy()
        wk = oracle.walk_sample(tok, par, nn, D, C.f64(r.target_logits), U, temperature, k)
        exact = wk["margin"] >= 1e-5
        assert exact.sum() >= 1
        gw = {key: v.cpu().numpy() for key, v in r.walk.items()}
        for b in np.flatnonzero(~exact):
            _replay_ok(tok[b], par[b], int(nn[b]), C.f64(r.target_logits)[b], U[b], temperature, k,
                       {key: gw[key][b] for key in _KEYS})
    else:
        wk = oracle.walk(tok, par, nn, D, target_logits=C.f64(r.target_logits))
        exact = np.ones(B, bool)
    for key in ("acc_nodes", "acc_len", "bonus", "emitted", "n_emitted"):
        np.testing.assert_array_equal(r.walk[key].cpu().numpy()[exact], wk[key][exact], err_msg=key)
    acc_nodes, acc_len = r.walk["acc_nodes"].cpu().numpy(), r.walk["acc_len"].cpu().numpy()
    assert acc_len.max() >= 1

    com = oracle.commit(acc_nodes, acc_len, P0, k_tree=C.f64(a.k_tree), v_tree=C.f64(a.v_tree), k_cache=kc0,
                        v_cache=vc0, x=C.f64(gi.x), conv_w=C.f64(gi.conv_w), beta=C.f64(gi.beta),
                        decay=C.f64(gi.decay), S=S0, conv_state=cs0, Hk=cfg["Hk"])
    np.testing.assert_array_equal(r.prefix_len.cpu().numpy(), com["prefix_len"])
    for b in range(B):
        rows = slice(int(P0[b]), int(P0[b] + acc_len[b] + 1))
        np.testing.assert_array_equal(C.f64(a.k_cache)[:, b, :, rows], com["k_cache"][:, b, :, rows])
        np.testing.assert_array_equal(C.f64(a.v_cache)[:, b, :, rows], com["v_cache"][:, b, :, rows])
    assert normwise(C.s_to_oracle(gi.S), com["S"], axes=(-2, -1)).max() <= TOL
    np.testing.assert_array_equal(C.f64(gi.conv_state), com["conv_state"])
