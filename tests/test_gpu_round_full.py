"""One full batched round (32 requests, drafter depth 15, vocabulary 151936, budget 64,
prefixes ~ U[1024, 32768], 16 attention + 48 GDN layers, bf16) in the configuration the
bench times, with planted acceptances, checked on samples the oracle can compute one by
one: every request's tree and walk, sampled attention rows and GDN units, and the commit
of sampled KV rows, GDN states and conv states.  Run twice: with fp32 attention and GDN
outputs (parity mode, within 2e-3), and with the bf16 outputs the bench times (within
2e-3 plus one bf16 rounding, 2^-8 of the vector's largest entry)."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import _cases as C
from tests._parity import TOL, assert_tree_equal, normwise
from tree_speculative_decoding_02_gb300 import ddt, synth
from tree_speculative_decoding_02_gb300.round import Round

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["fp32_out", "bf16_out"])
def test_full_batched_round_sampled(out_dtype):
    cfg = dict(synth.WORKLOADS[5])
    r = Round(cfg, device="cuda", workload=5, attn_out_dtype=out_dtype, gdn_out_dtype=out_dtype)
    tol = TOL if out_dtype == torch.float32 else TOL + 2.0 ** -8
    B, N, D = cfg["B"], r.N, cfg["D"]
    rng = np.random.default_rng(55)

    # the tree is a function of the drafter logits: build it once to plant acceptances
    ddt.ddt_build_tree(r.draft_logits, r.root_token, r.prefix_len, cfg["top_k"], cfg["budget"], out=r.tree,
                       workspace=r.build_ws)
    torch.cuda.synchronize()
    tok, par = r.tree["token"].cpu().numpy(), r.tree["parent"].cpu().numpy()
    nn = r.tree["n_nodes"].cpu().numpy()
    lens = rng.integers(0, D + 1, B)
    synth.plant_path(r.target_logits, tok, par, nn, lens)

    # pre-commit copies of what the commit rewrites, for the sampled units
    gdn_units = [(0, 0, 0), (47, 31, 47), (13, 7, 20), (30, 19, 2), (5, 26, 33)]
    S0 = {u: C.f64(r.gdn.S[u[0], u[1]]).swapaxes(-1, -2).copy() for u in gdn_units}     # [Hv][dk][dv]
    cs0 = {u: C.f64(r.gdn.conv_state[u[0], u[1]]) for u in gdn_units}
    P0 = r.prefix0.cpu().numpy()

    r.restore_prefix()
    r.step()
    torch.cuda.synchronize()
    assert (r.tree["status"] == 0).all() and (r.attn_status == 0).all() and (r.gdn_status == 0).all()
    assert (r.walk["status"] == 0).all() and (r.commit["status"] == 0).all()

    # build: every request
    orc = oracle.build_tree(C.f64(r.draft_logits), r.root_token.cpu().numpy(), P0, cfg["top_k"], cfg["budget"])
    gpu = {k: v.cpu().numpy() for k, v in r.tree.items()}
    for b in range(B):
        assert_tree_equal(gpu, orc, b)

    # walk: every request, against the planted target logits
    wk = oracle.walk(tok, par, nn, D, target_logits=C.f64(r.target_logits))
    for k in ("acc_nodes", "acc_len", "bonus", "emitted", "n_emitted"):
        np.testing.assert_array_equal(r.walk[k].cpu().numpy(), wk[k], err_msg=k)
    assert wk["acc_len"].max() >= 2          # the trees of this workload are at most 3 deep

    # attention: sampled (layer, request, row, query head)
    a, G, scale = r.attn, cfg["Hq"] // cfg["Hkv"], 1.0 / math.sqrt(cfg["d"])
    anc = gpu["anc"].view(np.uint32)
    for _ in range(12):
        l, b = int(rng.integers(cfg["Lf"])), int(rng.integers(B))
        row, hq = int(rng.integers(nn[b])), int(rng.integers(cfg["Hq"]))
        g, P, n = hq // G, int(P0[b]), int(nn[b])
        want = oracle.attn_row(C.f64(a.q[l, b, row, hq]), C.f64(a.k_cache[l, b, g, :P]), C.f64(a.v_cache[l, b, g, :P]),
                               C.f64(a.k_tree[l, b, :n, g]), C.f64(a.v_tree[l, b, :n, g]), anc[b, row], n, scale)
        err = normwise(C.f64(r.attn_o[l, b, row, hq]), want, axes=-1)
        assert err <= tol, (l, b, row, hq, err)

    # GDN: sampled (layer, request, value head), every node
    gi = r.gdn
    for (l, b, h) in gdn_units:
        n = int(nn[b])
        u = oracle.gdn_unit(C.f64(gi.x[l, b]), C.f64(gi.conv_w[l]), cs0[(l, b, h)], C.f64(gi.beta[l, b]),
                            C.f64(gi.decay[l, b]), S0[(l, b, h)][h], par[b], n, cfg["Hk"], cfg["Hv"], h)
        err = normwise(C.f64(r.gdn_o[l, b, :n, h]), u["o"][:n], axes=-1)
        assert err.max() <= tol, (l, b, h, err.max())

    # commit: KV rows land at prefix_len + j; the state and conv state follow the path
    src = r.commit["src_row"].cpu().numpy()
    dst = r.commit["dst_pos"].cpu().numpy()
    np.testing.assert_array_equal(r.prefix_len.cpu().numpy(), P0 + wk["acc_len"] + 1)
    for b in (0, 9, 31):
        for j in range(int(wk["acc_len"][b]) + 1):
            assert src[b, j] == wk["acc_nodes"][b, j] and dst[b, j] == P0[b] + j
            for l in (0, 15):
                assert torch.equal(a.k_cache[l, b, :, P0[b] + j], a.k_tree[l, b, src[b, j]])
                assert torch.equal(a.v_cache[l, b, :, P0[b] + j], a.v_tree[l, b, src[b, j]])
    for (l, b, h) in gdn_units:
        o = oracle.commit(wk["acc_nodes"][b:b + 1], wk["acc_len"][b:b + 1], [0], x=C.f64(gi.x[l:l + 1, b:b + 1]),
                          conv_w=C.f64(gi.conv_w[l:l + 1]), beta=C.f64(gi.beta[l:l + 1, b:b + 1]),
                          decay=C.f64(gi.decay[l:l + 1, b:b + 1]), S=S0[(l, b, h)][None, None],
                          conv_state=cs0[(l, b, h)][None, None], Hk=cfg["Hk"])
        err = normwise(C.f64(gi.S[l, b, h]).T, o["S"][0, 0, h], axes=(-2, -1))
        assert err <= TOL, (l, b, h, err)
        np.testing.assert_array_equal(C.f64(gi.conv_state[l, b]), o["conv_state"][0, 0])
