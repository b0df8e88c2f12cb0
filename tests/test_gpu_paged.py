"""GPU parity of the paged-KV calls (ddt_tree_attn_paged, ddt_commit_paged) against the
oracle on the gathered contiguous cache.  Every page row that is not a prefix row holds
NaN, so any read past a request's prefix, or of a page it does not own, shows up."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import _cases as C
from tests._parity import TOL, normwise
from tree_speculative_decoding_02_gb300 import ddt, synth

pytestmark = pytest.mark.gpu


def _paged(workload, L, B, N, Hq, Hkv, d, prefix, page, extra_rows=0):
    """q / tree K,V ~ N(0,1) bf16; a shuffled block table over B * max_pages + 3 pages;
    page rows outside the prefixes are NaN."""
    P = np.asarray(prefix, np.int32)
    max_pages = max(1, -(-(int(P.max()) + extra_rows) // page))
    num_pages = B * max_pages + 3
    g = synth.gen(workload, 40)
    bf = torch.bfloat16
    q = synth.normal((L, B, N, Hq, d), g=g, dtype=bf)
    k_tree = synth.normal((L, B, N, Hkv, d), g=g, dtype=bf)
    v_tree = synth.normal((L, B, N, Hkv, d), g=g, dtype=bf)
    k_pages = synth.normal((L, num_pages, Hkv, page, d), g=g, dtype=bf)
    v_pages = synth.normal((L, num_pages, Hkv, page, d), g=g, dtype=bf)
    table = torch.randperm(num_pages, generator=g)[:B * max_pages].reshape(B, max_pages).to(torch.int32)
    live = torch.zeros((num_pages, page), dtype=torch.bool)
    for b in range(B):
        for p in range(int(P[b])):
            live[int(table[b, p // page]), p % page] = True
    dead = ~live[None, :, None, :, None].expand(L, num_pages, Hkv, page, d)
    k_pages[dead] = float("nan")
    v_pages[dead] = float("nan")
    return dict(q=q, k_tree=k_tree, v_tree=v_tree, k_pages=k_pages, v_pages=v_pages, table=table, P=P,
                Pcap=max_pages * page)


def _gpu_attn(c, tree, out_dtype=torch.float32):
    t = C.tree_to_dev(tree)
    r = ddt.ddt_tree_attn_paged(c["q"].cuda(), c["k_tree"].cuda(), c["v_tree"].cuda(), c["k_pages"].cuda(),
                                c["v_pages"].cuda(), c["table"].cuda(), torch.as_tensor(c["P"]).cuda(), t["n_nodes"],
                                t["anc"], scale=1.0 / math.sqrt(c["q"].shape[-1]), out_dtype=out_dtype)
    torch.cuda.synchronize()
    return r


def _oracle_attn(c, tree, d):
    kc = oracle.gather_pages(C.f64(c["k_pages"]), c["table"].numpy(), c["P"], c["Pcap"])
    vc = oracle.gather_pages(C.f64(c["v_pages"]), c["table"].numpy(), c["P"], c["Pcap"])
    return oracle.tree_attn(C.f64(c["q"]), C.f64(c["k_tree"]), C.f64(c["v_tree"]), kc, vc, c["P"],
                            tree["n_nodes"], tree["anc"], 1 / math.sqrt(d))["o"]


def _check(got, want, tree):
    got = got.cpu().double().numpy()
    assert np.isfinite(got).all()
    for b in range(got.shape[1]):
        n = int(tree["n_nodes"][b])
        err = normwise(got[:, b, :n], want[:, b, :n], axes=-1)
        assert err.max() <= TOL, f"request {b}: max normwise error {err.max():.3g}"
        assert (got[:, b, n:] == 0).all()


@pytest.mark.parametrize("page,d", [(16, 128), (64, 256), (128, 64), (8, 256), (256, 128)])
def test_paged_attn_matches_oracle(page, d):
    """GQA group 6, prefixes 0, 1, a page edge, and ragged lengths over several pages."""
    prefix = [0, 1, page, 3 * page + 5, 700]
    tree, _ = C.tree_from_logits(3, len(prefix), 6, 300, 4, 40, std=2.0, boost=0.0, prefix=prefix)
    c = _paged(3, 2, len(prefix), 41, 24, 4, d, prefix, page)
    r = _gpu_attn(c, tree)
    _check(r["o"], _oracle_attn(c, tree, d), tree)
    assert (r["status"].cpu() == 0).all()


def test_paged_attn_long_prefix_split():
    """One request with a long prefix (split-KV partials) through 64-row pages."""
    prefix = [9000]
    tree, _ = C.tree_from_logits(3, 1, 15, 3000, 8, 64, prefix=prefix)
    c = _paged(5, 1, 1, 65, 24, 4, 256, prefix, 64)
    r = _gpu_attn(c, tree)
    _check(r["o"], _oracle_attn(c, tree, 256), tree)


def test_paged_attn_bad_block_table_flagged():
    prefix = [100, 100]
    tree, _ = C.tree_from_logits(3, 2, 6, 300, 4, 8, std=2.0, boost=0.0, prefix=prefix)
    c = _paged(3, 1, 2, 9, 4, 1, 64, prefix, 32)
    c["table"][1, 2] = 10 ** 6        # a page the request's prefix needs does not exist
    r = _gpu_attn(c, tree)
    assert r["status"].cpu().tolist() == [0, 1]
    assert (r["o"][:, 1] == 0).all()
    _check(r["o"][:, :1], _oracle_attn({**c, "table": c["table"][:1], "P": c["P"][:1],
                                        **{k: c[k][:, :1] for k in ("q", "k_tree", "v_tree")}},
                                       {k: v[:1] for k, v in tree.items()}, 64), {k: v[:1] for k, v in tree.items()})


@pytest.mark.parametrize("page", [16, 64])
def test_paged_commit_matches_oracle(page):
    """Accepted rows land at prefix_len + j through the block table; rows of other pages
    and past the new prefix keep their contents."""
    prefix = [0, page - 2, 2 * page + 3]
    B, N, A = 3, 25, 7
    tree, _ = C.tree_from_logits(4, B, 6, 300, 3, N - 1, std=2.0, boost=0.0, prefix=prefix)
    c = _paged(4, 2, B, N, 8, 2, 64, prefix, page, extra_rows=A)
    acc = np.full((B, A), -1, np.int32)
    al = np.zeros(B, np.int32)
    for b in range(B):                 # a root-to-leaf path, first child each step
        path = [0]
        while len(path) < A:
            kids = [x for x in range(1, int(tree["n_nodes"][b])) if tree["parent"][b][x] == path[-1]]
            if not kids:
                break
            path.append(kids[0])
        acc[b, :len(path)] = path
        al[b] = len(path) - 1
    kp, vp = c["k_pages"].cuda(), c["v_pages"].cuda()
    pl = torch.as_tensor(c["P"]).cuda()
    r = ddt.ddt_commit_paged(torch.as_tensor(acc).cuda(), torch.as_tensor(al).cuda(), pl, c["table"].cuda(),
                             k_tree=c["k_tree"].cuda(), v_tree=c["v_tree"].cuda(), k_pages=kp, v_pages=vp)
    torch.cuda.synchronize()
    kc = oracle.gather_pages(C.f64(c["k_pages"]), c["table"].numpy(), c["P"], c["Pcap"])
    vc = oracle.gather_pages(C.f64(c["v_pages"]), c["table"].numpy(), c["P"], c["Pcap"])
    o = oracle.commit(acc, al, c["P"], k_tree=C.f64(c["k_tree"]), v_tree=C.f64(c["v_tree"]), k_cache=kc, v_cache=vc)
    assert r["status"].cpu().tolist() == o["status"].tolist() == [0, 0, 0]
    np.testing.assert_array_equal(pl.cpu().numpy(), o["prefix_len"])
    np.testing.assert_array_equal(r["dst_pos"].cpu().numpy(), o["dst_pos"])
    got_k = oracle.gather_pages(np.nan_to_num(C.f64(kp), nan=0.0), c["table"].numpy(), o["prefix_len"], c["Pcap"])
    got_v = oracle.gather_pages(np.nan_to_num(C.f64(vp), nan=0.0), c["table"].numpy(), o["prefix_len"], c["Pcap"])
    np.testing.assert_array_equal(got_k, o["k_cache"])
    np.testing.assert_array_equal(got_v, o["v_cache"])
    # the three spare pages were never written
    used = set(c["table"].flatten().tolist())
    spare = [p for p in range(kp.shape[1]) if p not in used]
    assert torch.isnan(kp[:, spare].float()).all()


def test_paged_commit_bad_page_refused():
    prefix = [5, 5]
    B, N, A = 2, 9, 3
    tree, _ = C.tree_from_logits(4, B, 6, 300, 3, N - 1, std=2.0, boost=0.0, prefix=prefix)
    c = _paged(4, 1, B, N, 4, 1, 64, prefix, 8, extra_rows=A)
    c["table"][1, 0] = -1
    acc = np.array([[0, -1, -1], [0, -1, -1]], np.int32)
    pl = torch.as_tensor(c["P"]).cuda()
    kp = c["k_pages"].cuda()
    before = kp.clone()
    r = ddt.ddt_commit_paged(torch.as_tensor(acc).cuda(), torch.zeros(B, dtype=torch.int32, device="cuda"), pl,
                             c["table"].cuda(), k_tree=c["k_tree"].cuda(), v_tree=c["v_tree"].cuda(), k_pages=kp,
                             v_pages=c["v_pages"].cuda())
    torch.cuda.synchronize()
    assert r["status"].cpu().tolist() == [0, 1]
    assert pl.cpu().tolist() == [6, 5]
    changed = (kp.float().nan_to_num(3.0) != before.float().nan_to_num(3.0))
    pg = int(c["table"][0, 0])
    assert changed[:, pg].any() and not changed[:, [p for p in range(kp.shape[1]) if p != pg]].any()
