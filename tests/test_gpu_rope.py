"""GPU parity of ddt_rope_tree against the oracle: tree rows rotated at prefix_len + depth."""
import numpy as np
import pytest
import torch

import oracle
from tests import _cases as C
from tests._parity import TOL, normwise
from tree_speculative_decoding_02_gb300 import ddt, synth

pytestmark = pytest.mark.gpu


def _case(dtype, prefix, d=128, Hq=8, Hkv=2, L=2):
    tree, _ = C.tree_from_logits(3, len(prefix), 15, 3000, 8, 64, prefix=prefix)
    N = 65
    g = synth.gen(3, 50)
    q = synth.normal((L, len(prefix), N, Hq, d), g=g, dtype=dtype)
    k = synth.normal((L, len(prefix), N, Hkv, d), g=g, dtype=dtype)
    return tree, q, k


@pytest.mark.parametrize("rot,theta", [(128, 10000.0), (32, 1e6)])
def test_rope_fp32_matches_oracle(rot, theta):
    """Positions up to 40,000 + depth (angles of 4e4 radians), full and partial rotation."""
    tree, q, k = _case(torch.float32, [0, 4095, 40000])
    t = C.tree_to_dev(tree)
    qd, kd = q.cuda(), k.cuda()
    ddt.ddt_rope_tree(qd, kd, t["position"], t["n_nodes"], rot_dim=rot, theta=theta)
    torch.cuda.synchronize()
    wq = oracle.rope_tree(C.f64(q), tree["position"], tree["n_nodes"], rot, theta)
    wk = oracle.rope_tree(C.f64(k), tree["position"], tree["n_nodes"], rot, theta)
    for got, want in ((qd, wq), (kd, wk)):
        err = normwise(C.f64(got), want, axes=-1)
        assert err.max() <= TOL, err.max()
    assert err.max() <= 1e-5          # fp32 arithmetic after an fp64 angle: far inside the bar


def test_rope_bf16_is_one_rounding_and_padding_untouched():
    tree, q, k = _case(torch.bfloat16, [17, 30000])
    tree["n_nodes"][1] = 40                 # rows 40.. of request 1 become padding
    t = C.tree_to_dev(tree)
    qd = q.cuda()
    ddt.ddt_rope_tree(qd, k.cuda(), t["position"], t["n_nodes"])
    torch.cuda.synchronize()
    want = oracle.rope_tree(C.f64(q), tree["position"], tree["n_nodes"], 128)
    got = C.f64(qd)
    assert (np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-6).all()
    assert torch.equal(qd[:, 1, 40:].cpu(), q[:, 1, 40:])


@pytest.mark.parametrize("d,rot,prefix", [(256, 256, [0, 300, 4097]), (128, 64, [129, 7, 2000])])
def test_fused_rope_attention_is_rope_then_attention(d, rot, prefix):
    """ddt_tree_attn_rope on unrotated q equals ddt_rope_tree on q followed by
    ddt_tree_attn, bit for bit; both match the oracle's rotation followed by its
    attention.  Keys are rotated alone (q = None) for the fused call."""
    import math
    B, L, Hq, Hkv = len(prefix), 2, 12, 2
    tree, _ = C.tree_from_logits(3, B, 15, 3000, 8, 64, prefix=prefix)
    N = 65
    Pcap = max(prefix) + N + 5
    inp = synth.attn_inputs(L, B, N, Hq, Hkv, d, Pcap, np.asarray(prefix), workload=7, dtype=torch.bfloat16)
    t = C.tree_to_dev(tree)
    dev = lambda x: x.cuda().clone()  # noqa: E731
    scale = 1.0 / math.sqrt(d)
    qa, ka = dev(inp.q), dev(inp.k_tree)
    ddt.ddt_rope_tree(qa, ka, t["position"], t["n_nodes"], rot_dim=rot)
    ra = ddt.ddt_tree_attn(qa, ka, dev(inp.v_tree), dev(inp.k_cache), dev(inp.v_cache), inp.prefix_len.cuda(),
                           t["n_nodes"], t["anc"], scale=scale, out_dtype=torch.float32)
    kb = dev(inp.k_tree)
    ddt.ddt_rope_tree(None, kb, t["position"], t["n_nodes"], rot_dim=rot, Hq=Hq)
    rb = ddt.ddt_tree_attn_rope(dev(inp.q), kb, dev(inp.v_tree), dev(inp.k_cache), dev(inp.v_cache),
                                inp.prefix_len.cuda(), t["n_nodes"], t["anc"], t["position"], scale=scale, rot_dim=rot,
                                out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(ka, kb)
    assert torch.equal(ra["o"], rb["o"])
    assert (rb["status"].cpu() == 0).all()
    # the kernels see bf16 q and keys after rotation: the oracle's fp64 rotation, rounded
    # to bf16 the same way, is the input of the oracle's attention
    bf = lambda a: torch.as_tensor(a).to(torch.bfloat16).double().numpy()  # noqa: E731
    wq = bf(oracle.rope_tree(C.f64(inp.q), tree["position"], tree["n_nodes"], rot))
    wk = bf(oracle.rope_tree(C.f64(inp.k_tree), tree["position"], tree["n_nodes"], rot))
    want = oracle.tree_attn(wq, wk, C.f64(inp.v_tree), np.nan_to_num(C.f64(inp.k_cache)),
                            np.nan_to_num(C.f64(inp.v_cache)), inp.prefix_len.numpy(), tree["n_nodes"], tree["anc"],
                            scale)["o"]
    got = rb["o"].cpu().double().numpy()
    for b in range(B):
        n = int(tree["n_nodes"][b])
        err = normwise(got[:, b, :n], want[:, b, :n], axes=-1)
        assert err.max() <= TOL, err.max()


def test_fused_rope_paged_attention_is_rope_then_attention():
    """The paged variant, 64-row pages: bit for bit the unfused paged call."""
    import math
    from tests.test_gpu_paged import _paged
    B, L, Hq, Hkv, d, rot = 2, 2, 12, 2, 256, 128
    prefix = [300, 1500]
    tree, _ = C.tree_from_logits(3, B, 15, 3000, 8, 64, prefix=prefix)
    c = _paged(9, L, B, 65, Hq, Hkv, d, prefix, 64)
    t = C.tree_to_dev(tree)
    scale = 1.0 / math.sqrt(d)
    dev = lambda x: x.cuda().clone()  # noqa: E731
    qa, ka = dev(c["q"]), dev(c["k_tree"])
    ddt.ddt_rope_tree(qa, ka, t["position"], t["n_nodes"], rot_dim=rot)
    args = (dev(c["v_tree"]), dev(c["k_pages"]), dev(c["v_pages"]), c["table"].cuda(), torch.as_tensor(c["P"]).cuda(),
            t["n_nodes"], t["anc"])
    ra = ddt.ddt_tree_attn_paged(qa, ka, *args, scale=scale, out_dtype=torch.float32)
    kb = dev(c["k_tree"])
    ddt.ddt_rope_tree(None, kb, t["position"], t["n_nodes"], rot_dim=rot, Hq=Hq)
    rb = ddt.ddt_tree_attn_paged_rope(dev(c["q"]), kb, *args, t["position"], scale=scale, rot_dim=rot,
                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(ka, kb)
    assert torch.equal(ra["o"], rb["o"])
    assert (rb["status"].cpu() == 0).all()
