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
