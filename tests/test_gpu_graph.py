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
