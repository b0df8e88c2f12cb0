"""The bounded device waits give up instead of hanging: a wait on an mbarrier that
nothing signals reports DDT_ERR_TIMEOUT after its limit, and the context stays usable."""
import time

import pytest
import torch

from tree_speculative_decoding_02_gb300 import ddt, synth

pytestmark = pytest.mark.gpu


def test_wait_on_unsignalled_barrier_times_out():
    t0 = time.time()
    assert ddt.ddt_wait_selftest() == 5          # DDT_ERR_TIMEOUT
    dt = time.time() - t0
    assert 0.2 < dt < 30.0                       # about a second of SM clock cycles
    # the same context still runs the library afterwards
    g = synth.gen(1, 1)
    logits = synth.draft_logits(1, 4, 500, std=2.0, boost=0.0, g=g, dtype=torch.float32).cuda()
    out = ddt.ddt_build_tree(logits, torch.tensor([1], dtype=torch.int32, device="cuda"),
                             torch.tensor([0], dtype=torch.int32, device="cuda"), 4, 8)
    torch.cuda.synchronize()
    assert int(out["status"][0]) == 0 and int(out["n_nodes"][0]) == 9
