"""The bench's multi-rank path on CPU: two gloo ranks agree on the max-over-ranks time
and the summed node count (whole-job throughput), and the reference arm runs on rank 0
only."""
import argparse
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    torch.cuda.is_available = lambda: False   # gloo, whatever the machine has
    import torch.distributed as dist

    r, w, _ = bench.dist_setup(world)
    ms = 10.0 * (rank + 1)          # rank 1 is the slower one
    nodes = 100 * (rank + 1)
    mx = bench.all_max(ms, w, "cpu")
    total = bench.all_sum(nodes, w, "cpu")
    bench.barrier(w)
    out = bench.run_reference(argparse.Namespace(workload=1, warmup=0, steps=1), r, w) if r != 0 else None
    q.put((r, w, mx, total, out))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(rk, 2, port, q)) for rk in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    for _, _, mx, total, _ in res:
        assert mx == 20.0 and total == 300.0
        assert total / (mx / 1e3) == pytest.approx(15000.0)   # value = all ranks' nodes / max time
    assert res[1][4] is None                                   # reference arm: rank 1 does no work


def test_single_rank_helpers_are_identity():
    assert bench.all_max(3.5, 1, "cpu") == 3.5 and bench.all_sum(7, 1, "cpu") == 7.0
    bench.barrier(1)
    assert bench.dist_setup(1) == (0, 1, 0) or os.environ.get("WORLD_SIZE") not in (None, "1")
