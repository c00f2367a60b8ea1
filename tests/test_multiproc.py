"""The multi-GPU benchmark path is replicas only (the (sequence, head) problems are
independent, no data-path collective); its rank logic -- barrier and the max of the per-rank
times -- runs here as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    w, r, _ = bench.dist_setup(world)
    bench.barrier(w)
    t = bench.max_over_ranks(1.5 + rank, w)  # per-rank "time" in ms
    tokens = 1000
    value = w * tokens / (t / 1000.0)        # whole-job throughput from the slowest rank
    q.put((r, w, t, value))
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.skipif(not torch.distributed.is_available(), reason="no torch.distributed")
def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, t, value in res:
        assert w == 2
        assert t == pytest.approx(2.5)
        assert value == pytest.approx(2 * 1000 / 2.5e-3)
