"""The multi-GPU path of the benchmark on CPU: two gloo ranks.  The scan shards
as independent replicas (no data exchange between devices), so what the N>1
path adds is only the timing protocol: a barrier around the timed region,
the maximum time over ranks, and the whole-job value over all ranks' units."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(world, backend="gloo")
    bench.barrier(w)
    t_ms = 100.0 + 50.0 * r  # rank 1 is the slower one
    t_max = bench.max_over_ranks(t_ms, w)
    q.put((r, w, t_max, bench.job_value(1000, 4, w, t_max)))
    bench.barrier(w)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replica_timing_protocol():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for r, w, t_max, v in out:
        assert w == world
        assert t_max == 150.0  # every rank reports the slowest rank's time
        assert v == pytest.approx(1000 * 4 * world / 0.150)  # all ranks' units / that time
