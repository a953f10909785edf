"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

bs=1 decode does not shard; each rank is an independent replica.  The job's
throughput is all ranks' tokens over the slowest rank's time, and the ranks
meet only at barriers and these two reductions (no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as tmp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    w, r, _ = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.dist_barrier(w)
    tokens = 100 * (rank + 1)
    seconds = [0.5, 2.0][rank]
    value, t = bench.aggregate(w, tokens, seconds)
    q.put((rank, value, t))
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_aggregate_over_ranks(world):
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, t in out:
        assert t == 2.0                      # the slowest rank's time
        assert value == pytest.approx(300 / 2.0)   # all ranks' tokens over it
