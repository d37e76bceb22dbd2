"""bench.py's N > 1 host logic (replicas only: barrier + max of per-rank
times, whole-job throughput) on two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    bench.rank_barrier(w)
    local_seconds = 1.0 + rank            # rank 1 is the slower one
    slowest = bench.max_over_ranks_value(local_seconds, w, "cpu")
    value = bench.job_throughput(1e12, 3, w, slowest)
    bench.rank_barrier(w)
    dist.destroy_process_group()
    q.put((r, w, lr, slowest, value))


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r, w, lr, slowest, value) in enumerate(out):
        assert (r, w, lr) == (rank, 2, rank)
        assert slowest == 2.0                 # max over ranks
        assert value == pytest.approx(3.0)    # 2 ranks x 3 steps x 1 TB / 2 s
