"""bench.py on N > 1 GPUs runs independent replicas (the decode path has no
exchange step): every rank times its own steps, the job's time is the
slowest rank's and its throughput is the units of all ranks over that time.
This checks the host side of that on two gloo ranks on the CPU."""
import os
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))


def _rank(rank, ws, port, q):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        slowest = bench.max_over_ranks(1.5 + rank, ws)         # rank r took 1.5 + r seconds
        thr = bench.replica_throughput(100.0, 1.5 + rank, ws)  # 100 units per rank
        bench.barrier(ws)
        q.put((rank, slowest, thr))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_replicas_take_the_slowest_rank():
    ws, port = 2, 29500 + os.getpid() % 2000
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=100) for _ in range(ws))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, slowest, thr in got:
        assert slowest == 2.5                    # max over the ranks, on every rank
        assert thr == pytest.approx(2 * 100.0 / 2.5)


def test_one_rank_is_its_own_job():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.replica_throughput(10.0, 2.0, 1) == 5.0
