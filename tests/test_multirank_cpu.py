"""The N > 1 bench path on CPU: two gloo ranks (127.0.0.1) run the same
max-over-ranks timing reduction and whole-job throughput the GPU bench uses
under NCCL, with replicas that take different times."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    per_rank_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow replica
    bench.barrier(world)
    thr, slowest = bench.job_throughput(1e9, per_rank_ms, world)
    q.put((rank, thr, slowest))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_gloo_throughput_uses_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=90) for _ in range(world))
    for p in procs:
        p.join(30)
        assert p.exitcode == 0
    for rank, thr, slowest in res:
        assert slowest == 15.0
        assert abs(thr - 2e9 / 15e-3) < 1e-3 * thr


def test_single_rank_is_identity():
    import bench
    thr, slowest = bench.job_throughput(1e9, 4.0, 1)
    assert slowest == 4.0 and abs(thr - 1e9 / 4e-3) < 1
