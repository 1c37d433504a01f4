"""The multi-rank path of the benchmark (independent replicas, max-over-ranks
timing) on CPU ranks with the gloo backend, world size 2."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slow = bench.dist_max(10.0 + 5.0 * rank)          # rank 1 is the slowest
        value = bench.whole_job_throughput(1000.0, slow, world)
        q.put((rank, slow, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for _, slow, value in res:
        assert slow == 15.0
        assert abs(value - 1000.0 * 2 / 0.015) < 1e-6 * value
