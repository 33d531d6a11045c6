"""Host logic of the N-replica bench on CPU: two gloo ranks, max-over-ranks timing."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_seconds = 1.5 + rank  # rank 1 is the slow one
    bench.barrier(world)
    got = bench.aggregate_max(local_seconds, world)
    r, w, _ = bench.dist_env()
    q.put((rank, got, r, w))
    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [2.5, 2.5]          # both ranks see the slowest rank's time
    assert [(r[2], r[3]) for r in res] == [(0, 2), (1, 2)]


def test_single_rank_is_identity():
    import bench

    assert bench.aggregate_max(3.25, 1) == 3.25
