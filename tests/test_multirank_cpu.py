"""bench.py's multi-rank harness on the CPU: two gloo ranks rendezvous on
127.0.0.1, agree on the max of their timings and pass a barrier. The step
itself has no exchange between ranks (each rank runs its own replica), so
this is the only multi-process logic there is."""
import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    import bench
    world, r, _ = bench.dist_setup()
    v = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    bench.barrier(world)
    q.put((r, world, v, torch.distributed.get_backend()))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 15.0, "gloo"), (1, 2, 15.0, "gloo")]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
