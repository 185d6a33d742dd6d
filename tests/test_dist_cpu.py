"""The multi-GPU launch path of bench.py, exercised on the CPU with the gloo
backend and two ranks: rendezvous from the torchrun environment variables,
barrier, and the max / sum reductions over ranks that turn per-rank device
times into the job's time (weak scaling: each rank runs its own replica)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import bench
    r, w, local = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    dev = torch.device("cpu")
    mx = bench.max_over_ranks(dist, 10.0 + r, dev)
    sm = bench.sum_over_ranks(dist, 1.5 * (r + 1), dev)
    bench.barrier(dist)
    q.put((r, w, local, mx, sm))
    dist.destroy_process_group()


def test_two_rank_gloo_reductions():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    for r, w, local, mx, sm in results:
        assert w == world and local == r
        assert mx == 11.0
        assert sm == pytest.approx(1.5 + 3.0)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.0, None) == 3.0
    assert bench.sum_over_ranks(None, 3.0, None) == 3.0
