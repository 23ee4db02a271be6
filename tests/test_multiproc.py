"""The N > 1 path of bench.py on CPU: two gloo ranks.  Each rank runs its own
replica of the workload (weak scaling, no data-path collective); the line
takes the slowest rank's time (max over ranks) and rank 0 alone prints.  The
reference arm runs on rank 0 only; the other ranks exit 0 without work."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.rank_max(1.5 + rank, dist, "cpu")
        # the reference arm: ranks other than 0 return at once
        class A:
            steps, warmup = 1, 0
        ref = bench.run_reference(A, rank, world) if rank != 0 else 0
        dist.barrier()
        q.put((rank, got, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [2.5, 2.5]
    assert res[1][2] == 0


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.rank_max(3.25, None, "cpu") == 3.25
