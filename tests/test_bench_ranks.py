"""The multi-process path of bench.py on CPU (gloo, world size 2): the timed
value is the max over ranks, and only rank 0 reports. The forward has no data
exchange between GPUs (replicas), so this is the only cross-rank step."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_env()
    got = bench.max_over_ranks(10.0 * (rank + 1) + 0.25, w, device="cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, w, r, local, got))


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r, w, rr, lr) for r, w, rr, lr, _ in res] == [(0, 2, 0, 0), (1, 2, 1, 1)]
    assert all(got == pytest.approx(20.25) for *_, got in res)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
