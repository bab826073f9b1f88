"""The N-GPU harness of bench.py on CPU: world_size 2 over gloo.

Streams are independent, so ranks run replicas and exchange nothing on the
data path; the only cross-rank step is bench.combine_ranks (slowest rank's
times, total bytes).  Run as two processes on 127.0.0.1."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r: step 10+r ms, e2e 20+2r ms, attend 5+3r ms, 100*(r+1) bytes
    out = bench.combine_ranks(10.0 + rank, 20.0 + 2 * rank, 5.0 + 3 * rank, 100.0 * (rank + 1),
                              world, "cpu")
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


def test_combine_ranks_world2_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r] == (11.0, 22.0, 8.0, 300.0)


def test_combine_ranks_single():
    import bench
    assert bench.combine_ranks(1.0, 2.0, 3.0, 4.0, 1, "cpu") == (1.0, 2.0, 3.0, 4.0)
