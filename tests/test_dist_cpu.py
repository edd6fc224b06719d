"""The benchmark's multi-rank path on CPU: two gloo ranks rendezvous the way
torchrun launches them (127.0.0.1) and reduce their timings to the max."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    os.environ["CUDA_VISIBLE_DEVICES"] = ""
    import torch.distributed as dist
    import bench
    r, w, _ = bench.dist_setup(None)
    v = bench.reduce_max(1.5 * (rank + 1))
    q.put((r, w, v, dist.get_backend()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 and o[2] == 3.0 and o[3] == "gloo" for o in out)


def test_single_rank_reduce_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(2.5) == 2.5
