"""The benchmark's multi-rank plumbing on CPU: two gloo ranks, barrier and
max-over-ranks timing, and the reference arm running on rank 0 only.  Each rank
is an independent replica of the layer, so nothing else crosses ranks."""
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
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup(world)
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 * (r + 1), w)
    # the reference arm prints on rank 0 only; other ranks return at once
    other = bench.run_reference(None, None, w, r) if r != 0 else "rank0"
    dist.destroy_process_group()
    q.put((r, w, slowest, other))


def test_two_gloo_ranks_agree_on_the_slowest_time():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 and g[2] == 20.0 for g in got)
    assert got[1][3] is None
