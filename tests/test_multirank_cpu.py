"""Multi-rank host logic of bench.py on the CPU (gloo, world size 2): the
environment-driven rendezvous, the barrier around the timed region and the
max-over-ranks reduction of the step time. The GPU data path has no collective
(expert-parallel replicas), so this is all the multi-process logic there is."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, local = bench.dist_setup(None)
    assert dist.get_backend() == "gloo"
    # each rank "measured" a different time; all must agree on the max
    t = bench.allmax(10.0 + 5.0 * r, w, torch.device("cpu"))
    bench.barrier(w)
    q.put((r, w, local, t))
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU-only test (gloo)")
def test_two_ranks_rendezvous_barrier_and_max():
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
    assert [x[0] for x in res] == [0, 1]
    assert all(x[1] == 2 for x in res)
    assert all(x[3] == 15.0 for x in res)       # max over ranks


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.allmax(3.5, 1, torch.device("cpu")) == 3.5
    bench.barrier(1)
