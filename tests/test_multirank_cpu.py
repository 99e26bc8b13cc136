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


# ------------------------------------------------ expert-parallel split (gloo)
def _shard_worker(rank, world, port, q, sizes):
    """Each rank takes its experts' slice of group_sizes, rows, codes and scales
    (workloads.expert_shard), runs the oracle on that shard alone, and the
    shards are gathered on every rank."""
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from fp8_moe_routed_gb300 import workloads as W
    from oracle import oracle as orc
    dist.init_process_group("gloo")
    E, K, F, M = 4, 256, 128, 512
    gs = torch.tensor(sizes, dtype=torch.int32)
    T = int(gs.sum())
    x = W.fill_tail_garbage(W.activations(M, K, 1, outlier_frac=0.02), T)
    d = W.fill_tail_garbage(W.cotangent(M, 2 * F, 2), T)
    codes, scale = W.fp8_weights(E, K, 2 * F, 0.02, 3)
    sh = W.expert_shard(gs, rank, world, M=M)
    gsl, (xl, dl), (cl, sl) = sh.take(gs, rows=(x, d), experts=(codes, scale))
    h, _, bad0 = orc.gmm_fwd(xl, cl, sl, gsl, silu=True)
    dx, _, bad1 = orc.gmm_dlhs(dl, cl, sl, gsl)
    dw, bad2 = orc.tgmm(xl, dl, gsl)
    assert bad0 == bad1 == bad2 == 0
    mine = (sh.e0, sh.e1, sh.row0, sh.row1, h.view(torch.int16), dx.view(torch.int16), dw)
    got = [None] * world
    dist.all_gather_object(got, mine)
    # plain numpy arrays through the queue: a tensor would travel as a shared-
    # memory handle that can vanish when this process exits before it is read
    q.put((rank, [tuple(x.numpy() if torch.is_tensor(x) else x for x in g) for g in got]))
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU-only test (gloo)")
@pytest.mark.parametrize("sizes,aligned", [([200, 56, 130, 100], True),
                                           ([150, 0, 230, 100], False)])
def test_expert_parallel_shards_reassemble_the_single_rank_result(sizes, aligned):
    """World size 2, each rank holding half the experts and their rows: the
    union of the shards' oracle results equals the single-rank oracle's, and
    the shards cover every expert and every valid row once.

    The forward (with SwiGLU) and the dLHS are row-local: bit for bit always.
    The weight gradient quantizes per 128-row tile of the buffer a rank holds,
    so it is bit for bit when the shard boundary falls on a tile boundary
    (first case: rank 1 starts at row 256). Otherwise every tile of rank 1 is
    cut at other rows, each channel gets other scales, and dW differs by the
    FP8 quantization error itself (about a tenth of its rms here): the shards
    then compute a different, equally valid, quantization of the same
    product, and only its finiteness is checked."""
    from fp8_moe_routed_gb300 import workloads as W
    from oracle import oracle as orc
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q, sizes)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res = {r: [tuple(torch.from_numpy(x) if hasattr(x, "dtype") else x for x in g) for g in v]
           for r, v in res.items()}
    # both ranks gathered the same shards
    assert all(torch.equal(a, b) if torch.is_tensor(a) else a == b
               for s0, s1 in zip(res[0], res[1]) for a, b in zip(s0, s1))
    shards = res[0]
    E, K, F, M = 4, 256, 128, 512
    gs = torch.tensor(sizes, dtype=torch.int32)
    T = int(gs.sum())
    x = W.fill_tail_garbage(W.activations(M, K, 1, outlier_frac=0.02), T)
    d = W.fill_tail_garbage(W.cotangent(M, 2 * F, 2), T)
    codes, scale = W.fp8_weights(E, K, 2 * F, 0.02, 3)
    h, _, _ = orc.gmm_fwd(x, codes, scale, gs, silu=True)
    dx, _, _ = orc.gmm_dlhs(d, codes, scale, gs)
    dw, _ = orc.tgmm(x, d, gs)
    assert [(s[0], s[1]) for s in shards] == [(0, 2), (2, 4)]
    assert shards[0][2] == 0 and shards[0][3] == shards[1][2] and shards[1][3] == T
    assert (shards[1][2] % 128 == 0) == aligned
    for e0, e1, r0, r1, hs, dxs, dws in shards:
        assert torch.equal(hs, h.view(torch.int16)[r0:r1])
        assert torch.equal(dxs, dx.view(torch.int16)[r0:r1])
        if aligned:
            assert torch.equal(dws, dw[e0:e1])
        else:
            assert torch.isfinite(dws).all()


def test_expert_shard_clamps_like_the_kernels():
    from fp8_moe_routed_gb300 import workloads as W
    gs = torch.tensor([-3, 100, 300, 50], dtype=torch.int32)
    a, b = W.expert_shard(gs, 0, 2, M=256), W.expert_shard(gs, 1, 2, M=256)
    assert (a.e0, a.e1, a.row0, a.row1) == (0, 2, 0, 100)
    assert (b.e0, b.e1, b.row0, b.row1) == (2, 4, 100, 256)
    with pytest.raises(ValueError):
        W.expert_shard(gs, 2, 2)
