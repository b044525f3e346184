"""The N > 1 paths on CPU with gloo, world size 2.

* amax_allreduce: ranks hold different amaxes (their shards of a tensor);
  after the MAX all-reduce every rank has the elementwise maximum, and the
  oracle's scale update then yields identical scales on every rank.
* dbias_allreduce: each rank holds the db of its rows of dy (the oracle's
  column sums of its shard); after the SUM all-reduce both ranks hold the
  same bits, within the dbias tolerance of the column sums of the whole dy.
* bench.py's max-over-ranks timing reduction, with gloo standing in for
  NCCL: the slowest rank's time is what both ranks see.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, fn, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, fn(rank, world)))
    except Exception as e:  # surface the error in the parent
        q.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


def _run(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, fn, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


def _amax_case(rank, world):
    import oracle
    from cast_transpose_gb300.distributed import amax_allreduce
    # each rank's shard of 3 tensors: rank 1 holds the larger amax of tensor 0 and
    # 2, rank 0 of tensor 1; tensor 2 is all zero on rank 0
    shards = [oracle.amax(torch.randn(64, 32, generator=torch.Generator().manual_seed(10 * rank + i))
                          .to(torch.bfloat16) * (1 + rank if i != 1 else 2 - rank))
              for i in range(3)]
    if rank == 0:
        shards[2] = np.float32(0.0)
    hist = torch.zeros(4, 3)
    hist[0] = torch.tensor(np.array(shards, dtype=np.float32))
    local = hist[0].clone()
    amax_allreduce(hist[0])
    h, s, si = oracle.amax_and_scale_update(hist.numpy(), np.ones(3, np.float32),
                                            np.ones(3, np.float32), oracle.E4M3, 0)
    return {"local": local.numpy(), "reduced": hist[0].numpy().copy(), "scale": s}


def test_amax_allreduce_gloo_world2():
    out = _run(_amax_case)
    want = np.maximum(out[0]["local"], out[1]["local"])
    for r in (0, 1):
        assert np.array_equal(out[r]["reduced"], want)
    assert np.array_equal(out[0]["scale"].view(np.uint32), out[1]["scale"].view(np.uint32))


def _dbias_case(rank, world):
    import oracle
    from cast_transpose_gb300 import workloads
    from cast_transpose_gb300.distributed import dbias_allreduce
    dy = workloads.gradient_matrix("cpu", 512, 300, std=1e-2, outlier_fraction=1e-3)
    shard = dy[rank * 256:(rank + 1) * 256]
    db = torch.from_numpy(oracle.dbias(shard).copy())
    dbias_allreduce(db)
    return {"db": db.numpy().copy()}


def test_dbias_allreduce_gloo_world2():
    out = _run(_dbias_case)
    import oracle
    from cast_transpose_gb300 import workloads
    dy = workloads.gradient_matrix("cpu", 512, 300, std=1e-2, outlier_fraction=1e-3)
    ref = oracle.dbias(dy).astype(np.float64)
    tol = 1e-5 * dy.double().abs().sum(0).numpy() + 1e-6
    assert np.array_equal(out[0]["db"].view(np.uint32), out[1]["db"].view(np.uint32))
    assert np.all(np.abs(out[0]["db"].astype(np.float64) - ref) <= tol)


def test_dbias_allreduce_rejects_bf16():
    from cast_transpose_gb300.distributed import dbias_allreduce
    with pytest.raises(TypeError):
        dbias_allreduce(torch.zeros(4, dtype=torch.bfloat16))


def _timing_case(rank, world):
    import bench
    return bench._max_over_ranks(1.5 if rank == 0 else 2.25, world)


def test_max_over_ranks_gloo_world2():
    out = _run(_timing_case)
    assert out == {0: 2.25, 1: 2.25}


def test_amax_allreduce_single_process_is_noop():
    from cast_transpose_gb300.distributed import amax_allreduce
    a = torch.tensor([1.0, 2.0])
    assert amax_allreduce(a) is a and a.tolist() == [1.0, 2.0]
