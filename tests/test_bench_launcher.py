"""bench.py's N-rank path on the CPU (gloo, world size 2).

* spawn_ranks + _dist: two spawned ranks get the launcher environment and
  join one process group (gloo where there is no GPU, NCCL on GPUs).
* exchange_amaxes, the path's one exchange step: each rank casts its own
  shard of the list (the oracle stands in for the kernels here), the MAX
  all-reduce of the amax row gives both ranks the elementwise maximum, and
  the oracle's scale update then yields bit-identical scales on both ranks.
* _max_over_ranks / aggregate_value: the slowest rank's time and the
  whole-job value that rank 0 reports.
* main() with --gpus 2 and no WORLD_SIZE spawns its own ranks; the reference
  arm's line then reports n_gpus == 2 and only rank 0 prints.
"""
import json
import os

import numpy as np
import pytest
import torch

import bench


def _rank_body(outdir):
    import oracle
    from cast_transpose_gb300 import workloads
    world, rank, local = bench._dist()
    shapes = ((64, 96), (96, 64), (32, 64), (64, 128))
    xs = workloads.multi_list("cpu", count=8, shapes=shapes, zero=(3,), tiny=(5,), shard=rank)
    hist = torch.zeros(bench.HIST_LEN, len(xs))
    for i, x in enumerate(xs):
        hist[0, i] = float(oracle.amax(x))
    local_row = hist[0].clone()
    bench.exchange_amaxes(hist[0], world)
    h, s, si = oracle.amax_and_scale_update(hist.numpy(), np.ones(len(xs), np.float32),
                                            np.ones(len(xs), np.float32), oracle.E4M3, 0)
    t = bench._max_over_ranks(1.0 + rank, world)
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": world, "rank": rank, "local": local,
                   "local_row": local_row.numpy().view(np.uint32).tolist(),
                   "reduced_row": hist[0].numpy().view(np.uint32).tolist(),
                   "scale_bits": s.view(np.uint32).tolist(),
                   "scale_inv_bits": si.view(np.uint32).tolist(),
                   "t": t, "value": bench.aggregate_value(world, 10 ** 9, t)}, f)


def test_two_ranks_exchange_amaxes_and_agree_on_scales(tmp_path):
    bench.spawn_ranks(2, _rank_body, (str(tmp_path),))
    r = [json.load(open(tmp_path / f"rank{k}.json")) for k in range(2)]
    assert [x["world"] for x in r] == [2, 2] and [x["local"] for x in r] == [0, 1]
    loc = [np.array(x["local_row"], np.uint32).view(np.float32) for x in r]
    assert not np.array_equal(loc[0], loc[1])              # the shards differ
    expect = np.maximum(loc[0], loc[1])
    for x in r:
        assert np.array_equal(np.array(x["reduced_row"], np.uint32).view(np.float32), expect)
    assert r[0]["scale_bits"] == r[1]["scale_bits"]
    assert r[0]["scale_inv_bits"] == r[1]["scale_inv_bits"]
    assert r[0]["t"] == r[1]["t"] == 2.0                   # the slower rank's time
    assert r[0]["value"] == pytest.approx(2 * 10 ** 9 / 2e-3 / 1e9)


def test_main_spawns_ranks_and_reports_world(capfd):
    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        bench.main(["--gpus", "2", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    finally:
        os.environ.update(env)
    out = capfd.readouterr().out
    lines = [json.loads(l) for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1                                  # rank 0 alone prints
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
