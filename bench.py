"""Benchmark of the FP8 cast-transpose hot path on GB300.

Headline workload (one "step"): the list of 48 bf16 tensors cycling through
6144x12288, 12288x6144, 18432x6144 and 6144x24576 (each a TP=2 shard of a
12288-hidden layer), N(0, 0.02), tensors 7 and 30 all zero and tensors 15 and
44 rescaled to max|x| = 1e-30: one fp8_multi_cast_transpose launch (E4M3
data + transpose + amax into the current amax-history row + each tensor's
scale_inv) followed by one fp8_amax_and_scale_update over the 48 columns
(history length 16, margin 0).  The step is captured once in a CUDA graph and
replayed; inputs are resident in HBM and the 9.97 GB of inputs alone are 77x
the 129 MB L2, so every step streams from DRAM.

Metric: algorithmic GB/s (bytes read + written by the path: 4 bytes per
element for a cast-transpose, the scalars, and the history update) and its
fraction of the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

--gpus N > 1: one process per GPU (launched by torchrun, or spawned here when
WORLD_SIZE is unset).  Rank r casts shard r of the 48 layers (its own seeded
data, the same shapes); the one exchange of the path, the MAX all-reduce of
the 48-entry amax row ("[PyTorch] cuda graph support", feature list: amaxes
reduced within the current iteration), runs between the list launch and the
scale update, so every rank derives identical scales.  Per-rank work is fixed
("weak" scaling); the slowest rank's time counts.

--impl reference times the CPU oracle (plain single-threaded C) on a bounded
sample of the same workload.

Secondary lines (under "secondary", each with its own rate): the weight-like
4096x4096 step (8 casts + 8 updates, with and without CT_X_READY), the
gradient-like 8192x12288 dbias cast-transpose (E5M2), the activation
16384x12288 cast-transpose without a noop flag and with one clear and set, the 256x512
matrix, cast only, the FP8 transpose and a ragged 8191x12287 matrix (cast-transpose
and cast only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import socket
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "cast-transpose GB/s (bytes read+written) and % of GB300 HBM peak"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
HIST_LEN = 16
LIST_SHAPES = ((6144, 12288), (12288, 6144), (18432, 6144), (6144, 24576))
LIST_COUNT = 48
LIST_ELEMS = sum(r * c for r, c in (LIST_SHAPES[i % 4] for i in range(LIST_COUNT)))
LIST_BYTES = 4 * LIST_ELEMS + 12 * LIST_COUNT              # x in, q + qT out, scale/amax/scale_inv
UPDATE_BYTES = (2 * HIST_LEN + 3) * 4 * LIST_COUNT         # history read + rolled write, scale, scale_inv
STEP_BYTES = LIST_BYTES + UPDATE_BYTES
WORKLOAD = ("48-tensor list (12 each of 6144x12288, 12288x6144, 18432x6144, 6144x24576 bf16, "
            "N(0,0.02), tensors 7/30 zero, 15/44 at max|x|=1e-30): per step one E4M3 "
            "multi-tensor cast+transpose+amax launch, then the 48-column amax-history/scale "
            "update (L=16, margin 0)")
DIRECT_SOURCES = ["cast_transpose_gb300/csrc/ct_direct.cu", "cast_transpose_gb300/csrc/ct_device.cuh",
                  "cast_transpose_gb300/csrc/ct_gen_io.cuh"]
FAST_SOURCES = ["cast_transpose_gb300/csrc/ct_fast.cu", "cast_transpose_gb300/csrc/ct_device.cuh"]
# elements of the profiling case the list kernel's DRAM traffic was captured on
# (profile_case('list'): 3 tensors of each list shape at half size)
PROFILE_LIST_ELEMS = 3 * sum((r // 2) * (c // 2) for r, c in LIST_SHAPES)


def _peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "source": "fallback"}


def _source_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(key: str, sources, scale: float = 1.0):
    """DRAM read+write bytes per launch from the committed ncu summary
    (profiles/ncu_traffic.json), scaled by `scale` (units of the full launch
    over units of the captured one), or None when the entry is missing or
    was taken on another version of the kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
        e = d.get(key)
        if e and e.get("kernel_source_sha") == _source_hash(sources):
            return int(round(e["dram_bytes_per_launch"] * scale))
    except Exception:
        pass
    return None


def _pct_nominal(gbs: float) -> float:
    return round(100.0 * gbs / NOMINAL_HBM_GBS, 1)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# ranks
def _dist():
    """World size, rank and local rank from the launcher's environment; joins
    the process group when there is more than one rank (NCCL on GPUs, gloo
    where there is none)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            # communicator set-up lines (rank count) on stderr, off the JSON line
            os.environ.setdefault("NCCL_DEBUG", "INFO")
            os.environ.setdefault("NCCL_DEBUG_SUBSYS", "INIT")
            os.environ.setdefault("NCCL_DEBUG_FILE", "/dev/stderr")
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def exchange_amaxes(amax_row, world: int):
    """The path's one exchange step: MAX all-reduce of the contiguous amax row
    (history row 0, one fp32 per tensor) between the casts and the update."""
    if world > 1:
        from cast_transpose_gb300.distributed import amax_allreduce
        amax_allreduce(amax_row)
    return amax_row


def aggregate_value(world: int, bytes_per_rank: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_entry(local, world, port, target, targs):
    os.environ.update({"RANK": str(local), "LOCAL_RANK": str(local), "WORLD_SIZE": str(world),
                       "LOCAL_WORLD_SIZE": str(world), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    target(*targs)


def spawn_ranks(world: int, target, targs=()):
    """Run target(*targs) in `world` spawned processes, one per rank, with the
    environment torchrun would give them (rendezvous on 127.0.0.1)."""
    import torch.multiprocessing as mp
    mp.start_processes(_rank_entry, args=(world, _free_port(), target, targs), nprocs=world,
                       start_method="spawn", join=True)


# ---------------------------------------------------------------------------
def _list_state(ct, torch, dev, shard):
    from cast_transpose_gb300 import workloads
    xs = workloads.multi_list(dev, shard=shard)
    assert len(xs) == LIST_COUNT and sum(x.numel() for x in xs) == LIST_ELEMS
    outs = [ct.empty_outputs(x) for x in xs]
    n = LIST_COUNT
    st = {"xs": xs, "outs": outs,
          "hist": torch.zeros(HIST_LEN, n, device=dev),
          "scale": torch.ones(n, device=dev),
          "recipe_sinv": torch.ones(n, device=dev),
          "tensor_sinv": torch.zeros(n, device=dev)}
    return st


def _list_cast(ct, st, xs=None, outs=None):
    xs = st["xs"] if xs is None else xs
    outs = st["outs"] if outs is None else outs
    n = LIST_COUNT
    ct.fp8_multi_cast_transpose(xs, [st["scale"][i:i + 1] for i in range(n)],
                                [st["hist"][0, i:i + 1] for i in range(n)],
                                [st["tensor_sinv"][i:i + 1] for i in range(n)],
                                [o[0] for o in outs], [o[1] for o in outs], ct.E4M3)


def _list_update(ct, st):
    ct.fp8_amax_and_scale_update(st["hist"], st["scale"], st["recipe_sinv"], ct.E4M3, 0)


def run_gpu(args):
    import torch

    import cast_transpose_gb300 as ct

    world, rank, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = _peaks()
    st = _list_state(ct, torch, dev, shard=rank)

    def step():
        _list_cast(ct, st)
        exchange_amaxes(st["hist"][0], world)
        _list_update(ct, st)

    # eager warm-up (first call per device sets kernel attributes; the first
    # collective sets up the communicator), then capture
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step()
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()

    # Kernel timing inside the timed region: extra captures of the step carry
    # external event-record nodes on a side branch (after each stage the side
    # stream joins the main one and records an event), so each event fires
    # when that stage completes without holding back the next one.  The span
    # between consecutive events is that stage's share of the step; every
    # 4th replay of the timed loop uses one of these copies, and each copy's
    # events hold the times of its last replay.
    plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(plain):
        step()
    n_evented, every = 4, 4
    evented, kevs = [], []
    for _ in range(n_evented):
        try:
            ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
        except TypeError:      # torch without external events: no per-kernel times
            break
        side = torch.cuda.Stream(device=dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            main = torch.cuda.current_stream()
            side.wait_stream(main)
            with torch.cuda.stream(side):
                ev[0].record()
            _list_cast(ct, st)
            side.wait_stream(main)
            with torch.cuda.stream(side):
                ev[1].record()
            exchange_amaxes(st["hist"][0], world)
            _list_update(ct, st)
            side.wait_stream(main)
            with torch.cuda.stream(side):
                ev[2].record()
            main.wait_stream(side)
        evented.append(g)
        kevs.append(ev)

    def replay(i):
        if evented and i % every == every - 1:
            evented[(i // every) % len(evented)].replay()
        else:
            plain.replay()

    for i in range(args.warmup):
        replay(i)
    torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    _barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for i in range(args.steps):
        replay(i)
    t_end.record()
    torch.cuda.synchronize()
    _barrier(world)
    clocks = sampler.stop() if sampler else None
    elapsed_ms = t_start.elapsed_time(t_end)
    used = sorted({(i // every) % len(evented) for i in range(args.steps) if i % every == every - 1}) \
        if evented else []
    cast_ms = [kevs[j][0].elapsed_time(kevs[j][1]) for j in used]
    rest_ms = [kevs[j][1].elapsed_time(kevs[j][2]) for j in used]
    ms_per_step = _max_over_ranks(elapsed_ms / args.steps, world)

    e2e = list_e2e(ct, torch, dev, st, args, world)
    noop_lines = list_noop(ct, torch, dev, st, peaks) if (rank == 0 and args.extra) else {}
    if rank != 0:
        return
    value = aggregate_value(world, STEP_BYTES, ms_per_step)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "dtype_note": "bf16 in, FP8 (E4M3) codes out; the scale product is one fp32 multiply",
        "data": "synthetic (seeded bf16, the 48-tensor list recipe; rank r draws shard r), "
                "resident in HBM",
        "config": {
            "workload": WORKLOAD,
            "tensors": LIST_COUNT,
            "shapes": [list(s) for s in LIST_SHAPES],
            "fp8": "E4M3",
            "amax_history_len": HIST_LEN,
            "margin": 0,
            "bytes_per_step": STEP_BYTES,
            "cuda_graph": True,
            "l2": "inputs larger than L2: 9.97 GB of inputs + 9.97 GB of outputs per step "
                  "vs 129 MB L2",
            "parallelism": (f"{world} ranks, one per GPU: rank r casts shard r of the 48 layers; "
                            "MAX all-reduce of the amax row before the update") if world > 1
                           else "1 GPU",
            "pct_of_nominal_8000_gbs": _pct_nominal(value / world),
        },
        "gpu_launches": args.steps * 2,
        "e2e": e2e,
        "clocks": clocks,
    }
    if cast_ms:
        avg = statistics.mean(cast_ms)
        achieved = LIST_BYTES / (avg * 1e-3) / 1e9
        line["roofline"] = {
            "kernel": "direct_cast_transpose_kernel (fp8_multi_cast_transpose, 48 tensors, "
                      "one launch)",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "peak_source": peaks["source"] + " copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
            "pct_of_nominal_8000_gbs": _pct_nominal(achieved),
            "traffic": _traffic("direct_cast_transpose_kernel list", DIRECT_SOURCES,
                                LIST_ELEMS / PROFILE_LIST_ELEMS),
            "traffic_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum of the list launch "
                            "on the 12-tensor half-size profiling case, scaled to the full launch "
                            "by elements",
            "algorithmic_bytes_per_launch": LIST_BYTES,
            "avg_launch_us": round(avg * 1e3, 2),
            "launches_timed": len(cast_ms),
            "timing": "external CUDA event-record nodes on a side branch of the step graph "
                      "(span = the launch's share of the step); evented copies replace every "
                      "4th replay of the timed loop, the last replay of each copy is read",
            "share_of_step": round(sum(cast_ms) / max(sum(cast_ms) + sum(rest_ms), 1e-12), 4),
            "update_and_exchange_avg_us": round(statistics.mean(rest_ms) * 1e3, 2),
        }
    else:
        line["roofline"] = None
    if args.extra:
        del st
        torch.cuda.empty_cache()
        line["secondary"] = secondary(dev, peaks, args)
        line["secondary"].update(noop_lines)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(seconds=args.cpu_seconds)
    print(json.dumps(line), flush=True)


def list_e2e(ct, torch, dev, st, args, world) -> dict:
    """The headline step end to end through the public API: every step copies
    its 48 inputs in from pinned host memory, runs the list cast, the amax
    exchange (N > 1) and the update as eager calls, and copies the 96 FP8
    outputs and the scales back out.  Copy-in, compute and copy-out run on
    three streams with two device buffer sets, so step i+1's copy-in
    overlaps step i's copy-out (the link carries both directions at once);
    events order each set's reuse.  One stream per direction keeps each
    direction's copies in issue order."""
    xs, outs = st["xs"], st["outs"]
    n = len(xs)
    steps = max(3, min(args.steps, 50))
    host_in = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in xs]
    for h, x in zip(host_in, xs):
        h.copy_(x)
    host_q = [torch.empty(o[0].shape, dtype=torch.uint8, pin_memory=True) for o in outs]
    host_qt = [torch.empty(o[1].shape, dtype=torch.uint8, pin_memory=True) for o in outs]
    host_scale = torch.empty(2 * n, dtype=torch.float32, pin_memory=True)
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = sum(h.numel() for h in host_q) + sum(h.numel() for h in host_qt) + 8 * n
    sets = [(xs, outs), ([torch.empty_like(x) for x in xs], [ct.empty_outputs(x) for x in xs])]
    n_copy = 1
    s_in = [torch.cuda.Stream(device=dev) for _ in range(n_copy)]
    s_out = [torch.cuda.Stream(device=dev) for _ in range(n_copy)]
    s_comp = torch.cuda.Stream(device=dev)
    ev_in = [[torch.cuda.Event() for _ in range(n_copy)] for _ in range(2)]
    ev_out = [[torch.cuda.Event() for _ in range(n_copy)] for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    for e in ev_comp + [e for row in ev_out for e in row]:
        e.record(torch.cuda.current_stream())

    def e2e_step(i):
        b = i % 2
        bx, bo = sets[b]
        for c, s in enumerate(s_in):
            with torch.cuda.stream(s):
                s.wait_event(ev_comp[b])        # step i-2 no longer reads these inputs
                for k in range(c, n, n_copy):
                    bx[k].copy_(host_in[k], non_blocking=True)
                ev_in[b][c].record(s)
        with torch.cuda.stream(s_comp):
            for c in range(n_copy):
                s_comp.wait_event(ev_in[b][c])
                s_comp.wait_event(ev_out[b][c])  # step i-2's outputs have been copied out
            _list_cast(ct, st, bx, bo)
            exchange_amaxes(st["hist"][0], world)
            _list_update(ct, st)
            ev_comp[b].record(s_comp)
        for c, s in enumerate(s_out):
            with torch.cuda.stream(s):
                s.wait_event(ev_comp[b])
                for k in range(c, n, n_copy):
                    host_q[k].copy_(bo[k][0], non_blocking=True)
                    host_qt[k].copy_(bo[k][1], non_blocking=True)
                if c == 0:
                    host_scale[:n].copy_(st["scale"], non_blocking=True)
                    host_scale[n:].copy_(st["recipe_sinv"], non_blocking=True)
                ev_out[b][c].record(s)

    def joined():
        for s in (*s_in, s_comp, *s_out):
            torch.cuda.current_stream().wait_stream(s)

    for i in range(2):
        e2e_step(i)
    joined()
    torch.cuda.synchronize()
    _barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in (*s_in, s_comp, *s_out):
        s.wait_stream(torch.cuda.current_stream())
    for i in range(steps):
        e2e_step(i)
    joined()
    e1.record()
    torch.cuda.synchronize()
    ms = _max_over_ranks(e0.elapsed_time(e1) / steps, world)
    del sets[1], host_in, host_q, host_qt
    return {"value": round(aggregate_value(world, STEP_BYTES, ms), 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(ms, 4),
            "note": "every step: its 48 inputs copied in from pinned host memory, the step "
                    "through the public API (eager calls), the 96 FP8 outputs and the scales "
                    "copied out; copy-in / compute / copy-out on three streams with two buffer "
                    "sets, step i+1's copy-in overlapping step i's copy-out; bound by the host "
                    "link"}


def list_noop(ct, torch, dev, st, peaks) -> dict:
    """The 48-tensor list cast with a noop flag (the FP8 weight copies of
    lazy refresh: cast once per optimizer step, skipped in the other
    micro-batches): its rate with the flag at 0 and the skipped launch."""
    flag = torch.zeros(1, device=dev)
    res = {}

    def cast():
        n = LIST_COUNT
        ct.fp8_multi_cast_transpose(st["xs"], [st["scale"][i:i + 1] for i in range(n)],
                                    [st["hist"][0, i:i + 1] for i in range(n)],
                                    [st["tensor_sinv"][i:i + 1] for i in range(n)],
                                    [o[0] for o in st["outs"]], [o[1] for o in st["outs"]],
                                    ct.E4M3, noop_flag=flag)
    ms, best = _timed(torch, cast, iters=3, per_graph=3)
    res["cast_transpose 48-tensor list, noop flag 0"] = _rate_entry(
        ms, best, LIST_BYTES, peaks,
        "direct_loop_kernel (list): a looping first wave over 80% of the tiles, then chunks of "
        "tiles per group")
    flag.fill_(1.0)
    ms, best = _timed(torch, cast, per_graph=50)
    res["cast_transpose 48-tensor list, noop flag 1"] = {
        "us": round(ms * 1e3, 2), "us_best": round(best * 1e3, 2),
        "note": "the same launch skipped by the flag"}
    return res


# ---------------------------------------------------------------------------
def _timed(torch, fn, iters=10, per_graph=10):
    """Median and best per-launch time (ms) of `per_graph` back-to-back calls
    captured in one CUDA graph (sustained rate, as inside a training step)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            fn()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(iters):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) / per_graph for a, b in ts]
    return statistics.median(ms), min(ms)


def _rate_entry(ms, best, nbytes, peaks, kernel):
    gbs = nbytes / ms / 1e6
    return {"us": round(ms * 1e3, 2), "us_best": round(best * 1e3, 2), "GB/s": round(gbs, 1),
            "frac": round(gbs / peaks["hbm_gbs"], 4), "pct_of_nominal_8000_gbs": _pct_nominal(gbs),
            "algorithmic_bytes": nbytes, "kernel": kernel}


def weight_step(dev, peaks, steps) -> dict:
    """The weight-like 4096x4096 step: eight casts of x * 2^k (k = -4..3,
    resident copies), each followed by the scale update, in one CUDA graph;
    with CT_X_READY (the update before each cast writes only fp32 scalars)
    and on the default path; then the same two with the updates deferred
    (fp8_cast_transpose_pending, one fp8_amax_and_scale_update_pending per
    step: the same results).  Per-kernel spans come from external event
    nodes on a side branch of an evented copy of the graph."""
    import torch

    import cast_transpose_gb300 as ct
    from cast_transpose_gb300 import workloads
    base = workloads.weight_matrix(dev)
    xs = [workloads.weight_rescaled(base, k) for k in workloads.WEIGHT_EXPONENTS]
    del base
    outs = [ct.empty_outputs(x) for x in xs]
    hist = torch.zeros(HIST_LEN, 1, device=dev)
    scale = torch.ones(1, device=dev)
    recipe_sinv = torch.ones(1, device=dev)
    tensor_sinv = torch.zeros(len(xs), device=dev)
    cast_bytes = 4 * 4096 * 4096 + 12
    step_bytes = len(xs) * (cast_bytes + (2 * HIST_LEN + 3) * 4)

    def step(x_ready, ev=None, side=None):
        for k, x in enumerate(xs):
            ct.fp8_cast_transpose(x, scale, hist[0], tensor_sinv[k:k + 1], outs[k][0], outs[k][1],
                                  ct.E4M3, x_ready=x_ready)
            if ev is not None:
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    ev[1 + 2 * k].record()
            ct.fp8_amax_and_scale_update(hist, scale, recipe_sinv, ct.E4M3, 0)
            if ev is not None:
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    ev[2 + 2 * k].record()

    pend = torch.zeros(len(xs), 1, device=dev)

    def step_deferred(x_ready):
        # the same step with the 8 updates deferred: each cast derives the
        # scale the updates before it would have set, one update pass at the end
        for k, x in enumerate(xs):
            ct.fp8_cast_transpose_pending(x, hist, scale, pend, 0, k, tensor_sinv[k:k + 1],
                                          outs[k][0], outs[k][1], ct.E4M3, x_ready=x_ready)
        ct.fp8_amax_and_scale_update_pending(hist, scale, recipe_sinv, pend, ct.E4M3)

    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(True)
        step_deferred(True)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    res = {"workload": "weight-like bf16 4096x4096 N(0,0.02) x 2^k, k=-4..3: per step 8 x (E4M3 "
                       "cast+transpose+amax, then the update, L=16, margin 0), one CUDA graph",
           "bytes_per_step": step_bytes}
    variants = (("x_ready", lambda: step(True)), ("default_path", lambda: step(False)),
                ("deferred_updates_x_ready", lambda: step_deferred(True)),
                ("deferred_updates_default_path", lambda: step_deferred(False)))
    for key, fn in variants:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(5):
            g.replay()
        torch.cuda.synchronize()
        n = max(20, min(steps, 400))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / n
        res[key] = {"us_per_step": round(ms * 1e3, 2),
                    "GB/s": round(step_bytes / ms / 1e6, 1),
                    "pct_of_nominal_8000_gbs": _pct_nominal(step_bytes / ms / 1e6)}
    # per-kernel spans (CT_X_READY graph)
    try:
        spans = []
        for _ in range(4):
            ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(1 + 2 * len(xs))]
            side = torch.cuda.Stream(device=dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    ev[0].record()
                step(True, ev, side)
                torch.cuda.current_stream().wait_stream(side)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            spans.append([ev[j].elapsed_time(ev[j + 1]) for j in range(2 * len(xs))])
        cast = [sp[2 * k] for sp in spans for k in range(len(xs))]
        upd = [sp[2 * k + 1] for sp in spans for k in range(len(xs))]
        avg = statistics.mean(cast)
        res["cast_kernel"] = {
            "kernel": "fast_cast_transpose_kernel (TMA, persistent)",
            "avg_span_us": round(avg * 1e3, 2),
            "effective_GB/s": round(cast_bytes / avg / 1e6, 1),
            "frac_effective": round(cast_bytes / avg / 1e6 / peaks["hbm_gbs"], 4),
            "note": "span of each cast inside the step, from the completion of the update before "
                    "it; its first tile loads were issued during that update (CT_X_READY) and its "
                    "33.5 MB of FP8 output is still in L2 when it ends (ncu: 33.6 MB of DRAM "
                    "traffic per launch against 67.1 MB algorithmic), so this is an effective "
                    "rate, not DRAM bandwidth",
            "traffic": _traffic("fast_cast_transpose_kernel 4096x4096 E4M3", FAST_SOURCES),
        }
        res["update_kernel_avg_us"] = round(statistics.mean(upd) * 1e3, 2)
    except TypeError:
        pass
    return res


def secondary(dev, peaks, args) -> dict:
    """The other workloads, each on its own inputs (larger than L2 except
    where noted as launch-bound)."""
    import torch

    import cast_transpose_gb300 as ct
    from cast_transpose_gb300 import workloads
    res = {"weight_4096x4096_step": weight_step(dev, peaks, args.steps)}
    torch.cuda.empty_cache()
    s1, a0, si0 = (torch.tensor([v], dtype=torch.float32, device=dev) for v in (1.0, 0.0, 0.0))
    # gradient 8192x12288: dbias + E5M2 (two kernels)
    dy = workloads.gradient_matrix(dev)
    q, qt = ct.empty_outputs(dy)
    db = torch.empty(dy.shape[1], device=dev)
    ws = torch.empty(ct.dbias_workspace_size(*dy.shape), dtype=torch.uint8, device=dev)
    ms, best = _timed(torch, lambda: ct.fp8_dbias_cast_transpose(dy, s1, a0, si0, q, qt, db, ws,
                                                                 ct.E5M2))
    res["dbias_cast_transpose 8192x12288 E5M2"] = _rate_entry(
        ms, best, 4 * dy.numel() + 4 * dy.shape[1] + 12, peaks,
        "direct_cast_transpose_kernel (dbias) + dbias_finish_kernel")
    # the same with the CT_X_READY promise for dy (it holds here: nothing writes dy)
    ms, best = _timed(torch, lambda: ct.fp8_dbias_cast_transpose(dy, s1, a0, si0, q, qt, db, ws,
                                                                 ct.E5M2, x_ready=True))
    res["dbias_cast_transpose 8192x12288 E5M2, CT_DBIAS_X_READY"] = _rate_entry(
        ms, best, 4 * dy.numel() + 4 * dy.shape[1] + 12, peaks,
        "direct_cast_transpose_kernel (dbias) + dbias_finish_kernel; the first tiles of dy are "
        "loaded while the previous call's finish kernel runs (nothing writes dy)")
    del dy, q, qt, db, ws
    # activation 16384x12288: cast-transpose without and with a noop flag (clear,
    # then set), cast only, FP8 transpose
    x = workloads.activation_matrix(dev)
    q, qt = ct.empty_outputs(x)
    ms, best = _timed(torch, lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3))
    res["cast_transpose 16384x12288 E4M3"] = _rate_entry(
        ms, best, 4 * x.numel() + 12, peaks, "direct_cast_transpose_kernel")
    flag = torch.zeros(1, device=dev)
    ms, best = _timed(torch, lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3,
                                                           noop_flag=flag))
    res["cast_transpose 16384x12288 E4M3, noop flag 0"] = _rate_entry(
        ms, best, 4 * x.numel() + 12, peaks,
        "direct_loop_kernel: a looping first wave over 80% of the tiles, then one tile per "
        "256 threads")
    ms, best = _timed(torch, lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3,
                                                           x_ready=True))
    res["cast_transpose 16384x12288 E4M3, CT_X_READY"] = _rate_entry(
        ms, best, 4 * x.numel() + 12, peaks,
        "direct_cast_transpose_kernel; the first tiles are loaded while the previous launch ends "
        "(nothing writes x)")
    flag.fill_(1.0)
    ms, best = _timed(torch, lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3,
                                                           noop_flag=flag), per_graph=50)
    res["cast_transpose 16384x12288 E4M3, noop flag 1"] = {
        "us": round(ms * 1e3, 2), "us_best": round(best * 1e3, 2),
        "note": "the same launch skipped by the flag: each of its CTAs (the looping first wave "
                "and the 1280 after it) starts, waits for the preceding kernel, reads the flag "
                "and exits"}
    ms, best = _timed(torch, lambda: ct.fp8_cast(x, s1, a0, si0, q, ct.E4M3))
    res["cast 16384x12288 E4M3"] = _rate_entry(ms, best, 3 * x.numel() + 12, peaks,
                                               "direct_cast_transpose_kernel (cast only)")
    ms, best = _timed(torch, lambda: ct.fp8_transpose(q, qt))
    res["transpose 16384x12288 FP8"] = _rate_entry(ms, best, 2 * x.numel(), peaks,
                                                   "transpose_fast_kernel")
    # the cached transpose of lazy transpose caching: with a noop flag, clear then set
    flag = torch.zeros(1, device=dev)
    ms, best = _timed(torch, lambda: ct.fp8_transpose(q, qt, noop_flag=flag))
    res["transpose 16384x12288 FP8, noop flag 0"] = _rate_entry(
        ms, best, 2 * x.numel(), peaks,
        "transpose_fast_kernel: a looping first wave over 90% of the tiles, then one tile per CTA")
    flag.fill_(1.0)
    ms, best = _timed(torch, lambda: ct.fp8_transpose(q, qt, noop_flag=flag), per_graph=50)
    res["transpose 16384x12288 FP8, noop flag 1"] = {
        "us": round(ms * 1e3, 2), "us_best": round(best * 1e3, 2),
        "note": "the same launch skipped by the flag"}
    del x, q, qt
    # an odd token count: rows % 16 != 0, cols a multiple of 128 (the direct
    # kernel, transposed blocks at a different offset in every column)
    x = workloads.normal_bf16(8191, 12288, 1.0, 17, dev)
    q, qt = ct.empty_outputs(x)
    ms, best = _timed(torch, lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3))
    res["cast_transpose 8191x12288 E4M3 (odd rows)"] = _rate_entry(
        ms, best, 4 * x.numel() + 12, peaks, "direct_cast_transpose_kernel (odd-row stores)")
    del x, q, qt
    # ragged: odd rows and cols (the flat cast, then the FP8 transpose of q)
    sets = [(workloads.normal_bf16(8191, 12287, 1.0, 17 + k, dev),) for k in range(3)]
    sets = [(xk,) + ct.empty_outputs(xk) for (xk,) in sets]
    turn = [0]

    def rotating():
        xk, qk, qtk = sets[turn[0] % 3]
        turn[0] += 1
        ct.fp8_cast_transpose(xk, s1, a0, si0, qk, qtk, ct.E4M3)

    ms, best = _timed(torch, rotating, per_graph=12)
    res["cast_transpose 8191x12287 E4M3 (ragged), three buffer sets"] = _rate_entry(
        ms, best, 4 * sets[0][0].numel() + 12, peaks,
        "as the next line, each call on the next of three (x, q, qT) sets: no line of q or qT "
        "is reused from the call before")
    del sets
    xbuf = torch.empty(8191 * 12287 + 8, dtype=torch.bfloat16, device=dev)
    x = xbuf[1:1 + 8191 * 12287].view(8191, 12287)
    x.copy_(workloads.normal_bf16(8191, 12287, 1.0, 17, dev))
    q, qt = ct.empty_outputs(x)
    ms, best = _timed(torch, lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3))
    res["cast_transpose 8191x12287 E4M3 (ragged, x 2 bytes past a 16-byte boundary)"] = _rate_entry(
        ms, best, 4 * x.numel() + 12, peaks,
        "cast_flat_shift_kernel (aligned chunks shifted by x's offset), then "
        "transpose_odd_loop_kernel")
    del xbuf, x, q, qt
    x = workloads.normal_bf16(8191, 12287, 1.0, 17, dev)
    q, qt = ct.empty_outputs(x)
    ms, best = _timed(torch, lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3))
    res["cast_transpose 8191x12287 E4M3 (ragged)"] = _rate_entry(
        ms, best, 4 * x.numel() + 12, peaks,
        "cast_flat_kernel (q stored with the L2 evict-last priority), then "
        "transpose_odd_loop_kernel (tiles from the last one back, q mostly from L2)")
    ms, best = _timed(torch, lambda: ct.fp8_transpose(q, qt))
    res["transpose 8191x12287 FP8 (ragged)"] = _rate_entry(ms, best, 2 * x.numel(), peaks,
                                                            "transpose_odd_kernel")
    flag = torch.zeros(1, device=dev)
    ms, best = _timed(torch, lambda: ct.fp8_transpose(q, qt, noop_flag=flag))
    res["transpose 8191x12287 FP8 (ragged), noop flag 0"] = _rate_entry(
        ms, best, 2 * x.numel(), peaks,
        "transpose_odd_loop_kernel: a looping first wave over 90% of the tiles, then one tile per CTA")
    flag.fill_(1.0)
    ms, best = _timed(torch, lambda: ct.fp8_transpose(q, qt, noop_flag=flag), per_graph=50)
    res["transpose 8191x12287 FP8 (ragged), noop flag 1"] = {
        "us": round(ms * 1e3, 2), "us_best": round(best * 1e3, 2),
        "note": "the same launch skipped by the flag"}
    ms, best = _timed(torch, lambda: ct.fp8_cast(x, s1, a0, si0, q, ct.E4M3))
    res["cast 8191x12287 E4M3 (ragged)"] = _rate_entry(ms, best, 3 * x.numel() + 12, peaks,
                                                       "cast_flat_kernel")
    del x, q, qt
    # the small 256x512 matrix (launch-bound: microseconds)
    x = workloads.single_matrix(dev)
    q, qt = ct.empty_outputs(x)
    ms, best = _timed(torch, lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3),
                      per_graph=50)
    res["cast_transpose 256x512 E4M3"] = {"us": round(ms * 1e3, 2), "us_best": round(best * 1e3, 2),
                                          "kernel": "fast_cast_transpose_kernel (launch-bound)"}
    # the 48-column update alone (latency-bound)
    hist = torch.rand(HIST_LEN, LIST_COUNT, device=dev)
    sc, rs = torch.ones(LIST_COUNT, device=dev), torch.ones(LIST_COUNT, device=dev)
    ms, best = _timed(torch, lambda: ct.fp8_amax_and_scale_update(hist, sc, rs, ct.E4M3, 0))
    res["amax_and_scale_update n=48 L=16"] = {"us": round(ms * 1e3, 2),
                                              "us_best": round(best * 1e3, 2),
                                              "kernel": "scale_update_warp_kernel"}
    return res


# ---------------------------------------------------------------------------
# CPU oracle baselines (the oracle as it stands, on the host cores)
SAMPLE_TENSORS = (0, 1, 2, 3)     # one tensor of each list shape


def _sample_inputs():
    """Tensors 0..3 of the list (one per shape), drawn on the CPU with the same
    recipe, as bf16 bit patterns."""
    import numpy as np
    import torch

    from cast_transpose_gb300 import workloads
    return [workloads.multi_tensor(i, "cpu").view(torch.int16).numpy().view(np.uint16)
            for i in SAMPLE_TENSORS]


def _oracle_update_48(oracle, np, state):
    hist, scale, sinv = state
    return oracle.amax_and_scale_update(hist, scale, sinv, oracle.E4M3, 0)


def cpu_baseline(seconds: float = 10.0) -> dict:
    """The single-threaded C oracle on 4 of the 48 tensors (one of each
    shape) plus the 48-column update, repeated for about `seconds`: GB/s of
    algorithmic bytes, which scales linearly to the 48-tensor step."""
    import numpy as np

    import oracle
    xs = _sample_inputs()
    state = (np.zeros((HIST_LEN, LIST_COUNT), np.float32), np.ones(LIST_COUNT, np.float32),
             np.ones(LIST_COUNT, np.float32))
    per_pass = sum(4 * x.size + 12 for x in xs) + UPDATE_BYTES
    done, passes, t0 = 0, 0, time.perf_counter()
    while True:
        hist = state[0]
        for k, x in zip(SAMPLE_TENSORS, xs):
            r = oracle.cast_transpose(x, float(state[1][k]), oracle.E4M3, amax_in=float(hist[0, k]))
            hist[0, k] = r["amax"]
        state = _oracle_update_48(oracle, np, state)
        done += per_pass
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(done / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{passes} pass(es) over 4 of the 48 tensors (one of each shape, "
                      f"{per_pass / 1e9:.2f} GB of algorithmic bytes per pass) + the 48-column "
                      f"update through the single-threaded C oracle, {dt:.1f} s; GB/s scales "
                      f"linearly to the 19.9 GB step; {os.cpu_count()} host cores, 1 used"}


def _oracle_rows_worker(shm_names, shapes, conn):
    """Spawned worker of cpu_baseline_all_cores: attaches the shared inputs,
    then casts the row blocks it is sent with the oracle as it stands and
    answers each with the block's amax."""
    from multiprocessing import shared_memory

    import numpy as np

    import oracle
    shms = [shared_memory.SharedMemory(name=n) for n in shm_names]
    try:
        xs = [np.ndarray(s, dtype=np.uint16, buffer=m.buf) for s, m in zip(shapes, shms)]
        conn.send("ready")
        while True:
            msg = conn.recv()
            if msg is None:
                break
            k, r0, r1, scale = msg
            r = oracle.cast_transpose(xs[k][r0:r1], scale, oracle.E4M3)
            conn.send(float(r["amax"]))
        del xs
    finally:
        for m in shms:
            m.close()


def cpu_baseline_all_cores(seconds: float = 10.0) -> dict:
    """The oracle on every host core: the same 4-tensor sample, each tensor
    split into row blocks, one per spawned worker process running the
    oracle's code as it stands; the amaxes are merged and the 48-column
    update run in this process."""
    import multiprocessing as mp
    from multiprocessing import shared_memory

    import numpy as np

    import oracle
    xs = _sample_inputs()
    workers = max(1, os.cpu_count() or 1)
    shms = [shared_memory.SharedMemory(create=True, size=x.nbytes) for x in xs]
    procs, conns = [], []
    per_pass = sum(4 * x.size + 12 for x in xs) + UPDATE_BYTES
    try:
        for x, m in zip(xs, shms):
            np.ndarray(x.shape, dtype=np.uint16, buffer=m.buf)[:] = x
        ctx = mp.get_context("spawn")
        for _ in range(workers):
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_rows_worker,
                            args=([m.name for m in shms], [x.shape for x in xs], b), daemon=True)
            p.start()
            procs.append(p)
            conns.append(a)
        for c in conns:
            if not c.poll(300) or c.recv() != "ready":
                raise RuntimeError("oracle worker did not start")
        state = (np.zeros((HIST_LEN, LIST_COUNT), np.float32), np.ones(LIST_COUNT, np.float32),
                 np.ones(LIST_COUNT, np.float32))

        def one_pass(state):
            hist = state[0]
            for j, (k, x) in enumerate(zip(SAMPLE_TENSORS, xs)):
                rows = x.shape[0]
                bounds = [rows * w // workers for w in range(workers + 1)]
                for w, c in enumerate(conns):
                    c.send((j, bounds[w], bounds[w + 1], float(state[1][k])))
                a = np.float32(hist[0, k])
                for c in conns:
                    a = np.float32(max(a, np.float32(c.recv())))   # amaxes are >= 0 (no NaN here)
                hist[0, k] = a
            return _oracle_update_48(oracle, np, state)

        state = one_pass(state)                  # warm-up
        passes, t0 = 0, time.perf_counter()
        while True:
            state = one_pass(state)
            passes += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
    finally:
        for c in conns:
            try:
                c.send(None)
            except Exception:
                pass
        for p in procs:
            p.join(timeout=30)
        for m in shms:
            m.close()
            m.unlink()
    return {"value": round(passes * per_pass / dt / 1e9, 4), "unit": UNIT, "cores": workers,
            "kind": "oracle",
            "sample": f"{passes} pass(es) over the same 4-tensor sample + update; each tensor "
                      f"split into {workers} row blocks run by {workers} spawned processes of "
                      f"the C oracle (as it stands); {dt:.1f} s"}


REF_ROWS = 128   # rows of each list tensor per reference step


def run_reference(args):
    """The reference arm: the C oracle, single-threaded, on a bounded sample
    of the headline workload per step -- the first REF_ROWS rows of each of
    the 48 tensors (drawn on the CPU with the list recipe), cast-transposed
    with the current scales, then the 48-column update."""
    import numpy as np
    import torch

    import oracle
    from cast_transpose_gb300 import workloads
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    shapes = tuple((REF_ROWS, c) for _, c in LIST_SHAPES)
    xs = [t.view(torch.int16).numpy().view(np.uint16)
          for t in workloads.multi_list("cpu", shapes=shapes)]
    step_bytes = sum(4 * x.size + 12 for x in xs) + UPDATE_BYTES
    state = (np.zeros((HIST_LEN, LIST_COUNT), np.float32), np.ones(LIST_COUNT, np.float32),
             np.ones(LIST_COUNT, np.float32))

    def step(state):
        hist = state[0]
        for k, x in enumerate(xs):
            r = oracle.cast_transpose(x, float(state[1][k]), oracle.E4M3, amax_in=float(hist[0, k]))
            hist[0, k] = r["amax"]
        return _oracle_update_48(oracle, np, state)

    for _ in range(args.warmup):
        state = step(state)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        state = step(state)
    dt = time.perf_counter() - t0
    value = step_bytes * args.steps / dt / 1e9
    sample = (f"each step: the first {REF_ROWS} rows of each of the 48 list tensors "
              f"({step_bytes / 1e6:.0f} MB of algorithmic bytes) cast+transposed with the "
              f"current scales, then the 48-column update, through the single-threaded C oracle")
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / max(args.steps, 1), 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "dtype_note": "bf16 in, FP8 (E4M3) codes out; the scale product is one fp32 multiply",
        "data": "synthetic (seeded bf16, the 48-tensor list recipe)",
        "config": {"workload": WORKLOAD, "tensors": LIST_COUNT,
                   "shapes": [list(s) for s in LIST_SHAPES], "fp8": "E4M3",
                   "amax_history_len": HIST_LEN, "margin": 0, "parallelism": "host, 1 thread"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
def profile_case(name: str) -> None:
    """Three launches of each kernel on one workload, for a profiler to
    capture, e.g. `ncu --clock-control none -k regex:<kernel> -s 2 -c 1
    python bench.py --profile-case <name>`:
      'activation': cast-transpose of the 16384x12288 activation, E4M3;
      'gradient':   dbias cast-transpose of the 8192x12288 gradient, E5M2
                    (the direct-load kernel and the finish kernel);
      'list':       a 12-tensor list (the four list shapes at half size), then
                    three 48-column scale updates;
      'cast':       cast only of the activation, then three FP8 transposes;
      'general':    cast-transpose of a ragged 8191x12287 matrix whose x
                    starts 2 bytes past a 16-byte boundary and whose q and qT
                    start 1 byte past one (the general cast kernel);
      'shifted':    the same x with aligned q and qT (the flat cast of a
                    shifted x, then the odd-shape transpose);
      'ragged':     cast-transpose of a ragged 8191x12287 matrix (the flat cast
                    kernel, then the FP8 transpose of q), then three FP8
                    transposes of q (the odd-shape transpose kernel);
      'flat':       three plain casts of the ragged 8191x12287 matrix (the flat
                    cast kernel);
      'odd':        cast-transpose of an 8191x12288 matrix (rows % 16 != 0:
                    the direct kernel's odd-row stores);
      'loop':       the same with a noop flag at 0 (the looping grid that calls
                    with a noop flag take);
      'noop':       three launches of the activation cast-transpose with the
                    noop flag set;
      'weight':     three steps of the weight-like 4096x4096 workload (eight
                    casts of x * 2^k with CT_X_READY, each followed by the
                    scale update), the persistent TMA kernel."""
    import torch

    import cast_transpose_gb300 as ct
    from cast_transpose_gb300 import workloads
    dev = torch.device("cuda", 0)
    s1, a0, si0 = (torch.tensor([v], dtype=torch.float32, device=dev) for v in (1.0, 0.0, 0.0))
    if name == "list":
        # 12 tensors, 3 of each list shape at half size in both dimensions (1.2 GB in)
        shapes = tuple((r // 2, c // 2) for r, c in LIST_SHAPES)
        xs = workloads.multi_list(dev, count=12, shapes=shapes, zero=(), tiny=())
        assert sum(x.numel() for x in xs) == PROFILE_LIST_ELEMS
        outs = [ct.empty_outputs(x) for x in xs]
        n = len(xs)
        sc, am, si = (torch.ones(n, device=dev), torch.zeros(n, device=dev), torch.zeros(n, device=dev))
        for _ in range(3):
            ct.fp8_multi_cast_transpose(xs, [sc[i:i + 1] for i in range(n)],
                                        [am[i:i + 1] for i in range(n)],
                                        [si[i:i + 1] for i in range(n)], [o[0] for o in outs],
                                        [o[1] for o in outs], ct.E4M3)
        hist = torch.rand(16, 48, device=dev)
        sc48, rs48 = torch.ones(48, device=dev), torch.ones(48, device=dev)
        for _ in range(3):
            ct.fp8_amax_and_scale_update(hist, sc48, rs48, ct.E4M3, 0)
    elif name == "cast":
        x = workloads.activation_matrix(dev)
        q, qt = ct.empty_outputs(x)
        for _ in range(3):
            ct.fp8_cast(x, s1, a0, si0, q, ct.E4M3)
        for _ in range(3):
            ct.fp8_transpose(q, qt)
    elif name == "general":
        n = 8191 * 12287
        buf = torch.empty(n + 8, dtype=torch.bfloat16, device=dev)
        x = buf[1:1 + n].view(8191, 12287)
        x.copy_(workloads.normal_bf16(8191, 12287, 1.0, 17, dev))
        qbuf = torch.empty(2 * n + 32, dtype=torch.uint8, device=dev)
        q, qt = qbuf[1:1 + n].view(8191, 12287), qbuf[n + 17:2 * n + 17].view(12287, 8191)
        for _ in range(3):
            ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3)
    elif name == "shifted":
        buf = torch.empty(8191 * 12287 + 8, dtype=torch.bfloat16, device=dev)
        x = buf[1:1 + 8191 * 12287].view(8191, 12287)
        x.copy_(workloads.normal_bf16(8191, 12287, 1.0, 17, dev))
        q, qt = ct.empty_outputs(x)
        for _ in range(3):
            ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3)
    elif name == "ragged":
        x = workloads.normal_bf16(8191, 12287, 1.0, 17, dev)
        q, qt = ct.empty_outputs(x)
        for _ in range(3):
            ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3)
        for _ in range(3):
            ct.fp8_transpose(q, qt)
    elif name == "odd":
        x = workloads.normal_bf16(8191, 12288, 1.0, 17, dev)
        q, qt = ct.empty_outputs(x)
        for _ in range(3):
            ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3)
    elif name == "flat":
        x = workloads.normal_bf16(8191, 12287, 1.0, 17, dev)
        q, qt = ct.empty_outputs(x)
        for _ in range(3):
            ct.fp8_cast(x, s1, a0, si0, q, ct.E4M3)
    elif name in ("activation", "loop", "noop"):
        x = workloads.activation_matrix(dev)
        q, qt = ct.empty_outputs(x)
        flag = None if name == "activation" else \
            torch.full((1,), 1.0 if name == "noop" else 0.0, device=dev)
        for _ in range(3):
            ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3, noop_flag=flag)
    elif name == "weight":
        base = workloads.weight_matrix(dev)
        xs = [workloads.weight_rescaled(base, k) for k in workloads.WEIGHT_EXPONENTS]
        outs = [ct.empty_outputs(x) for x in xs]
        hist = torch.zeros(HIST_LEN, 1, device=dev)
        scale, rsinv = torch.ones(1, device=dev), torch.ones(1, device=dev)
        tsinv = torch.zeros(len(xs), device=dev)
        for _ in range(3):
            for k, x in enumerate(xs):
                ct.fp8_cast_transpose(x, scale, hist[0], tsinv[k:k + 1], outs[k][0], outs[k][1],
                                      ct.E4M3, x_ready=True)
                ct.fp8_amax_and_scale_update(hist, scale, rsinv, ct.E4M3, 0)
    elif name == "gradient":
        dy = workloads.gradient_matrix(dev)
        q, qt = ct.empty_outputs(dy)
        db = torch.empty(dy.shape[1], device=dev)
        ws = torch.empty(ct.dbias_workspace_size(*dy.shape), dtype=torch.uint8, device=dev)
        for _ in range(3):
            ct.fp8_dbias_cast_transpose(dy, s1, a0, si0, q, qt, db, ws, ct.E5M2)
    else:
        raise SystemExit(f"unknown profile case {name!r}")
    torch.cuda.synchronize()
    print(f"profile case {name}: 3 launches done")


def _parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra", action=argparse.BooleanOptionalAction, default=True,
                    help="also time the secondary workloads")
    ap.add_argument("--profile-case",
                    choices=["activation", "gradient", "list", "cast", "general", "shifted", "ragged",
                             "flat", "odd",
                             "loop", "noop", "weight"],
                    default=None,
                    help="only run 3 launches of one workload's kernel (for ncu) and exit")
    return ap.parse_args(argv)


def _run(argv):
    args = _parse(argv)
    if args.profile_case:
        profile_case(args.profile_case)
        return
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = _parse(argv)
    world_env = os.environ.get("WORLD_SIZE")
    if args.gpus > 1 and world_env is None:
        if args.impl == "gb300":
            import torch
            have = torch.cuda.device_count()
            if have < args.gpus:
                raise SystemExit(f"--gpus {args.gpus}: only {have} GPU(s) visible")
        spawn_ranks(args.gpus, _run, (argv,))
        return
    if world_env is not None and int(world_env) != args.gpus and args.gpus != 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world_env}")
    _run(argv)


if __name__ == "__main__":
    main()
