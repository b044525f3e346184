"""Benchmark of the FP8 cast-transpose hot path on GB300.

Workload (one "step"): the weight-like bf16 4096x4096 matrix, N(0, 0.02),
rescaled by 2^k for k = -4..3 (eight distinct resident copies); for each k
one E4M3 cast + transpose + amax (fp8_cast_transpose, writing into the
current amax-history slot) followed by one delayed-scaling update
(fp8_amax_and_scale_update, history length 16, margin 0).  The step is
captured once in a CUDA graph and replayed; inputs are resident in HBM and
the eight inputs plus eight output pairs (512 MB) exceed the 129 MB L2, so
every cast streams from DRAM.

Metric: algorithmic GB/s (bytes read + written by the path, 4 bytes per
element for a cast-transpose plus the scalars) and its fraction of the
measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

--impl reference times the CPU oracle (plain single-threaded C) on a bounded
sample of the same workload.  Under torchrun (N > 1) every rank runs an
independent replica (the path has no exchange step), the slowest rank's
time counts, and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "cast-transpose GB/s (bytes read+written) and % of GB300 HBM peak"
UNIT = "GB/s"
ROWS, COLS = 4096, 4096
HIST_LEN = 16
EXPONENTS = tuple(range(-4, 4))
CAST_BYTES = 4 * ROWS * COLS + 12           # bf16 in, FP8 data + transpose out, scale/amax/scale_inv
UPDATE_BYTES = (2 * HIST_LEN + 3) * 4       # history read + rolled write, scale, scale_inv
STEP_BYTES = len(EXPONENTS) * (CAST_BYTES + UPDATE_BYTES)
WORKLOAD = ("weight-like bf16 4096x4096 N(0,0.02) x 2^k, k=-4..3: per step 8 x (E4M3 "
            "cast+transpose+amax, then amax-history/scale update, L=16, margin 0)")
KERNEL_SOURCES = ["cast_transpose_gb300/csrc/ct_fast.cu", "cast_transpose_gb300/csrc/ct_device.cuh"]


def _peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "source": "fallback"}


def _kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic_per_launch():
    """dram read+write bytes per cast-transpose launch of this workload, from
    the committed ncu summary, if it was taken on the current kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
        e = d.get("fast_cast_transpose_kernel 4096x4096 E4M3")
        if e and e.get("kernel_source_sha") == _kernel_hash():
            return int(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
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
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
def run_gpu(args):
    import torch

    import cast_transpose_gb300 as ct
    from cast_transpose_gb300 import workloads

    world, rank, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = _peaks()

    base = workloads.weight_matrix(dev)
    xs = [workloads.weight_rescaled(base, k) for k in EXPONENTS]
    del base
    outs = [ct.empty_outputs(x) for x in xs]
    hist = torch.zeros(HIST_LEN, 1, device=dev)
    scale = torch.ones(1, device=dev)
    recipe_sinv = torch.ones(1, device=dev)
    tensor_sinv = torch.zeros(len(xs), device=dev)

    # CT_X_READY (x_ready=True): each cast follows the scale update, which
    # writes only fp32 scalars, and the inputs were written before the timed
    # region (or, end to end, by copies the compute stream waits for), so the
    # cast may load its first tiles while the update finishes.  The step on
    # the default path is timed too, after the timed region.
    def step(x_ready=True):
        for k, x in enumerate(xs):
            ct.fp8_cast_transpose(x, scale, hist[0], tensor_sinv[k:k + 1], outs[k][0], outs[k][1],
                                  ct.E4M3, x_ready=x_ready)
            ct.fp8_amax_and_scale_update(hist, scale, recipe_sinv, ct.E4M3, 0)

    # eager warm-up (first call per device sets kernel attributes), then capture
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step()
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()

    # Kernel timing inside the timed region.  Extra captures of the step
    # carry external event-record nodes on a side branch: after each kernel
    # the side stream joins the main one and records an event, so the event
    # fires when that kernel completes without holding back the next kernel
    # (which depends on the kernel only, through its programmatic edge).  The
    # span between consecutive events is each kernel's share of the critical
    # path; the spans of one replay add up to the whole step.  Every 8th
    # replay of the timed loop uses one of these copies; after the loop each
    # copy's events hold the times of its last replay.
    plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(plain):
        step()
    n_evented, every = 8, 8
    evented, kevs = [], []
    for _ in range(n_evented):
        try:
            ev = [torch.cuda.Event(enable_timing=True, external=True)
                  for _ in range(1 + 2 * len(xs))]
        except TypeError:      # torch without external events: no per-kernel times
            break
        side = torch.cuda.Stream(device=dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            main = torch.cuda.current_stream()
            side.wait_stream(main)
            with torch.cuda.stream(side):
                ev[0].record()
            for k, x in enumerate(xs):
                ct.fp8_cast_transpose(x, scale, hist[0], tensor_sinv[k:k + 1], outs[k][0],
                                      outs[k][1], ct.E4M3, x_ready=True)
                side.wait_stream(main)
                with torch.cuda.stream(side):
                    ev[1 + 2 * k].record()
                ct.fp8_amax_and_scale_update(hist, scale, recipe_sinv, ct.E4M3, 0)
                side.wait_stream(main)
                with torch.cuda.stream(side):
                    ev[2 + 2 * k].record()
            main.wait_stream(side)
        evented.append(g)
        kevs.append(ev)
    launches_per_step = 2 * len(xs)

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
    cast_ms, upd_ms, step_ev_ms = [], [], []
    for j in used:
        ev = kevs[j]
        cast_ms += [ev[2 * k].elapsed_time(ev[1 + 2 * k]) for k in range(len(xs))]
        upd_ms += [ev[1 + 2 * k].elapsed_time(ev[2 + 2 * k]) for k in range(len(xs))]
        step_ev_ms.append(ev[0].elapsed_time(ev[-1]))
    ms_per_step = _max_over_ranks(elapsed_ms / args.steps, world)

    # ---- end to end: host buffers in, host results out, public API calls ----
    # Every step copies its 8 inputs in from pinned host memory, runs the
    # step through the public API (eager calls) and copies the FP8 data, the
    # transposes and the scales back out.  Two device buffer sets and separate
    # streams for copy-in (two), compute and copy-out (two) let step i+1's
    # copy-in overlap step i's copy-out and keep several copy engines busy;
    # events order each buffer set's reuse.
    e2e_steps = max(3, min(args.steps, 200))
    host_in = [x.cpu().pin_memory() for x in xs]
    host_q = [torch.empty(o[0].shape, dtype=torch.uint8).pin_memory() for o in outs]
    host_qt = [torch.empty(o[1].shape, dtype=torch.uint8).pin_memory() for o in outs]
    host_scale = torch.empty(2, dtype=torch.float32).pin_memory()
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = sum(h.numel() for h in host_q) + sum(h.numel() for h in host_qt) + 8
    sets = [(xs, outs), ([torch.empty_like(x) for x in xs], [ct.empty_outputs(x) for x in xs])]
    n_copy = 2                                   # copy streams per direction
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
        for c, st in enumerate(s_in):
            with torch.cuda.stream(st):
                st.wait_event(ev_comp[b])        # step i-2 no longer reads these inputs
                for k in range(c, len(xs), n_copy):
                    bx[k].copy_(host_in[k], non_blocking=True)
                ev_in[b][c].record(st)
        with torch.cuda.stream(s_comp):
            for c in range(n_copy):
                s_comp.wait_event(ev_in[b][c])
                s_comp.wait_event(ev_out[b][c])  # step i-2's outputs have been copied out
            for k in range(len(xs)):
                ct.fp8_cast_transpose(bx[k], scale, hist[0], tensor_sinv[k:k + 1], bo[k][0],
                                      bo[k][1], ct.E4M3, x_ready=True)
                ct.fp8_amax_and_scale_update(hist, scale, recipe_sinv, ct.E4M3, 0)
            ev_comp[b].record(s_comp)
        for c, st in enumerate(s_out):
            with torch.cuda.stream(st):
                st.wait_event(ev_comp[b])
                for k in range(c, len(xs), n_copy):
                    host_q[k].copy_(bo[k][0], non_blocking=True)
                    host_qt[k].copy_(bo[k][1], non_blocking=True)
                if c == 0:
                    host_scale[0:1].copy_(scale, non_blocking=True)
                    host_scale[1:2].copy_(recipe_sinv, non_blocking=True)
                ev_out[b][c].record(st)

    def joined(streams):
        for st in streams:
            torch.cuda.current_stream().wait_stream(st)

    for i in range(2):
        e2e_step(i)
    joined((*s_in, s_comp, *s_out))
    torch.cuda.synchronize()
    _barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for st in (*s_in, s_comp, *s_out):
        st.wait_stream(torch.cuda.current_stream())
    for i in range(e2e_steps):
        e2e_step(i)
    joined((*s_in, s_comp, *s_out))
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)

    # The same step with every cast on the default path (no CT_X_READY: the
    # cast reads nothing of x before the update before it has completed),
    # after the timed region.
    default_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(default_graph):
        step(x_ready=False)
    for _ in range(3):
        default_graph.replay()
    torch.cuda.synchronize()
    n_default = max(3, min(args.steps, 200))
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    d0.record()
    for _ in range(n_default):
        default_graph.replay()
    d1.record()
    torch.cuda.synchronize()
    default_ms = _max_over_ranks(d0.elapsed_time(d1) / n_default, world)

    if rank != 0:
        return
    value = world * STEP_BYTES / (ms_per_step * 1e-3) / 1e9
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
        "data": "synthetic (seeded N(0,0.02) bf16, resident in HBM)",
        "config": {
            "workload": WORKLOAD,
            "shape": [ROWS, COLS],
            "fp8": "E4M3",
            "amax_history_len": HIST_LEN,
            "margin": 0,
            "bytes_per_step": STEP_BYTES,
            "cuda_graph": True,
            "l2": "inputs larger than L2: 8 distinct 32 MB inputs + 8 output pairs = 512 MB "
                  "working set per step vs 129 MB L2, each cast reads an input last touched "
                  "7 casts earlier",
            "parallelism": f"replicas x{world}",
            "pct_of_nominal_8000_gbs": round(100 * value / world / 8000.0, 1),
        },
        "gpu_launches": args.steps * launches_per_step,
        "x_ready": {
            "used": True,
            "why": "every cast is called with CT_X_READY: the kernel before it in the stream is "
                   "the scale update (fp32 scalars only) and the inputs were written before the "
                   "timed region (end to end: by copies the compute stream waits for), so the "
                   "cast may load its first tiles while the update finishes",
            "default_path_ms_per_step": round(default_ms, 6),
            "default_path_value": round(world * STEP_BYTES / (default_ms * 1e-3) / 1e9, 1),
            "default_path_steps": n_default,
        },
        "e2e": {
            "value": round(world * STEP_BYTES / (e2e_ms * 1e-3) / 1e9, 1),
            "unit": UNIT,
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "steps": e2e_steps,
            "ms_per_step": round(e2e_ms, 4),
            "note": "every step: its 8 inputs copied in from pinned host memory, the step "
                    "through the public API (eager calls), FP8 data + transposes + scales copied "
                    "out; copy-in (2 streams) / compute / copy-out (2 streams) with two buffer "
                    "sets, so step i+1's copy-in overlaps step i's copy-out",
        },
        "clocks": clocks,
    }
    if cast_ms:
        avg = statistics.mean(cast_ms)
        achieved = CAST_BYTES / (avg * 1e-3) / 1e9
        line["roofline"] = {
            "kernel": "fast_cast_transpose_kernel (fp8_cast_transpose, 4096x4096 E4M3)",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "peak_source": peaks["source"] + " copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
            "traffic": _traffic_per_launch(),
            "algorithmic_bytes_per_launch": CAST_BYTES,
            "avg_launch_us": round(avg * 1e3, 3),
            "launches_timed": len(cast_ms),
            "timing": "external CUDA event-record nodes on a side branch of the step graph, "
                      "one after each kernel (span = the kernel's share of the critical path); "
                      "evented copies replace every 8th replay of the timed loop, the last "
                      "replay of each copy is read",
            "share_of_step": round(sum(cast_ms) / max(sum(step_ev_ms), 1e-12), 4),
            "update_kernel_avg_us": round(statistics.mean(upd_ms) * 1e3, 3) if upd_ms else None,
            "evented_step_us": round(statistics.mean(step_ev_ms) * 1e3, 2) if step_ev_ms else None,
        }
    else:
        line["roofline"] = None
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(seconds=args.cpu_seconds)
    if args.extra:
        line["extra_kernels"] = extra_kernels(dev, peaks)
    print(json.dumps(line))


# ---------------------------------------------------------------------------
def _oracle_step_sample(xs_bits, state, rows_sample):
    """One bounded sample of a step through the CPU oracle: the first
    `rows_sample` rows of each of the 8 inputs cast+transposed with the
    current scale, then the update."""
    import numpy as np

    import oracle
    hist, scale, sinv = state
    for x in xs_bits:
        r = oracle.cast_transpose(x[:rows_sample], float(scale[0]), oracle.E4M3,
                                  amax_in=float(hist[0, 0]))
        hist[0, 0] = r["amax"]
        hist, scale, sinv = oracle.amax_and_scale_update(hist, scale, sinv, oracle.E4M3, 0)
    return (hist, scale, sinv), len(xs_bits) * (4 * rows_sample * COLS + 12 + UPDATE_BYTES)


def _oracle_inputs():
    import numpy as np
    import torch

    from cast_transpose_gb300 import workloads
    base = workloads.weight_matrix("cpu")
    return [workloads.weight_rescaled(base, k).view(torch.int16).numpy().view(np.uint16)
            for k in EXPONENTS]


def cpu_baseline(seconds: float = 10.0) -> dict:
    import numpy as np
    xs = _oracle_inputs()
    state = (np.zeros((HIST_LEN, 1), np.float32), np.ones(1, np.float32), np.ones(1, np.float32))
    done, t0 = 0, time.perf_counter()
    steps = 0
    while True:
        state, b = _oracle_step_sample(xs, state, ROWS)
        done += b
        steps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(done / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{steps} full step(s) of the workload (8 x 4096x4096 cast+transpose+amax "
                      f"+ update) through the single-threaded C oracle, {dt:.1f} s, on "
                      f"{os.cpu_count()} host cores (1 used)"}


def _oracle_rows_worker(shm_name, n_inputs, conn):
    """Spawned worker of cpu_baseline_all_cores: attaches the shared inputs,
    then casts the row blocks it is sent with the oracle as it stands and
    answers each with the block's amax."""
    from multiprocessing import shared_memory

    import numpy as np

    import oracle
    shm = shared_memory.SharedMemory(name=shm_name)
    try:
        xs = np.ndarray((n_inputs, ROWS, COLS), dtype=np.uint16, buffer=shm.buf)
        conn.send("ready")
        while True:
            msg = conn.recv()
            if msg is None:
                break
            k, r0, r1, scale = msg
            r = oracle.cast_transpose(xs[k, r0:r1], scale, oracle.E4M3)
            conn.send(float(r["amax"]))
        del xs
    finally:
        shm.close()


def cpu_baseline_all_cores(seconds: float = 10.0) -> dict:
    """The oracle on every host core: each cast of the step is split into
    row blocks, one per spawned worker process (the oracle's code as it
    stands, run on a block of rows); the amaxes are merged and the update run
    in this process before the next cast, which needs its scale."""
    import multiprocessing as mp
    from multiprocessing import shared_memory

    import numpy as np

    import oracle
    xs = _oracle_inputs()
    n = len(xs)
    workers = max(1, os.cpu_count() or 1)
    shm = shared_memory.SharedMemory(create=True, size=n * ROWS * COLS * 2)
    procs, conns = [], []
    try:
        shared = np.ndarray((n, ROWS, COLS), dtype=np.uint16, buffer=shm.buf)
        shared[:] = np.stack(xs)
        ctx = mp.get_context("spawn")
        for _ in range(workers):
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_rows_worker, args=(shm.name, n, b), daemon=True)
            p.start()
            procs.append(p)
            conns.append(a)
        for c in conns:
            if not c.poll(300) or c.recv() != "ready":
                raise RuntimeError("oracle worker did not start")
        bounds = [ROWS * w // workers for w in range(workers + 1)]
        hist = np.zeros((HIST_LEN, 1), np.float32)
        scale, sinv = np.ones(1, np.float32), np.ones(1, np.float32)

        def step():
            nonlocal hist, scale, sinv
            for k in range(n):
                for w, c in enumerate(conns):
                    c.send((k, bounds[w], bounds[w + 1], float(scale[0])))
                a = np.float32(hist[0, 0])
                for c in conns:
                    a = np.float32(max(a, np.float32(c.recv())))   # amaxes are >= 0 (no NaN here)
                hist[0, 0] = a
                hist, scale, sinv = oracle.amax_and_scale_update(hist, scale, sinv, oracle.E4M3, 0)

        step()                                   # warm-up
        steps, t0 = 0, time.perf_counter()
        while True:
            step()
            steps += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
        del shared
    finally:
        for c in conns:
            try:
                c.send(None)
            except Exception:
                pass
        for p in procs:
            p.join(timeout=30)
        shm.close()
        shm.unlink()
    return {"value": round(steps * STEP_BYTES / dt / 1e9, 4), "unit": UNIT, "cores": workers,
            "kind": "oracle",
            "sample": f"{steps} full step(s) of the workload; each of the 8 casts split into "
                      f"{workers} row blocks run by {workers} spawned processes of the C oracle "
                      f"(as it stands), the update in between; {dt:.1f} s"}


def run_reference(args):
    import numpy as np
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    rows_sample = 64            # each step: 8 x 64x4096 slices, a few ms of oracle work
    xs = _oracle_inputs()
    state = (np.zeros((HIST_LEN, 1), np.float32), np.ones(1, np.float32), np.ones(1, np.float32))
    for _ in range(args.warmup):
        state, _ = _oracle_step_sample(xs, state, rows_sample)
    done, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        state, b = _oracle_step_sample(xs, state, rows_sample)
        done += b
    dt = time.perf_counter() - t0
    value = done / dt / 1e9
    sample = (f"each step: the first {rows_sample} rows of each of the 8 inputs (8 x "
              f"{rows_sample}x4096 cast+transpose+amax + 8 updates) through the "
              f"single-threaded C oracle")
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
        "data": "synthetic (seeded N(0,0.02) bf16)",
        "config": {"workload": WORKLOAD, "shape": [ROWS, COLS], "fp8": "E4M3",
                   "amax_history_len": HIST_LEN, "margin": 0, "parallelism": "host, 1 thread"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


# ---------------------------------------------------------------------------
def extra_kernels(dev, peaks) -> dict:
    """Sustained throughput of the other kernels on their own workloads
    (inputs larger than L2): CUDA-graph-captured back-to-back launches, CUDA
    events around each replay; per launch the median ("us", "GB/s") and the
    best replay ("us_best")."""
    import torch

    import cast_transpose_gb300 as ct
    from cast_transpose_gb300 import workloads

    bests = []   # best per-launch time of each timed() call, in call order

    def timed(fn, iters=10, per_graph=10):
        """Median per-launch time of `per_graph` back-to-back calls captured
        in one CUDA graph (sustained rate, as inside a training step); the
        best replay is kept in `bests`."""
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
        bests.append(min(ms))
        return statistics.median(ms)

    res = {}
    s1, a0, si0 = (torch.tensor([v], dtype=torch.float32, device=dev) for v in (1.0, 0.0, 0.0))
    # activation 16384x12288, E4M3 cast-transpose
    x = workloads.activation_matrix(dev)
    q, qt = ct.empty_outputs(x)
    ms = timed(lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3))
    b = 4 * x.numel() + 12
    res["cast_transpose 16384x12288 E4M3"] = {"us": round(ms * 1e3, 2), "GB/s": round(b / ms / 1e6, 1),
                                               "frac": round(b / ms / 1e6 / peaks["hbm_gbs"], 4),
                                               "kernel": "direct_cast_transpose_kernel"}
    del x, q, qt
    # gradient 8192x12288, dbias + E5M2
    dy = workloads.gradient_matrix(dev)
    q, qt = ct.empty_outputs(dy)
    db = torch.empty(dy.shape[1], device=dev)
    ws = torch.empty(ct.dbias_workspace_size(*dy.shape), dtype=torch.uint8, device=dev)
    ms = timed(lambda: ct.fp8_dbias_cast_transpose(dy, s1, a0, si0, q, qt, db, ws, ct.E5M2))
    b = 4 * dy.numel() + 4 * dy.shape[1] + 12
    res["dbias_cast_transpose 8192x12288 E5M2"] = {"us": round(ms * 1e3, 2),
                                                    "GB/s": round(b / ms / 1e6, 1),
                                                    "frac": round(b / ms / 1e6 / peaks["hbm_gbs"], 4),
                                                    "kernel": "direct_cast_transpose_kernel + dbias_finish_kernel"}
    del dy, q, qt
    # 48-tensor list, one multi launch
    xs = workloads.multi_list(dev)
    outs = [ct.empty_outputs(x) for x in xs]
    n = len(xs)
    sc, am, si = (torch.ones(n, device=dev), torch.zeros(n, device=dev), torch.zeros(n, device=dev))
    args = ([sc[i:i + 1] for i in range(n)], [am[i:i + 1] for i in range(n)],
            [si[i:i + 1] for i in range(n)], [o[0] for o in outs], [o[1] for o in outs])
    ms = timed(lambda: ct.fp8_multi_cast_transpose(xs, *args, ct.E4M3), iters=3, per_graph=2)
    b = sum(4 * x.numel() + 12 for x in xs)
    res["multi_cast_transpose 48 tensors E4M3"] = {"us": round(ms * 1e3, 2),
                                                    "GB/s": round(b / ms / 1e6, 1),
                                                    "frac": round(b / ms / 1e6 / peaks["hbm_gbs"], 4),
                                                    "kernel": "direct_cast_transpose_kernel (list)"}
    # the 48-column update that follows the list (latency-bound: microseconds)
    hist = torch.rand(16, n, device=dev)
    rs = torch.ones(n, device=dev)
    ms = timed(lambda: ct.fp8_amax_and_scale_update(hist, sc, rs, ct.E4M3, 0))
    res["amax_and_scale_update n=48 L=16"] = {"us": round(ms * 1e3, 2),
                                              "kernel": "scale_update_warp_kernel"}
    del xs, outs, args
    # the small 256x512 matrix (launch-bound: microseconds)
    x = workloads.single_matrix(dev)
    q, qt = ct.empty_outputs(x)
    ms = timed(lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3), iters=10, per_graph=50)
    res["cast_transpose 256x512 E4M3"] = {"us": round(ms * 1e3, 2), "kernel": "fast_cast_transpose_kernel"}
    ms = timed(lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3, x_ready=True), iters=10,
               per_graph=50)
    res["cast_transpose 256x512 E4M3, CT_X_READY"] = {"us": round(ms * 1e3, 2),
                                                      "kernel": "fast_cast_transpose_kernel"}
    # activation: cast only (3 B/element), the gated launch with the flag set, FP8 byte transpose
    x = workloads.activation_matrix(dev)
    q, qt = ct.empty_outputs(x)
    ms = timed(lambda: ct.fp8_cast(x, s1, a0, si0, q, ct.E4M3))
    b = 3 * x.numel() + 12
    res["cast 16384x12288 E4M3"] = {"us": round(ms * 1e3, 2), "GB/s": round(b / ms / 1e6, 1),
                                    "frac": round(b / ms / 1e6 / peaks["hbm_gbs"], 4),
                                    "kernel": "direct_cast_transpose_kernel (cast only)"}
    flag = torch.ones(1, device=dev)
    ms = timed(lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3, noop_flag=flag),
               per_graph=50)
    res["cast_transpose 16384x12288, noop flag set"] = {"us": round(ms * 1e3, 2)}
    ms = timed(lambda: ct.fp8_transpose(q, qt))
    b = 2 * x.numel()
    res["transpose 16384x12288 FP8"] = {"us": round(ms * 1e3, 2), "GB/s": round(b / ms / 1e6, 1),
                                        "frac": round(b / ms / 1e6 / peaks["hbm_gbs"], 4),
                                        "kernel": "transpose_fast_kernel"}
    del x, q, qt
    # a ragged shape (odd rows and cols): the general kernel
    x = workloads.normal_bf16(8191, 12287, 1.0, 17, dev)
    q, qt = ct.empty_outputs(x)
    ms = timed(lambda: ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3))
    b = 4 * x.numel() + 12
    res["cast_transpose 8191x12287 E4M3 (ragged)"] = {"us": round(ms * 1e3, 2),
                                                      "GB/s": round(b / ms / 1e6, 1),
                                                      "frac": round(b / ms / 1e6 / peaks["hbm_gbs"], 4),
                                                      "kernel": "general_cast_kernel"}
    assert len(bests) == len(res)   # one timed() call per entry, in the same order
    for entry, best in zip(res.values(), bests):
        entry["us_best"] = round(best * 1e3, 2)
    return res


def profile_case(name: str) -> None:
    """Three launches of each kernel on one workload, for a profiler to
    capture (ncu -k regex:<kernel> -s 2 -c 1):
      'activation': cast-transpose of the 16384x12288 activation, E4M3;
      'gradient':   dbias cast-transpose of the 8192x12288 gradient, E5M2
                    (the direct-load kernel and the finish kernel);
      'list':       a 12-tensor list (the four list shapes at half size), then
                    three 48-column scale updates;
      'cast':       cast only of the activation, then three FP8 transposes;
      'general':    cast-transpose of a ragged 8191x12287 matrix, then three
                    FP8 transposes of its q (the general kernels)."""
    import torch

    import cast_transpose_gb300 as ct
    from cast_transpose_gb300 import workloads
    dev = torch.device("cuda", 0)
    s1, a0, si0 = (torch.tensor([v], dtype=torch.float32, device=dev) for v in (1.0, 0.0, 0.0))
    if name == "list":
        # 12 tensors, 3 of each list shape at half size in both dimensions (1.2 GB in)
        shapes = tuple((r // 2, c // 2) for r, c in workloads.MULTI_SHAPES)
        xs = workloads.multi_list(dev, count=12, shapes=shapes, zero=(), tiny=())
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
        # ragged: neither dimension a multiple of 16 (the general kernel)
        x = workloads.normal_bf16(8191, 12287, 1.0, 17, dev)
        q, qt = ct.empty_outputs(x)
        for _ in range(3):
            ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3)
        for _ in range(3):
            ct.fp8_transpose(q, qt)
    elif name == "activation":
        x = workloads.activation_matrix(dev)
        q, qt = ct.empty_outputs(x)
        for _ in range(3):
            ct.fp8_cast_transpose(x, s1, a0, si0, q, qt, ct.E4M3)
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra", action=argparse.BooleanOptionalAction, default=True,
                    help="also time the dbias, multi-tensor and activation workloads")
    ap.add_argument("--profile-case", choices=["activation", "gradient", "list", "cast", "general"],
                    default=None,
                    help="only run 3 launches of one workload's kernel (for ncu) and exit")
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args.profile_case)
        return
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
