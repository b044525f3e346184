"""Failure detection without a GPU fault, and CUDA-graph capture of every
entry point.

* The kernels' mbarrier waits are bounded.  ct_selftest_bounded_wait runs the
  same bounded wait on a barrier nothing completes: it must give up after
  its short limit, mark the device diagnostic word, and leave the context
  usable (a cast right after it is still bit-exact).
* Every entry point can be recorded in a torch.cuda.CUDAGraph and replayed,
  with the noop flag ("[PyTorch] Refactor FP8 workspaces in linear modules":
  the transpose kernel captured, then skipped at replay) switching the
  recorded work off: replay 1 (flag 0) matches the oracle, replay 2 (flag 1,
  new input) leaves every output byte unchanged.
"""
import time

import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
import oracle
from cast_transpose_gb300 import workloads
from gpu_util import dbias_tolerance_ok, f32_bits, scalar

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    ct.device_error(clear=True)
    t0 = time.perf_counter()
    ct.selftest_bounded_wait(20000)            # 20 ms on a barrier nobody arrives at
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert ct.device_error() & 2, "the bounded wait did not report its timeout"
    assert 0.015 < elapsed < 5.0
    assert ct.device_error(clear=True) & 1 == 0  # no kernel wait timed out
    assert ct.device_error() == 0
    x = workloads.normal_bf16(256, 384, 1.0, 31)
    q, qt = ct.empty_outputs(x.cuda())
    a, si = scalar(0.0), scalar(0.0)
    ct.fp8_cast_transpose(x.cuda(), scalar(1.0), a, si, q, qt, ct.E4M3)
    torch.cuda.synchronize()
    ref = oracle.cast_transpose(x, 1.0, ct.E4M3)
    assert np.array_equal(q.cpu().numpy(), ref["q"])
    assert ct.device_error() == 0


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                                   # warm-up outside the graph
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _bytes(ts):
    return [t.view(torch.uint8).cpu().numpy().copy() for t in ts]


def test_graph_dbias_cast_transpose_with_noop():
    ct.device_error(clear=True)
    rows, cols = 2048, 1536
    dy = workloads.gradient_matrix("cuda", rows, cols)
    q, qt = ct.empty_outputs(dy)
    db = torch.empty(cols, device="cuda")
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    s, a, si, flag = scalar(1.0), scalar(0.0), scalar(0.0), scalar(0.0)
    g = _capture(lambda: ct.fp8_dbias_cast_transpose(dy, s, a, si, q, qt, db, ws, ct.E5M2,
                                                     noop_flag=flag))
    a.zero_()
    g.replay()
    torch.cuda.synchronize()
    x_cpu = dy.cpu()
    ref = oracle.cast_transpose(x_cpu, 1.0, ct.E5M2)
    assert np.array_equal(q.cpu().numpy(), ref["q"]) and np.array_equal(qt.cpu().numpy(), ref["qt"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    assert dbias_tolerance_ok(db.cpu().numpy(), oracle.dbias(x_cpu), x_cpu)
    snap = _bytes([q, qt, db, a, si])
    dy.copy_(workloads.normal_bf16(rows, cols, 7.0, 3, "cuda"))
    flag.fill_(1.0)
    g.replay()
    torch.cuda.synchronize()
    for b0, b1 in zip(snap, _bytes([q, qt, db, a, si])):
        assert np.array_equal(b0, b1)
    assert ct.device_error() == 0


def test_graph_multi_update_transpose_with_noop():
    ct.device_error(clear=True)
    shapes = [(512, 768), (1024, 256), (96, 1040)]
    xs = [workloads.normal_bf16(r, c, 2.0, 60 + i, "cuda") for i, (r, c) in enumerate(shapes)]
    n = len(xs)
    L = 8
    hist = torch.zeros(L, n, device="cuda")
    scales = torch.tensor([1.0, 2.0, 0.5], device="cuda")
    rsi = torch.ones(n, device="cuda")
    tsi = torch.zeros(n, device="cuda")
    outs = [ct.empty_outputs(x) for x in xs]
    t_again = torch.empty(shapes[0][0] * shapes[0][1], dtype=torch.uint8, device="cuda")
    flag = scalar(0.0)

    def step():
        ct.fp8_multi_cast_transpose(xs, [scales[i:i + 1] for i in range(n)],
                                    [hist[0, i:i + 1] for i in range(n)],
                                    [tsi[i:i + 1] for i in range(n)], [o[0] for o in outs],
                                    [o[1] for o in outs], ct.E4M3, noop_flag=flag)
        ct.fp8_transpose(outs[0][0].view(shapes[0]), t_again, noop_flag=flag)
        ct.fp8_amax_and_scale_update(hist, scales, rsi, ct.E4M3, 0, noop_flag=flag)

    g = _capture(step)          # the warm-up ran one step eagerly
    h = np.zeros((L, n), np.float32)
    sc = np.array([1.0, 2.0, 0.5], np.float32)
    si = np.ones(n, np.float32)

    def oracle_step(h, sc, si):
        for i, x in enumerate(xs):
            r = oracle.cast_transpose(x.cpu(), float(sc[i]), ct.E4M3)
            h[0, i] = r["amax"]
        return oracle.amax_and_scale_update(h, sc, si, ct.E4M3, 0)

    h, sc, si = oracle_step(h, sc, si)          # the eager warm-up step
    g.replay()
    torch.cuda.synchronize()
    last = [oracle.cast_transpose(x.cpu(), float(sc[i]), ct.E4M3) for i, x in enumerate(xs)]
    h, sc, si = oracle_step(h, sc, si)
    for i, x in enumerate(xs):
        assert np.array_equal(outs[i][0].cpu().numpy(), last[i]["q"]), i
        assert np.array_equal(outs[i][1].cpu().numpy(), last[i]["qt"]), i
    assert np.array_equal(t_again.cpu().numpy(), last[0]["qt"].reshape(-1))
    assert np.array_equal(hist.cpu().numpy().view(np.uint32), h.view(np.uint32))
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), sc.view(np.uint32))
    snap = _bytes([hist, scales, rsi, tsi, t_again] + [t for o in outs for t in o])
    for x in xs:
        x.mul_(3.0)
    flag.fill_(1.0)
    g.replay()
    torch.cuda.synchronize()
    after = _bytes([hist, scales, rsi, tsi, t_again] + [t for o in outs for t in o])
    for b0, b1 in zip(snap, after):
        assert np.array_equal(b0, b1)
    assert ct.device_error() == 0


def test_concurrent_calls_from_two_threads_on_two_streams():
    """The library keeps no per-call state: two host threads casting different
    tensors on their own streams at the same time both get exact results."""
    import threading
    xs_cpu = [workloads.normal_bf16(4096, 2048, 1.0 + i, 900 + i) for i in range(2)]
    xs = [x.cuda() for x in xs_cpu]
    res = [None, None]
    errs = []

    def work(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                q, qt = ct.empty_outputs(xs[i])
                a, si = scalar(0.0), scalar(0.0)
                for _ in range(20):
                    a.zero_()
                    ct.fp8_cast_transpose(xs[i], scalar(0.5 * (i + 1)), a, si, q, qt,
                                          ct.E4M3 if i == 0 else ct.E5M2)
                st.synchronize()
                res[i] = (q.cpu().numpy(), qt.cpu().numpy(), a.item())
        except Exception as e:      # surfaced below
            errs.append(e)

    ts = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    for i in range(2):
        ref = oracle.cast_transpose(xs_cpu[i], 0.5 * (i + 1), ct.E4M3 if i == 0 else ct.E5M2)
        assert np.array_equal(res[i][0], ref["q"]) and np.array_equal(res[i][1], ref["qt"])
        assert f32_bits(res[i][2]) == f32_bits(ref["amax"])
