"""noop_flag and CUDA-graph capture ("[PyTorch] Refactor FP8 workspaces in
linear modules": the transpose kernel must be captured in the graph and
skipped at replay through a noop flag; "[PyTorch] cuda graph support":
transposes made persistent for graph capture).

* every entry point writes nothing when the flag holds a nonzero value;
* the activation workload (16384x12288, 0.5 * Student-t(3), E4M3) captured
  in one torch.cuda.CUDAGraph: replay 1 with flag 0 matches the oracle;
  then the input is overwritten, the flag set to 1 and replay 2 leaves
  every output byte-identical.
"""
import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
import oracle
from cast_transpose_gb300 import workloads
from gpu_util import Guarded, f32_bits, scalar

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_error():
    ct.device_error(clear=True)
    yield
    assert ct.device_error() == 0


def _bytes(t):
    return t.view(torch.uint8).cpu().numpy().copy()


@pytest.mark.parametrize("shape", [(256, 512), (33, 65)])
def test_noop_every_entry_point(shape):
    rows, cols = shape
    x = workloads.normal_bf16(rows, cols, 1.0, 77, "cuda")
    n = rows * cols
    on, off = scalar(1.0), scalar(0.0)
    bufs = {k: Guarded(n) for k in ("q", "qt")}
    db = Guarded(cols, dtype=torch.float32)
    s, a, si = scalar(2.0), scalar(0.0), scalar(-3.0)
    ws = torch.zeros(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    hist = torch.rand(16, 3, device="cuda")
    sc, sci = torch.ones(3, device="cuda"), torch.ones(3, device="cuda")
    tq = Guarded(n)
    state = lambda: [_bytes(b.buf) for b in (bufs["q"], bufs["qt"], db, tq)] + \
        [_bytes(t) for t in (a, si, hist, sc, sci)]
    before = state()
    ct.fp8_cast_transpose(x, s, a, si, bufs["q"].t, bufs["qt"].t, ct.E4M3, noop_flag=on)
    ct.fp8_cast(x, s, a, si, bufs["q"].t, ct.E4M3, noop_flag=on)
    ct.fp8_dbias_cast_transpose(x, s, a, si, bufs["q"].t, bufs["qt"].t, db.t, ws, ct.E5M2,
                                noop_flag=on)
    ct.fp8_multi_cast_transpose([x], [s], [a], [si], [bufs["q"].t], [bufs["qt"].t], ct.E4M3,
                                noop_flag=on)
    ct.fp8_amax_and_scale_update(hist, sc, sci, ct.E4M3, 0, noop_flag=on)
    ct.fp8_transpose(bufs["q"].t.view(rows, cols), tq.t, noop_flag=on)
    torch.cuda.synchronize()
    after = state()
    for b0, b1 in zip(before, after):
        assert np.array_equal(b0, b1)
    # and with the flag at 0 the same call does write
    ct.fp8_cast_transpose(x, s, a, si, bufs["q"].t, bufs["qt"].t, ct.E4M3, noop_flag=off)
    torch.cuda.synchronize()
    ref = oracle.cast_transpose(x.cpu(), 2.0, ct.E4M3)
    assert np.array_equal(bufs["q"].numpy().reshape(rows, cols), ref["q"])
    assert f32_bits(si.item()) == f32_bits(ref["scale_inv"])


def test_activation_graph_replay_with_noop():
    x = workloads.activation_matrix("cuda")
    rows, cols = x.shape
    x_cpu = x.cpu()
    q, qt = ct.empty_outputs(x)
    scale, amax, sinv = scalar(1.0), scalar(0.0), scalar(0.0)
    flag = scalar(0.0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):        # warm-up outside the graph
        ct.fp8_cast_transpose(x, scale, amax, sinv, q, qt, ct.E4M3, noop_flag=flag)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    q.fill_(0)
    qt.fill_(0)
    amax.zero_()
    sinv.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ct.fp8_cast_transpose(x, scale, amax, sinv, q, qt, ct.E4M3, noop_flag=flag)
    torch.cuda.synchronize()
    assert int(q.sum()) == 0 and int(qt.sum()) == 0     # capture itself ran nothing

    g.replay()                            # replay 1: flag 0, transpose computed
    torch.cuda.synchronize()
    ref = oracle.cast_transpose(x_cpu, 1.0, ct.E4M3)
    assert np.array_equal(q.cpu().numpy(), ref["q"])
    assert np.array_equal(qt.cpu().numpy(), ref["qt"])
    assert f32_bits(amax.item()) == f32_bits(ref["amax"])
    assert sinv.item() == 1.0

    snap = [_bytes(t) for t in (q, qt, amax, sinv)]
    x.copy_(workloads.normal_bf16(rows, cols, 3.0, 5, "cuda"))   # new input
    flag.fill_(1.0)
    g.replay()                            # replay 2: flag 1, cached transpose kept
    torch.cuda.synchronize()
    for before, t in zip(snap, (q, qt, amax, sinv)):
        assert np.array_equal(before, _bytes(t))
