"""GPU parity of the deferred scale updates: a run of K
fp8_cast_transpose_pending calls on one history column, then one
fp8_amax_and_scale_update_pending, against the oracle running the sequence
they stand for -- cast k with the current scale, its amax max-merged into
history row 0, then the delayed-scaling update -- K times.  Every cast's q,
qT and scale_inv, and the history, scale and scale_inv after the run, are
compared bit for bit; the pending rows must be zero again.
"""
import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
import oracle
from cast_transpose_gb300 import workloads
from gpu_util import Guarded, f32_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_error():
    ct.device_error(clear=True)
    yield
    assert ct.device_error() == 0


def _history(L, n, seed):
    rng = np.random.default_rng(seed)
    h = (rng.random((L, n)) * 10.0 ** rng.integers(-3, 3, size=(L, n))).astype(np.float32)
    h[0] = 0.0            # what the previous update leaves in row 0
    return h


def _inputs(rows, cols, K, seed, special):
    """K bf16 matrices: one seeded base times 2^e_k, so the amaxes (and the
    scales) change from cast to cast.  `special` puts in an all-zero matrix
    (amax 0: the guard keeps the scale), a tiny one (fp8_max / amax overflows)
    and one holding a NaN."""
    base = workloads.normal_bf16(rows, cols, 1.0, seed)
    exps = [0, 3, -2, 5, 1, -4, 2, 0, 6, -1, 4, -3, 1, 2, -2, 3][:K]
    xs = [(base.float() * 2.0 ** e).to(torch.bfloat16) for e in exps]
    if special and K >= 5:
        xs[1] = torch.zeros_like(base)
        xs[2] = torch.full_like(base, 1e-38)
        nan = base.clone()
        nan[rows // 2, cols // 3] = float("nan")
        xs[4] = nan
    return xs


def _oracle_run(xs, h, s, si, col, fmt, margin, algo):
    """The undeferred sequence on the CPU: per cast, its q / qT / scale_inv."""
    outs = []
    for x in xs:
        ref = oracle.cast_transpose(x, float(s[col]), fmt, amax_in=float(h[0, col]))
        h[0, col] = ref["amax"]
        outs.append(ref)
        h, s, si = oracle.amax_and_scale_update(h, s, si, fmt, margin, algo=algo)
    return outs, h, s, si


def _gpu_run(xs, hd, sd, sid, pend, col, fmt, margin, algo, x_ready):
    rows, cols = xs[0].shape
    res = []
    for k, x in enumerate(xs):
        q, qt = Guarded(rows * cols), Guarded(rows * cols)
        sinv = torch.full((1,), -1.0, device="cuda")
        ct.fp8_cast_transpose_pending(x, hd, sd, pend, col, k, sinv, q.t, qt.t, fmt, margin, algo,
                                      x_ready=x_ready)
        res.append((q, qt, sinv))
    ct.fp8_amax_and_scale_update_pending(hd, sd, sid, pend, fmt, margin, algo)
    torch.cuda.synchronize()
    return res


def _check(res, outs, rows, cols):
    for k, ((q, qt, sinv), ref) in enumerate(zip(res, outs)):
        q.check()
        qt.check()
        assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"]), k
        assert np.array_equal(qt.numpy().reshape(cols, rows), ref["qt"]), k
        assert f32_bits(sinv.item()) == f32_bits(ref["scale_inv"]), k


def _bits(t):
    return t.cpu().numpy().view(np.uint32)


# (rows, cols): 1024 and 2048 tiles (the TMA kernel, which takes deferred-
# update casts of aligned shapes at every size), rows % 16 != 0 and
# cols % 8 != 0 (the general kernel)
SHAPES = [(4096, 4096), (8192, 4096), (1000, 1040), (300, 263)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmt,margin,algo,L,K,n,col", [
    (ct.E4M3, 0, ct.AMAX_MAX, 16, 8, 1, 0),
    (ct.E5M2, 1, ct.AMAX_MAX, 16, 8, 3, 2),
    (ct.E4M3, 0, ct.AMAX_MOST_RECENT, 16, 8, 2, 1),
    (ct.E4M3, 2, ct.AMAX_MAX, 4, 4, 1, 0),       # K = L: c_0 leaves the window
    (ct.E5M2, 0, ct.AMAX_MAX, 40, 6, 2, 0),      # rows shared by every window
])
def test_pending_run_matches_sequential_oracle(shape, fmt, margin, algo, L, K, n, col):
    rows, cols = shape
    xs = _inputs(rows, cols, K, seed=rows + cols + K, special=(L == 16 and algo == ct.AMAX_MAX))
    h = _history(L, n, seed=L * 7 + n)
    s = np.linspace(0.5, 3.0, n).astype(np.float32)
    si = np.zeros(n, np.float32)
    outs, h_ref, s_ref, si_ref = _oracle_run(xs, h.copy(), s.copy(), si.copy(), col, fmt, margin,
                                             algo)
    hd, sd, sid = (torch.from_numpy(a.copy()).cuda() for a in (h, s, si))
    pend = torch.zeros(K, n, device="cuda")
    res = _gpu_run([x.cuda() for x in xs], hd, sd, sid, pend, col, fmt, margin, algo,
                   x_ready=(K % 2 == 0))
    _check(res, outs, rows, cols)
    assert np.array_equal(_bits(hd), h_ref.view(np.uint32))
    assert np.array_equal(_bits(sd), s_ref.view(np.uint32))
    assert np.array_equal(_bits(sid), si_ref.view(np.uint32))
    assert not pend.any()


def test_pending_run_replayed_in_a_graph():
    """The run captured once (8 casts with CT_X_READY, then the update) and
    replayed for three steps: every replay derives its scales from the
    history the previous replay left."""
    rows, cols, K, L = 4096, 4096, 8, 16
    xs_cpu = _inputs(rows, cols, K, seed=11, special=False)
    xs = [x.cuda() for x in xs_cpu]
    h = _history(L, 1, seed=5)
    s = np.array([1.0], np.float32)
    si = np.zeros(1, np.float32)
    hd, sd, sid = (torch.from_numpy(a.copy()).cuda() for a in (h, s, si))
    pend = torch.zeros(K, 1, device="cuda")
    qs = [ct.empty_outputs(x) for x in xs]
    sinvs = torch.zeros(K, device="cuda")

    def run():
        for k, x in enumerate(xs):
            ct.fp8_cast_transpose_pending(x, hd, sd, pend, 0, k, sinvs[k:k + 1], qs[k][0],
                                          qs[k][1], ct.E4M3, x_ready=True)
        ct.fp8_amax_and_scale_update_pending(hd, sd, sid, pend, ct.E4M3)

    run()                      # warm up (and the first step)
    outs, h, s, si = _oracle_run(xs_cpu, h, s, si, 0, ct.E4M3, 0, ct.AMAX_MAX)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side), torch.cuda.graph(g):
        run()
    torch.cuda.current_stream().wait_stream(side)
    for step in range(3):
        g.replay()
        torch.cuda.synchronize()
        outs, h, s, si = _oracle_run(xs_cpu, h, s, si, 0, ct.E4M3, 0, ct.AMAX_MAX)
        for k in (0, 3, K - 1):
            assert np.array_equal(qs[k][0].cpu().numpy(), outs[k]["q"]), (step, k)
            assert np.array_equal(qs[k][1].cpu().numpy(), outs[k]["qt"]), (step, k)
        assert np.array_equal(_bits(sinvs), np.array([o["scale_inv"] for o in outs],
                                                     np.float32).view(np.uint32)), step
        assert np.array_equal(_bits(hd), h.view(np.uint32)), step
        assert np.array_equal(_bits(sd), s.view(np.uint32)), step
        assert np.array_equal(_bits(sid), si.view(np.uint32)), step
        assert not pend.any()


def test_pending_noop_flag_set_writes_nothing():
    rows, cols = 512, 512
    x = workloads.normal_bf16(rows, cols, 1.0, 3, "cuda")
    hd = torch.rand(16, 1, device="cuda")
    sd, sid = torch.ones(1, device="cuda"), torch.zeros(1, device="cuda")
    h0, s0 = hd.clone(), sd.clone()
    pend = torch.zeros(2, 1, device="cuda")
    q, qt = Guarded(rows * cols), Guarded(rows * cols)
    q.t.fill_(0x5A)
    qt.t.fill_(0x5A)
    sinv = torch.full((1,), -1.0, device="cuda")
    flag = torch.ones(1, device="cuda")
    ct.fp8_cast_transpose_pending(x, hd, sd, pend, 0, 1, sinv, q.t, qt.t, noop_flag=flag)
    ct.fp8_amax_and_scale_update_pending(hd, sd, sid, pend, noop_flag=flag)
    torch.cuda.synchronize()
    q.check()
    qt.check()
    assert (q.numpy() == 0x5A).all() and (qt.numpy() == 0x5A).all() and sinv.item() == -1.0
    assert torch.equal(hd, h0) and torch.equal(sd, s0) and sid.item() == 0.0 and not pend.any()
