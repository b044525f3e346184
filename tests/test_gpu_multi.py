"""GPU parity of fp8_multi_cast_transpose (one launch over a tensor list).

Every list is compared in full.  The 48-tensor list (12 each of 6144x12288,
12288x6144, 18432x6144, 6144x24576, N(0, 0.02), two all-zero and two
rescaled to max|x| = 1e-30) is compared byte for byte, q and qT of every
tensor, with the oracle run on every host core (tests/oracle_pool.py); its
amaxes, scale-inverses and the 48-column scale update (zero-amax guard) are
compared exactly.
"""
import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
import oracle
from cast_transpose_gb300 import workloads
from gpu_util import Guarded, f32_bits
from oracle_pool import OraclePool

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_error():
    ct.device_error(clear=True)
    yield
    assert ct.device_error() == 0


def _run_list(xs, scales_val, fmt, misalign=()):
    n = len(xs)
    scales = torch.tensor(scales_val, dtype=torch.float32, device="cuda")
    amax = torch.zeros(n, device="cuda")
    sinv = torch.zeros(n, device="cuda")
    outs, outs_t = [], []
    for i, x in enumerate(xs):
        m = x.numel()
        outs.append(Guarded(m, offset=1 if i in misalign else 0))
        outs_t.append(Guarded(m))
    ct.fp8_multi_cast_transpose(xs, [scales[i:i + 1] for i in range(n)],
                                [amax[i:i + 1] for i in range(n)],
                                [sinv[i:i + 1] for i in range(n)],
                                [o.t for o in outs], [o.t for o in outs_t], fmt)
    torch.cuda.synchronize()
    return outs, outs_t, amax.cpu().numpy(), sinv.cpu().numpy()


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
def test_small_mixed_list(fmt):
    shapes = [(256, 384), (33, 65), (128, 128), (0, 16), (144, 272), (1, 1), (4096, 16),
              (16, 4096)]
    xs_cpu = [workloads.normal_bf16(r, c, 40.0, 50 + i) for i, (r, c) in enumerate(shapes)]
    scales = [1.0, 0.5, 2.0, 1.0, 3.0, 1.0, 0.25, 8.0]
    outs, outs_t, amax, sinv = _run_list([x.cuda() for x in xs_cpu], scales, fmt, misalign=(2,))
    for i, x in enumerate(xs_cpu):
        r, c = x.shape
        outs[i].check()
        outs_t[i].check()
        if x.numel() == 0:
            assert amax[i] == 0.0 and sinv[i] == 0.0
            continue
        ref = oracle.cast_transpose(x, scales[i], fmt)
        assert np.array_equal(outs[i].numpy().reshape(r, c), ref["q"]), i
        assert np.array_equal(outs_t[i].numpy().reshape(c, r), ref["qt"]), i
        assert f32_bits(amax[i]) == f32_bits(ref["amax"]), i
        assert f32_bits(sinv[i]) == f32_bits(ref["scale_inv"]), i


def test_list_longer_than_one_launch():
    xs_cpu = [workloads.normal_bf16(16 * (1 + i % 5), 32 * (1 + i % 3), 1.0, 300 + i)
              for i in range(70)]
    scales = [float(1 + i % 4) for i in range(70)]
    outs, outs_t, amax, sinv = _run_list([x.cuda() for x in xs_cpu], scales, ct.E4M3)
    for i, x in enumerate(xs_cpu):
        r, c = x.shape
        ref = oracle.cast_transpose(x, scales[i], ct.E4M3)
        assert np.array_equal(outs[i].numpy().reshape(r, c), ref["q"]), i
        assert np.array_equal(outs_t[i].numpy().reshape(c, r), ref["qt"]), i
        assert f32_bits(amax[i]) == f32_bits(ref["amax"]), i


def test_multi_48_tensor_list_with_update():
    """The whole 48-tensor list (4.98e9 elements) against the oracle: every
    byte of every q and qT, every amax, scale_inv, and the 48-column update."""
    n = workloads.MULTI_COUNT
    xs = workloads.multi_list("cuda")
    scales = torch.ones(n, device="cuda")
    L = 16
    hist = torch.zeros(L, n, device="cuda")
    tsinv = torch.zeros(n, device="cuda")
    outs = [torch.empty(x.numel(), dtype=torch.uint8, device="cuda") for x in xs]
    outs_t = [torch.empty(x.numel(), dtype=torch.uint8, device="cuda") for x in xs]
    ct.fp8_multi_cast_transpose(xs, [scales[i:i + 1] for i in range(n)],
                                [hist[0, i:i + 1] for i in range(n)],
                                [tsinv[i:i + 1] for i in range(n)], outs, outs_t, ct.E4M3)
    amax_gpu = hist[0].cpu().numpy().copy()
    recipe_sinv = torch.ones(n, device="cuda")
    ct.fp8_amax_and_scale_update(hist, scales, recipe_sinv, ct.E4M3, 0)
    torch.cuda.synchronize()

    amax_ref = np.zeros(n, np.float32)
    with OraclePool() as pool:
        for i, x in enumerate(xs):
            r, c = x.shape
            xin = pool.input_bf16(r, c)
            torch.from_numpy(xin.view(np.int16)).copy_(x.view(torch.int16))
            q, qt = pool.output_q(r, c), pool.output_qt(r, c)
            torch.from_numpy(q).copy_(outs[i].view(r, c))
            torch.from_numpy(qt).copy_(outs_t[i].view(c, r))
            res = pool.check_cast_transpose(r, c, 1.0, ct.E4M3)
            del xin, q, qt
            assert res["bad_q"] == 0, (i, res["bad_q"], "q bytes differ, first at", res["first_q"])
            assert res["bad_qt"] == 0, (i, res["bad_qt"], "qT bytes differ, first at",
                                        res["first_qt"])
            amax_ref[i] = res["amax"]
            assert f32_bits(amax_gpu[i]) == f32_bits(amax_ref[i]), (i, amax_gpu[i], amax_ref[i])
            assert tsinv[i].item() == 1.0
    assert np.all(amax_ref[list(workloads.MULTI_ZERO)] == 0.0)
    tiny = amax_ref[list(workloads.MULTI_TINY)]
    assert np.all((tiny > 0) & (tiny < 1.1e-30))

    h_ref = np.zeros((L, n), np.float32)
    h_ref[0] = amax_ref
    h_ref, s_ref, si_ref = oracle.amax_and_scale_update(h_ref, np.ones(n, np.float32),
                                                        np.ones(n, np.float32), ct.E4M3, 0)
    assert np.array_equal(hist.cpu().numpy(), h_ref)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(recipe_sinv.cpu().numpy().view(np.uint32), si_ref.view(np.uint32))
    assert np.all(s_ref[list(workloads.MULTI_ZERO)] == 1.0)     # amax 0: scale kept


def test_per_tensor_formats_in_one_launch():
    """fp8_multi_cast_transpose_ex: E4M3 and E5M2 entries mixed in one list
    (TMA-path and general-path shapes)."""
    shapes = [(256, 384), (512, 128), (33, 65), (1024, 1040), (128, 4096), (96, 96)]
    fmts = [ct.E4M3, ct.E5M2, ct.E5M2, ct.E4M3, ct.E5M2, ct.E4M3]
    xs_cpu = [workloads.normal_bf16(r, c, 300.0, 700 + i) for i, (r, c) in enumerate(shapes)]
    n = len(xs_cpu)
    scales = torch.tensor([1.0, 4.0, 0.5, 2.0, 8.0, 1.0], device="cuda")
    amax = torch.zeros(n, device="cuda")
    sinv = torch.zeros(n, device="cuda")
    outs = [Guarded(x.numel()) for x in xs_cpu]
    outs_t = [Guarded(x.numel()) for x in xs_cpu]
    ct.fp8_multi_cast_transpose_ex([x.cuda() for x in xs_cpu], [scales[i:i + 1] for i in range(n)],
                                   [amax[i:i + 1] for i in range(n)],
                                   [sinv[i:i + 1] for i in range(n)], [o.t for o in outs],
                                   [o.t for o in outs_t], fmts)
    torch.cuda.synchronize()
    a, si = amax.cpu().numpy(), sinv.cpu().numpy()
    for i, x in enumerate(xs_cpu):
        r, c = x.shape
        outs[i].check()
        outs_t[i].check()
        ref = oracle.cast_transpose(x, float(scales[i].item()), fmts[i])
        assert np.array_equal(outs[i].numpy().reshape(r, c), ref["q"]), i
        assert np.array_equal(outs_t[i].numpy().reshape(c, r), ref["qt"]), i
        assert f32_bits(a[i]) == f32_bits(ref["amax"]), i
        assert f32_bits(si[i]) == f32_bits(ref["scale_inv"]), i
