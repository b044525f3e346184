"""Full-size parity of the ragged shapes the benchmark times, each through the
path it takes: every byte of q and qT against the oracle (rows split over
spawned oracle processes on all host cores).

  * 8191 x 12287 cast-transpose: the flat cast, then the odd-shape FP8
    transpose of q;
  * 8191 x 12288 cast-transpose: the direct kernel's odd-row variant (whole
    aligned qT blocks with a halo from the tile above);
  * 8191 x 12287 and 8191 x 12288 cast-transposes of an x 2 and 14 bytes
    past a 16-byte boundary: the flat cast of a shifted x, then the odd-shape
    transpose;
  * 8191 x 12287 FP8 transpose of an existing q, and of a q that starts at an
    odd byte, written to a qT at an odd byte.

Smaller cases (against the single-process oracle) cover row ends off the
direct kernel's alignment, and the flat cast + transpose from one wave of
tiles of the looping launch (q stored evict-last, tiles in reverse order),
with and without a noop flag at 0.
"""
import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
from cast_transpose_gb300 import workloads
import oracle
from gpu_util import Guarded, f32_bits, scalar
from oracle_pool import OraclePool

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_error():
    ct.device_error(clear=True)
    yield
    assert ct.device_error() == 0


@pytest.mark.parametrize("shape,fmt,x_shift", [((8191, 12287), ct.E4M3, 0),
                                               ((8191, 12288), ct.E5M2, 0),
                                               ((8191, 12287), ct.E4M3, 1),
                                               ((8191, 12288), ct.E5M2, 7)])
def test_ragged_cast_transpose_in_full(shape, fmt, x_shift):
    """x_shift: x starts that many bf16 elements past a 16-byte boundary (the
    flat cast then shifts every chunk by the same byte offset)."""
    rows, cols = shape
    x = workloads.normal_bf16(rows, cols, 1.0, 17 + cols, "cuda")
    n = rows * cols
    if x_shift:
        big = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
        big[x_shift:x_shift + n] = x.reshape(-1)
        x = big[x_shift:x_shift + n].view(rows, cols)
    q, qt = Guarded(n), Guarded(n)
    s, a, si = scalar(1.75), scalar(0.0), scalar(-1.0)
    ct.fp8_cast_transpose(x, s, a, si, q.t, qt.t, fmt)
    torch.cuda.synchronize()
    q.check()
    qt.check()
    with OraclePool() as pool:
        xin = pool.input_bf16(rows, cols)
        xin[:] = x.cpu().view(torch.int16).numpy().view(np.uint16)
        qv = pool.output_q(rows, cols)
        qv[:] = q.numpy().reshape(rows, cols)
        qtv = pool.output_qt(rows, cols)
        qtv[:] = qt.numpy().reshape(cols, rows)
        res = pool.check_cast_transpose(rows, cols, 1.75, fmt, check_qt=True)
        del xin, qv, qtv
    assert res["bad_q"] == 0, ("FP8 data differs from the oracle", res["first_q"])
    assert res["bad_qt"] == 0, ("transpose differs from the oracle", res["first_qt"])
    assert f32_bits(a.item()) == f32_bits(res["amax"])
    assert f32_bits(si.item()) == f32_bits(np.float32(1.0) / np.float32(1.75))


@pytest.mark.parametrize("in_off,out_off", [(0, 0), (5, 11)])
def test_odd_shape_fp8_transpose_in_full(in_off, out_off):
    """The transpose is a byte permutation: qT must be exactly q's transpose."""
    rows, cols = 8191, 12287
    n = rows * cols
    g = torch.Generator(device="cuda").manual_seed(23)
    src = Guarded(n, offset=in_off)
    src.t.copy_(torch.randint(0, 256, (n,), dtype=torch.int32, device="cuda", generator=g)
                .to(torch.uint8))
    dst = Guarded(n, offset=out_off)
    ct.fp8_transpose(src.t.view(rows, cols), dst.t.view(cols, rows))
    torch.cuda.synchronize()
    src.check()
    dst.check()
    q = src.numpy().reshape(rows, cols)
    assert np.array_equal(dst.numpy().reshape(cols, rows), q.T)


@pytest.mark.parametrize("shape", [(280, 250), (131, 255), (33, 127), (145, 383), (301, 263)])
@pytest.mark.parametrize("x_shift,out_off", [(0, 10), (3, 0), (7, 15), (0, 1)])
def test_ragged_kernel_row_ends(shape, x_shift, out_off):
    """rows % 16 != 0 off the direct kernel's alignment (x off 16 bytes, or q
    and qT at odd bytes; the general kernel, or the flat cast and the
    odd-shape transpose), on shapes whose last column tile is nearly full:
    every row end, at q offsets that put it anywhere in its 16-byte block."""
    rows, cols = shape
    x_cpu = workloads.normal_bf16(rows, cols, 3.0, rows * 7 + cols)
    n = rows * cols
    big = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
    big[x_shift:x_shift + n] = x_cpu.reshape(-1).cuda()
    x = big[x_shift:x_shift + n].view(rows, cols)
    q, qt = Guarded(n, offset=out_off), Guarded(n, offset=out_off)
    s, a, si = scalar(0.625), scalar(0.0), scalar(-1.0)
    ct.fp8_cast_transpose(x, s, a, si, q.t, qt.t, ct.E4M3)
    torch.cuda.synchronize()
    q.check()
    qt.check()
    ref = oracle.cast_transpose(x_cpu, 0.625, ct.E4M3)
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    assert np.array_equal(qt.numpy().reshape(cols, rows), ref["qt"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    assert f32_bits(si.item()) == f32_bits(ref["scale_inv"])


@pytest.mark.parametrize("flag", [None, 0.0])
@pytest.mark.parametrize("shape", [(2000, 5003), (1937, 9731)])
def test_flat_cast_then_transpose_from_one_wave(shape, flag):
    """Shapes of 640 and 1232 tiles: the flat cast stores q with the L2
    evict-last priority and the looping transpose launch takes the tiles from
    the last one back, demoting the lines it stages; with no noop flag and
    with one at 0.  Every byte of q and qT against the oracle."""
    rows, cols = shape
    x_cpu = workloads.normal_bf16(rows, cols, 4.0, rows + cols)
    n = rows * cols
    q, qt = Guarded(n), Guarded(n)
    s, a, si = scalar(0.8125), scalar(0.0), scalar(-1.0)
    noop = None if flag is None else torch.full((1,), flag, device="cuda")
    ct.fp8_cast_transpose(x_cpu.cuda(), s, a, si, q.t, qt.t, ct.E4M3, noop_flag=noop)
    torch.cuda.synchronize()
    q.check()
    qt.check()
    ref = oracle.cast_transpose(x_cpu, 0.8125, ct.E4M3)
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    assert np.array_equal(qt.numpy().reshape(cols, rows), ref["qt"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    assert f32_bits(si.item()) == f32_bits(ref["scale_inv"])
