"""GPU parity of the general kernel (any shape, any alignment) against the
oracle, bit-exact.  It is reached by every shape whose rows or cols are not
multiples of 16 and by every buffer that is not 16-byte aligned.  The cases
drive each of its load forms (one aligned 16-byte block, two covering blocks
shifted by every even byte offset, element by element at the ends of x) and
each store form (16-, 8-, 4-, 2- and 1-byte aligned q chunks and qT blocks,
full and partial), with and without dbias.
"""
import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
import oracle
from cast_transpose_gb300 import workloads
from gpu_util import Guarded, assert_same_cast, cast_transpose_gpu, dbias_tolerance_ok, f32_bits, scalar

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_error():
    ct.device_error(clear=True)
    yield
    assert ct.device_error() == 0


def _shifted(x_cpu, elems):
    """x on the GPU at an offset of `elems` bf16 elements (2 bytes each) from
    a 256-byte-aligned allocation."""
    n = x_cpu.numel()
    big = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
    big[elems:elems + n] = x_cpu.reshape(-1).cuda()
    return big[elems:elems + n].view(x_cpu.shape)


@pytest.mark.parametrize("x_shift", range(8))
@pytest.mark.parametrize("shape", [(160, 264), (131, 257), (256, 136), (64, 1000)])
def test_x_offsets(shape, x_shift):
    rows, cols = shape
    x_cpu = workloads.normal_bf16(rows, cols, 20.0, 3000 + rows + cols + x_shift)
    x = _shifted(x_cpu, x_shift)
    got = cast_transpose_gpu(x, 1.5, ct.E4M3, amax_in=0.25)
    assert_same_cast(got, oracle.cast_transpose(x_cpu, 1.5, ct.E4M3, amax_in=0.25))


@pytest.mark.parametrize("out_offset", [1, 2, 3, 4, 5, 6, 8, 12])
@pytest.mark.parametrize("shape", [(272, 384), (257, 130)])
def test_output_offsets(shape, out_offset):
    rows, cols = shape
    x_cpu = workloads.normal_bf16(rows, cols, 5.0, 77 + out_offset)
    got = cast_transpose_gpu(x_cpu.cuda(), 0.75, ct.E5M2, out_offset=out_offset)
    assert_same_cast(got, oracle.cast_transpose(x_cpu, 0.75, ct.E5M2))


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
@pytest.mark.parametrize("shape", [(1031, 2053), (4099, 777), (129, 16385)])
def test_ragged_larger(fmt, shape):
    rows, cols = shape
    x_cpu = workloads.normal_bf16(rows, cols, 80.0, 11 + rows)
    got = cast_transpose_gpu(_shifted(x_cpu, 3), 2.0, fmt)
    assert_same_cast(got, oracle.cast_transpose(x_cpu, 2.0, fmt))


@pytest.mark.parametrize("x_shift", [1, 4])
def test_dbias_misaligned(x_shift):
    rows, cols = 1000, 771
    x_cpu = workloads.gradient_matrix("cpu", rows, cols, std=1e-2, outlier_fraction=1e-3)
    dy = _shifted(x_cpu, x_shift)
    n = rows * cols
    q, qt = Guarded(n, offset=3), Guarded(n, offset=1)
    db = Guarded(cols, dtype=torch.float32)
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    ws.fill_(0x7F)
    s, a, si = scalar(3.0), scalar(0.0), scalar(0.0)
    ct.fp8_dbias_cast_transpose(dy, s, a, si, q.t, qt.t, db.t, ws, ct.E5M2)
    torch.cuda.synchronize()
    for g in (q, qt, db):
        g.check()
    ref = oracle.cast_transpose(x_cpu, 3.0, ct.E5M2)
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    assert np.array_equal(qt.numpy().reshape(cols, rows), ref["qt"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    assert dbias_tolerance_ok(db.numpy(), oracle.dbias(x_cpu), x_cpu)


def test_cast_only_misaligned():
    rows, cols = 333, 555
    x_cpu = workloads.normal_bf16(rows, cols, 9.0, 5)
    q = Guarded(rows * cols, offset=7)
    s, a, si = scalar(1.25), scalar(0.0), scalar(0.0)
    ct.fp8_cast(_shifted(x_cpu, 5), s, a, si, q.t, ct.E4M3)
    torch.cuda.synchronize()
    q.check()
    ref = oracle.cast_transpose(x_cpu, 1.25, ct.E4M3, want_qt=False)
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    assert f32_bits(si.item()) == f32_bits(ref["scale_inv"])


def test_single_row_and_column_misaligned():
    for shape in [(1, 4099), (4099, 1), (2, 2), (1, 9)]:
        x_cpu = workloads.normal_bf16(*shape, 1.0, shape[0] * 7 + shape[1])
        got = cast_transpose_gpu(_shifted(x_cpu, 1), 1.0, ct.E4M3, out_offset=3)
        assert_same_cast(got, oracle.cast_transpose(x_cpu, 1.0, ct.E4M3))


@pytest.mark.parametrize("in_shift", [0, 1, 3, 7, 8, 13])
@pytest.mark.parametrize("shape", [(131, 257), (256, 200), (1031, 2053)])
def test_fp8_transpose_general(shape, in_shift):
    """fp8_transpose on shapes / offsets outside the 16-byte fast path: every
    byte offset class of the input, outputs at odd offsets."""
    rows, cols = shape
    g = torch.Generator().manual_seed(rows + 7 * cols + in_shift)
    q_cpu = torch.randint(0, 256, (rows, cols), dtype=torch.uint8, generator=g)
    big = torch.empty(rows * cols + 32, dtype=torch.uint8, device="cuda")
    big[in_shift:in_shift + rows * cols] = q_cpu.reshape(-1).cuda()
    out = Guarded(rows * cols, offset=(in_shift * 5) % 16)
    ct.fp8_transpose(big[in_shift:in_shift + rows * cols].view(rows, cols), out.t)
    torch.cuda.synchronize()
    out.check()
    assert np.array_equal(out.numpy().reshape(cols, rows), oracle.fp8_transpose(q_cpu.numpy()))


def test_random_shapes_offsets_and_paths():
    """A seeded sweep of 200 cases: rows and cols in [1, 700] (multiples of 8 and
    16 drawn often, so every kernel is reached), x shifted by 0..7 elements,
    q and qT by 0..15 bytes, both formats, a random scale: the full outputs
    of the cast-transpose and the dbias variant against the oracle."""
    rng = np.random.default_rng(20261202)
    for case in range(200):
        pick = rng.integers(0, 3, size=2)
        rows = int([rng.integers(1, 701), 16 * rng.integers(1, 44), 8 * rng.integers(1, 88)][pick[0]])
        cols = int([rng.integers(1, 701), 16 * rng.integers(1, 44), 8 * rng.integers(1, 88)][pick[1]])
        x_shift = int(rng.integers(0, 8)) if rng.random() < 0.5 else 0
        out_shift = int(rng.integers(0, 16)) if rng.random() < 0.5 else 0
        fmt = int(rng.integers(0, 2))
        scale = float(np.float32(2.0 ** rng.uniform(-6, 6)))
        x_cpu = workloads.normal_bf16(rows, cols, float(rng.uniform(0.1, 100)), 9000 + case)
        x = _shifted(x_cpu, x_shift)
        got = cast_transpose_gpu(x, scale, fmt, out_offset=out_shift)
        ref = oracle.cast_transpose(x_cpu, scale, fmt)
        assert_same_cast(got, ref)
        n = rows * cols
        q, qt = Guarded(n, offset=out_shift), Guarded(n, offset=out_shift)
        db = Guarded(cols, dtype=torch.float32)
        ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
        ct.fp8_dbias_cast_transpose(x, scalar(scale), scalar(0.0), scalar(0.0), q.t, qt.t, db.t, ws,
                                    fmt)
        torch.cuda.synchronize()
        for g in (q, qt, db):
            g.check()
        assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"]), (case, rows, cols)
        assert np.array_equal(qt.numpy().reshape(cols, rows), ref["qt"]), (case, rows, cols)
        assert dbias_tolerance_ok(db.numpy(), oracle.dbias(x_cpu), x_cpu), (case, rows, cols)
