"""fp8_dbias_cast_transpose_noalloc: the dbias cast-transpose for callers
that cannot allocate device memory where they call it (code inside an
allocator or memory-pool callback, where allocating again would recurse or
deadlock, or a runtime that has reserved all device memory up front).
Instead of a caller workspace it uses a fixed scratch array that the library
keeps on the GPU.

Checked through the C ABI on two calls in a row with different inputs (the
shared scratch keeps the previous call's contents, which must not leak into
the next one), against both the oracle and fp8_dbias_cast_transpose with a
normal workspace: FP8 data, transpose, amax and scale_inv bit-exact, db
within the dbias tolerance of the other tests.  This file sorts last so that
a run stopping at its first failure has run everything else before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
import oracle
from cast_transpose_gb300 import workloads
from gpu_util import Guarded, dbias_tolerance_ok, f32_bits, scalar
from oracle_pool import OraclePool

pytestmark = pytest.mark.gpu

CT_OK, CT_ERR_WORKSPACE = 0, 7


def _noalloc_fn():
    fn = ct.lib().fp8_dbias_cast_transpose_noalloc
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp, vp, i32, vp, vp]
    fn.restype = i32
    return fn


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _run_noalloc(dy, scale, fmt):
    rows, cols = dy.shape
    n = rows * cols
    q, qt = Guarded(n), Guarded(n)
    db = Guarded(cols, dtype=torch.float32)
    s, a, si = scalar(scale), scalar(0.0), scalar(0.0)
    st = _noalloc_fn()(dy.data_ptr(), rows, cols, s.data_ptr(), a.data_ptr(), si.data_ptr(),
                       q.t.data_ptr(), qt.t.data_ptr(), db.t.data_ptr(), fmt, None, _stream())
    assert st == CT_OK, ct.lib().ct_status_string(st)
    torch.cuda.synchronize()
    for g in (q, qt, db):
        g.check()
    return {"q": q.numpy(), "qt": qt.numpy(), "db": db.numpy(), "amax": a.item(),
            "scale_inv": si.item()}


def _run_with_workspace(dy, scale, fmt):
    rows, cols = dy.shape
    q, qt = ct.empty_outputs(dy)
    db = torch.empty(cols, device="cuda")
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    s, a, si = scalar(scale), scalar(0.0), scalar(0.0)
    ct.fp8_dbias_cast_transpose(dy, s, a, si, q, qt, db, ws, fmt)
    torch.cuda.synchronize()
    return {"q": q.cpu().numpy().reshape(-1), "qt": qt.cpu().numpy().reshape(-1),
            "db": db.cpu().numpy(), "amax": a.item(), "scale_inv": si.item()}


@pytest.mark.parametrize("shape,fmt", [((2048, 4096), ct.E5M2), ((1000, 1030), ct.E4M3),
                                       ((8192, 16384), ct.E5M2)])   # the largest it accepts
def test_noalloc_matches_oracle_and_workspace_version_twice(shape, fmt):
    ct.device_error(clear=True)
    rows, cols = shape
    inputs = [workloads.gradient_matrix("cuda", rows, cols, std=1e-3, outlier_fraction=1e-3),
              workloads.normal_bf16(rows, cols, 2.0, 4242, "cuda")]
    with OraclePool() as pool:
        for call, dy in enumerate(inputs):            # two calls in a row, different data
            got = _run_noalloc(dy, 1.5, fmt)
            dy_cpu = dy.cpu()
            # the oracle: every byte of q and qT, amax, scale_inv, db
            xin = pool.input_bf16(rows, cols)
            xin[:] = dy_cpu.view(torch.int16).numpy().view(np.uint16)
            q, qt = pool.output_q(rows, cols), pool.output_qt(rows, cols)
            q[:] = got["q"].reshape(rows, cols)
            qt[:] = got["qt"].reshape(cols, rows)
            res = pool.check_cast_transpose(rows, cols, 1.5, fmt)
            del xin, q, qt
            assert res["bad_q"] == 0, (call, "FP8 data differs from the oracle", res["first_q"])
            assert res["bad_qt"] == 0, (call, "transpose differs from the oracle", res["first_qt"])
            assert f32_bits(got["amax"]) == f32_bits(res["amax"])
            sinv_ref = oracle.cast_transpose(dy_cpu[:1], 1.5, fmt)["scale_inv"]
            assert f32_bits(got["scale_inv"]) == f32_bits(sinv_ref)
            assert dbias_tolerance_ok(got["db"], oracle.dbias(dy_cpu), dy_cpu), \
                f"call {call}: db outside the tolerance of the oracle's column sums"
            # the entry point with a caller workspace: the same bytes, db within tolerance
            ref = _run_with_workspace(dy, 1.5, fmt)
            assert np.array_equal(got["q"], ref["q"]), f"call {call}: FP8 data differs"
            assert np.array_equal(got["qt"], ref["qt"]), f"call {call}: transpose differs"
            assert f32_bits(got["amax"]) == f32_bits(ref["amax"])
            assert f32_bits(got["scale_inv"]) == f32_bits(ref["scale_inv"])
            assert dbias_tolerance_ok(got["db"], ref["db"], dy_cpu), f"call {call}: db differs"
    assert ct.device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    fn = _noalloc_fn()
    # ceil(8320/128) * 16384 partials * 4 bytes > 4 MiB: refused before any launch
    fake = 0x10000000
    st = fn(fake, 8320, 16384, fake * 2, fake * 3, fake * 4, fake * 5, fake * 6, fake * 7,
            ct.E5M2, None, None)
    assert st == CT_ERR_WORKSPACE
    # the largest shape it accepts: 8192 x 16384
    assert ct.dbias_workspace_size(8192, 16384) <= 4 << 20 < ct.dbias_workspace_size(8320, 16384)
