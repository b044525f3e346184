"""GPU parity of fp8_dbias_cast_transpose against the CPU oracle.

FP8 bytes, transpose, amax and scale_inv bit-exact; db within
|db - db_ref| <= 1e-5 * sum_i |dy[i, j]| + 1e-6 (db_ref accumulated in
double by the oracle).  Includes the 8192x12288 gradient-like dy (N(0, 1e-3)
with 0.01% +-5.0 outliers, E5M2) for two steps: scale 1, then the scale
the update derives from the first step's amax.
"""
import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
import oracle
from cast_transpose_gb300 import workloads
from gpu_util import Guarded, dbias_tolerance_ok, f32_bits, scalar

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_error():
    ct.device_error(clear=True)
    yield
    assert ct.device_error() == 0


def run_dbias(dy, scale, fmt, amax_in=0.0):
    rows, cols = dy.shape
    n = rows * cols
    q, qt = Guarded(n), Guarded(n)
    db = Guarded(cols, dtype=torch.float32)
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    ws.fill_(0x7F)   # garbage: the kernel must not depend on its contents
    s, a, si = scalar(scale), scalar(amax_in), scalar(0.0)
    ct.fp8_dbias_cast_transpose(dy, s, a, si, q.t, qt.t, db.t, ws, fmt)
    torch.cuda.synchronize()
    for g in (q, qt, db):
        g.check()
    return {"q": q.numpy().reshape(rows, cols), "qt": qt.numpy().reshape(cols, rows),
            "db": db.numpy(), "amax": a.item(), "scale_inv": si.item()}


def check(got, x_cpu, scale, fmt, amax_in=0.0):
    ref = oracle.cast_transpose(x_cpu, scale, fmt, amax_in=amax_in)
    assert np.array_equal(got["q"], ref["q"]), "FP8 data differs"
    assert np.array_equal(got["qt"], ref["qt"]), "transpose differs"
    assert f32_bits(got["amax"]) == f32_bits(ref["amax"])
    assert f32_bits(got["scale_inv"]) == f32_bits(ref["scale_inv"])
    db_ref = oracle.dbias(x_cpu)
    assert dbias_tolerance_ok(got["db"], db_ref, x_cpu), \
        np.max(np.abs(got["db"] - db_ref))
    return ref


SHAPES = [(1, 1), (3, 17), (128, 128), (127, 129), (129, 256), (1000, 48), (2048, 272),
          (4112, 1040), (131072, 256), (131000, 33)]


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes(fmt, shape):
    rows, cols = shape
    x_cpu = workloads.gradient_matrix("cpu", rows, cols, std=1e-3, outlier_fraction=1e-3)
    check(run_dbias(x_cpu.cuda(), 1.0, fmt), x_cpu, 1.0, fmt)


def test_deterministic():
    x = workloads.gradient_matrix("cuda", 2048, 1024)
    a = run_dbias(x, 1.0, ct.E5M2)
    b = run_dbias(x, 1.0, ct.E5M2)
    assert np.array_equal(a["db"].view(np.uint32), b["db"].view(np.uint32))


def test_gradient_8192x12288_two_steps():
    dy = workloads.gradient_matrix("cuda")
    x_cpu = dy.cpu()
    assert int((x_cpu.float().abs() == 5.0).sum()) == round(1e-4 * dy.numel())
    got = run_dbias(dy, 1.0, ct.E5M2)
    ref = check(got, x_cpu, 1.0, ct.E5M2)
    assert ref["amax"] == 5.0
    # second step with the scale the update derives (57344 / 5)
    hist = np.zeros((16, 1), np.float32)
    hist[0, 0] = ref["amax"]
    _, s, _ = oracle.amax_and_scale_update(hist, np.ones(1, np.float32), np.ones(1, np.float32),
                                           ct.E5M2, 0)
    got2 = run_dbias(dy, float(s[0]), ct.E5M2)
    check(got2, x_cpu, float(s[0]), ct.E5M2)


def _bf16_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def dbias_bf16_tolerance_ok(db_bits, x_cpu) -> bool:
    """bf16 db: the fp32 bound widened by the bf16 rounding (half a bf16 ulp,
    at most 2^-8 of the value): |db - ref| <= T + 2^-8 (|ref| + T), with
    T = 1e-5 * sum_i |dy[i, j]| + 1e-6 and ref the oracle's double sum."""
    ref = oracle.dbias(x_cpu).astype(np.float64)
    t = 1e-5 * x_cpu.double().abs().sum(dim=0).numpy() + 1e-6
    got = _bf16_to_f32(db_bits).astype(np.float64)
    return bool(np.all(np.abs(got - ref) <= t + 2.0 ** -8 * (np.abs(ref) + t)))


@pytest.mark.parametrize("shape,x_shift", [((2048, 272), 0), ((4112, 8208), 0), ((1000, 771), 1),
                                           ((131072, 256), 0)])
def test_bf16_db(shape, x_shift):
    """CT_DBIAS_BF16 on the TMA, direct and general paths: FP8 outputs
    bit-exact, db within the bf16 bound, and equal to the oracle's bf16 db
    on at least 99% of the columns (the rest sit on a bf16 rounding edge)."""
    rows, cols = shape
    x_cpu = workloads.gradient_matrix("cpu", rows, cols, std=1e-3, outlier_fraction=1e-3)
    big = torch.empty(rows * cols + 8, dtype=torch.bfloat16, device="cuda")
    big[x_shift:x_shift + rows * cols] = x_cpu.reshape(-1).cuda()
    dy = big[x_shift:x_shift + rows * cols].view(rows, cols)
    n = rows * cols
    q, qt = Guarded(n), Guarded(n)
    db = Guarded(cols, dtype=torch.bfloat16)
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    ws.fill_(0x7F)
    s, a, si = scalar(2.0), scalar(0.0), scalar(0.0)
    ct.fp8_dbias_cast_transpose(dy, s, a, si, q.t, qt.t, db.t, ws, ct.E5M2)
    torch.cuda.synchronize()
    for g in (q, qt, db):
        g.check()
    ref = oracle.cast_transpose(x_cpu, 2.0, ct.E5M2)
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    assert np.array_equal(qt.numpy().reshape(cols, rows), ref["qt"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    bits = db.t.view(torch.int16).cpu().numpy().view(np.uint16)
    assert dbias_bf16_tolerance_ok(bits, x_cpu)
    assert np.mean(bits == oracle.dbias_bf16(x_cpu)) >= 0.99


@pytest.mark.parametrize("db_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(512, 256), (4112, 8208), (300, 70)])
def test_db_of_inf_and_nan_columns(shape, db_dtype):
    """Columns holding +Inf, -Inf, NaN, and +Inf with -Inf: db is +Inf, -Inf,
    NaN and NaN (the IEEE sums the oracle gives); the other columns are
    unaffected."""
    rows, cols = shape
    x = workloads.gradient_matrix("cpu", rows, cols, std=1e-2, outlier_fraction=0.0).float()
    x[rows // 3, 3] = float("inf")
    x[rows - 1, 5] = float("-inf")
    x[0, 7] = float("nan")
    x[1, 9] = float("inf")
    x[rows - 2, 9] = float("-inf")
    x_cpu = x.to(torch.bfloat16)
    ref = oracle.dbias(x_cpu)
    assert np.isposinf(ref[3]) and np.isneginf(ref[5]) and np.isnan(ref[7]) and np.isnan(ref[9])
    q, qt = ct.empty_outputs(x_cpu.cuda())
    db = torch.empty(cols, dtype=db_dtype, device="cuda")
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    ct.fp8_dbias_cast_transpose(x_cpu.cuda(), scalar(1.0), scalar(0.0), scalar(0.0), q, qt, db, ws,
                                ct.E5M2)
    torch.cuda.synchronize()
    got = db.float().cpu().numpy()
    assert np.isposinf(got[3]) and np.isneginf(got[5]) and np.isnan(got[7]) and np.isnan(got[9])
    rest = np.ones(cols, bool)
    rest[[3, 5, 7, 9]] = False
    if db_dtype == torch.float32:
        assert np.all(np.abs(got[rest].astype(np.float64) - ref[rest]) <=
                      1e-5 * x_cpu.double().abs().sum(0).numpy()[rest] + 1e-6)
    else:
        bits = db.view(torch.int16).cpu().numpy().view(np.uint16)
        assert bits[7] == 0x7FFF and bits[9] == 0x7FFF      # canonical NaN (the oracle's reading)
        assert np.array_equal(bits[[3, 5]], oracle.dbias_bf16(x_cpu)[[3, 5]])


def test_gradient_8192x12288_bf16_db_two_steps():
    """The gradient workload with a bf16 db, in the same two steps as the fp32
    case: scale 1, then the scale the update derives from the first amax."""
    dy = workloads.gradient_matrix("cuda")
    x_cpu = dy.cpu()
    rows, cols = dy.shape
    q, qt = ct.empty_outputs(dy)
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    hist = np.zeros((16, 1), np.float32)
    s_val = 1.0
    for step in range(2):
        db = torch.empty(cols, dtype=torch.bfloat16, device="cuda")
        a, si = scalar(0.0), scalar(0.0)
        ct.fp8_dbias_cast_transpose(dy, scalar(s_val), a, si, q, qt, db, ws, ct.E5M2)
        torch.cuda.synchronize()
        ref = oracle.cast_transpose(x_cpu, s_val, ct.E5M2)
        assert np.array_equal(q.cpu().numpy(), ref["q"]), step
        assert np.array_equal(qt.cpu().numpy(), ref["qt"]), step
        assert f32_bits(a.item()) == f32_bits(ref["amax"]), step
        bits = db.view(torch.int16).cpu().numpy().view(np.uint16)
        assert dbias_bf16_tolerance_ok(bits, x_cpu), step
        assert np.mean(bits == oracle.dbias_bf16(x_cpu)) >= 0.99, step
        hist[0, 0] = ref["amax"]
        hist, s_arr, _ = oracle.amax_and_scale_update(hist, np.float32([s_val]), np.ones(1, np.float32),
                                                      ct.E5M2, 0)
        s_val = float(s_arr[0])


@pytest.mark.parametrize("shape", [(4096, 8192), (4095, 4096)])
def test_graph_replays_with_new_data_and_a_shared_workspace(shape):
    """The per-tile column sums live in the workspace between the two kernels
    of a call; a replay of a captured call must add only its own sums, never
    a previous replay's.  Three replays with different data in the same
    (captured) buffers, each compared with the oracle; then another shape
    through the same workspace."""
    rows, cols = shape
    dy = torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda")
    q, qt = ct.empty_outputs(dy)
    db = torch.empty(cols, device="cuda")
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    s, a, si = scalar(1.0), scalar(0.0), scalar(0.0)
    dy.copy_(workloads.normal_bf16(rows, cols, 1.0, 900, "cuda"))
    ct.fp8_dbias_cast_transpose(dy, s, a, si, q, qt, db, ws, ct.E5M2)   # eager warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side), torch.cuda.graph(g):
        ct.fp8_dbias_cast_transpose(dy, s, a, si, q, qt, db, ws, ct.E5M2)
    torch.cuda.current_stream().wait_stream(side)
    for rep in range(3):
        x_cpu = workloads.normal_bf16(rows, cols, 0.5 + rep, 901 + rep)
        dy.copy_(x_cpu)
        a.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert dbias_tolerance_ok(db.cpu().numpy(), oracle.dbias(x_cpu), x_cpu), rep
        ref = oracle.cast_transpose(x_cpu, 1.0, ct.E5M2)
        assert np.array_equal(q.cpu().numpy(), ref["q"]), rep
        assert f32_bits(a.item()) == f32_bits(ref["amax"]), rep
    # another shape (direct path too: rows % 16 != 0) through the same workspace
    x2 = workloads.normal_bf16(1001, 2048, 3.0, 950)
    dy2 = x2.cuda()
    q2, qt2 = ct.empty_outputs(dy2)
    db2 = torch.empty(2048, device="cuda")
    a2, si2 = scalar(0.0), scalar(0.0)
    ct.fp8_dbias_cast_transpose(dy2, scalar(2.0), a2, si2, q2, qt2, db2, ws, ct.E4M3)
    torch.cuda.synchronize()
    check({"q": q2.cpu().numpy(), "qt": qt2.cpu().numpy(), "db": db2.cpu().numpy(),
           "amax": a2.item(), "scale_inv": si2.item()}, x2, 2.0, ct.E4M3)
