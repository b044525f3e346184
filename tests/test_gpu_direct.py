"""GPU parity of the large-launch kernel (one 128x128 tile per CTA, direct
16-byte loads) that the library picks for launches of 2048 tiles or more:
ragged shapes (row and column tile counts not multiples of 128), every entry
point that reaches it (cast + transpose, cast only, dbias, tensor lists with
one or per-tensor formats), the noop flag and graph replay.  Bit-exact
against the oracle; db within the dbias tolerance.
"""
import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
import oracle
from cast_transpose_gb300 import workloads
from gpu_util import Guarded, assert_same_cast, cast_transpose_gpu, dbias_tolerance_ok, f32_bits, scalar

pytestmark = pytest.mark.gpu

# >= 2048 tiles of 128x128, neither dimension a multiple of 128
RAGGED = [(4112, 8208), (2064, 16400), (16400, 2064)]


def _tiles(rows, cols):
    return -(-rows // 128) * -(-cols // 128)


@pytest.fixture(autouse=True)
def _no_device_error():
    ct.device_error(clear=True)
    yield
    assert ct.device_error() == 0


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
@pytest.mark.parametrize("shape", RAGGED)
def test_ragged_cast_transpose(fmt, shape):
    rows, cols = shape
    assert _tiles(rows, cols) >= 2048
    x_cpu = workloads.normal_bf16(rows, cols, 50.0, 900 + rows + cols)
    got = cast_transpose_gpu(x_cpu.cuda(), 2.5, fmt, amax_in=0.125)
    assert_same_cast(got, oracle.cast_transpose(x_cpu, 2.5, fmt, amax_in=0.125))


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
@pytest.mark.parametrize("shape", RAGGED + [(8192, 8200)])
def test_noop_flag_zero(fmt, shape):
    """A call given a noop flag (here 0) takes the looping grid of a few
    waves: ragged tile counts (an odd count leaves a CTA half idle) and, at
    8192 x 8200, about 7 tiles per group of 256 threads."""
    rows, cols = shape
    x_cpu = workloads.normal_bf16(rows, cols, 50.0, 700 + rows + cols)
    got = cast_transpose_gpu(x_cpu.cuda(), 0.375, fmt, amax_in=0.25, noop=scalar(0.0))
    assert_same_cast(got, oracle.cast_transpose(x_cpu, 0.375, fmt, amax_in=0.25))


def test_all_bf16_patterns_tiled():
    """Every bf16 pattern, repeated to a 4096 x 8192 matrix (2048 tiles)."""
    base = workloads.bf16_all_patterns().reshape(-1)
    g = torch.Generator().manual_seed(5)
    x_cpu = base[torch.randperm(65536, generator=g).repeat(512)].reshape(4096, 8192).contiguous()
    got = cast_transpose_gpu(x_cpu.cuda(), 3.7, ct.E5M2)
    assert_same_cast(got, oracle.cast_transpose(x_cpu, float(np.float32(3.7)), ct.E5M2))


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
@pytest.mark.parametrize("shape", RAGGED)
def test_cast_only_noop_flag_zero(fmt, shape):
    """A plain cast given a noop flag (here 0) takes the looping grid too."""
    rows, cols = shape
    x_cpu = workloads.normal_bf16(rows, cols, 30.0, 43 + rows)
    q = Guarded(rows * cols)
    s, a, si = scalar(0.75), scalar(0.0), scalar(0.0)
    ct.fp8_cast(x_cpu.cuda(), s, a, si, q.t, fmt, noop_flag=scalar(0.0))
    torch.cuda.synchronize()
    q.check()
    ref = oracle.cast_transpose(x_cpu, 0.75, fmt, want_qt=False)
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    assert f32_bits(si.item()) == f32_bits(ref["scale_inv"])


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
def test_ragged_cast_only(fmt):
    rows, cols = RAGGED[0]
    x_cpu = workloads.normal_bf16(rows, cols, 30.0, 41)
    q = Guarded(rows * cols)
    s, a, si = scalar(0.75), scalar(0.0), scalar(0.0)
    ct.fp8_cast(x_cpu.cuda(), s, a, si, q.t, fmt)
    torch.cuda.synchronize()
    q.check()
    ref = oracle.cast_transpose(x_cpu, 0.75, fmt, want_qt=False)
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    assert f32_bits(si.item()) == f32_bits(ref["scale_inv"])


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
@pytest.mark.parametrize("shape", RAGGED[:2])
def test_ragged_dbias(fmt, shape):
    rows, cols = shape
    x_cpu = workloads.gradient_matrix("cpu", rows, cols, std=1e-3, outlier_fraction=1e-3)
    n = rows * cols
    q, qt = Guarded(n), Guarded(n)
    db = Guarded(cols, dtype=torch.float32)
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    ws.fill_(0x7F)
    s, a, si = scalar(4.0), scalar(0.0), scalar(0.0)
    ct.fp8_dbias_cast_transpose(x_cpu.cuda(), s, a, si, q.t, qt.t, db.t, ws, fmt)
    torch.cuda.synchronize()
    for g in (q, qt, db):
        g.check()
    ref = oracle.cast_transpose(x_cpu, 4.0, fmt)
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    assert np.array_equal(qt.numpy().reshape(cols, rows), ref["qt"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    assert f32_bits(si.item()) == f32_bits(ref["scale_inv"])
    assert dbias_tolerance_ok(db.numpy(), oracle.dbias(x_cpu), x_cpu)


def test_dbias_deterministic():
    x = workloads.gradient_matrix("cuda", 4112, 8208)
    cols = x.shape[1]
    ws = torch.empty(ct.dbias_workspace_size(*x.shape), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        q, qt = ct.empty_outputs(x)
        db = torch.empty(cols, device="cuda")
        ct.fp8_dbias_cast_transpose(x, scalar(1.0), scalar(0.0), scalar(0.0), q, qt, db, ws, ct.E5M2)
        outs.append(db.cpu().numpy().view(np.uint32))
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("noop", [None, 0.0])
@pytest.mark.parametrize("per_tensor_fmt", [False, True])
def test_list_launch(per_tensor_fmt, noop):
    """One list launch of >= 2048 tiles: ragged entries, a one-tile-row entry,
    and one entry that takes the general kernel (33 x 65).  With a noop flag
    (here 0) the list takes the looping grid: tiles of different tensors in
    one group's run."""
    shapes = [(4112, 1040), (2048, 2064), (16, 4096), (1024, 4096), (1040, 4096), (33, 65),
              (4096, 4096), (144, 272)]
    fmts = [ct.E4M3, ct.E5M2, ct.E5M2, ct.E4M3, ct.E5M2, ct.E4M3, ct.E4M3, ct.E5M2]
    if not per_tensor_fmt:
        fmts = [ct.E4M3] * len(shapes)
    assert sum(_tiles(r, c) for r, c in shapes if r % 16 == 0 and c % 16 == 0) >= 2048
    xs_cpu = [workloads.normal_bf16(r, c, 200.0, 1200 + i) for i, (r, c) in enumerate(shapes)]
    n = len(xs_cpu)
    scales = torch.tensor([1.0, 4.0, 0.5, 2.0, 8.0, 1.0, 0.25, 3.0], device="cuda")
    amax = torch.full((n,), 0.5, device="cuda")
    sinv = torch.zeros(n, device="cuda")
    outs = [Guarded(x.numel()) for x in xs_cpu]
    outs_t = [Guarded(x.numel()) for x in xs_cpu]
    args = ([x.cuda() for x in xs_cpu], [scales[i:i + 1] for i in range(n)],
            [amax[i:i + 1] for i in range(n)], [sinv[i:i + 1] for i in range(n)],
            [o.t for o in outs], [o.t for o in outs_t])
    flag = None if noop is None else scalar(noop)
    if per_tensor_fmt:
        ct.fp8_multi_cast_transpose_ex(*args, fmts, noop_flag=flag)
    else:
        ct.fp8_multi_cast_transpose(*args, ct.E4M3, noop_flag=flag)
    torch.cuda.synchronize()
    a, si = amax.cpu().numpy(), sinv.cpu().numpy()
    for i, x in enumerate(xs_cpu):
        r, c = x.shape
        outs[i].check()
        outs_t[i].check()
        ref = oracle.cast_transpose(x, float(scales[i].item()), fmts[i], amax_in=0.5)
        assert np.array_equal(outs[i].numpy().reshape(r, c), ref["q"]), i
        assert np.array_equal(outs_t[i].numpy().reshape(c, r), ref["qt"]), i
        assert f32_bits(a[i]) == f32_bits(ref["amax"]), i
        assert f32_bits(si[i]) == f32_bits(ref["scale_inv"]), i


def test_noop_and_graph_replay():
    """Captured once; replay with flag 1 leaves every output as it was,
    replay with flag 0 after a new input matches the oracle."""
    rows, cols = RAGGED[0]
    x_cpu = workloads.normal_bf16(rows, cols, 10.0, 3)
    x = x_cpu.cuda()
    q, qt = ct.empty_outputs(x)
    db = torch.zeros(cols, device="cuda")
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    s, a, si = scalar(1.0), scalar(0.0), scalar(0.0)
    flag = scalar(0.0)

    def run():
        ct.fp8_dbias_cast_transpose(x, s, a, si, q, qt, db, ws, ct.E4M3, noop_flag=flag)

    run()   # first call outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    flag.fill_(1.0)
    snap = [t.clone() for t in (q, qt, db, a, si)]
    x.copy_(workloads.normal_bf16(rows, cols, 10.0, 4).cuda())
    g.replay()
    torch.cuda.synchronize()
    for before, now in zip(snap, (q, qt, db, a, si)):
        assert torch.equal(before.view(torch.uint8), now.view(torch.uint8))
    x2 = workloads.normal_bf16(rows, cols, 10.0, 5)
    x.copy_(x2.cuda())
    flag.fill_(0.0)
    a.fill_(0.0)
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.cast_transpose(x2, 1.0, ct.E4M3)
    assert np.array_equal(q.cpu().numpy(), ref["q"])
    assert np.array_equal(qt.cpu().numpy(), ref["qt"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    assert dbias_tolerance_ok(db.cpu().numpy(), oracle.dbias(x2), x2)


@pytest.mark.parametrize("tile_rows", [2047, 2048])
def test_dispatch_boundary(tile_rows):
    """2047 tiles (persistent TMA kernel) and 2048 tiles (direct kernel) of a
    one-tile-wide matrix, dbias included: the same bits either side."""
    rows, cols = 128 * tile_rows, 128
    x_cpu = workloads.gradient_matrix("cpu", rows, cols, std=1e-2, outlier_fraction=1e-4)
    n = rows * cols
    q, qt = Guarded(n), Guarded(n)
    db = Guarded(cols, dtype=torch.float32)
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    s, a, si = scalar(2.0), scalar(0.0), scalar(0.0)
    ct.fp8_dbias_cast_transpose(x_cpu.cuda(), s, a, si, q.t, qt.t, db.t, ws, ct.E4M3)
    torch.cuda.synchronize()
    for g in (q, qt, db):
        g.check()
    ref = oracle.cast_transpose(x_cpu, 2.0, ct.E4M3)
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    assert np.array_equal(qt.numpy().reshape(cols, rows), ref["qt"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])
    assert dbias_tolerance_ok(db.numpy(), oracle.dbias(x_cpu), x_cpu)


def test_long_list_direct_then_persistent():
    """70 tensors: the first launch of 64 (2048 tiles) takes the direct
    kernel, the remaining 6 the persistent one."""
    shapes = [(512, 1024)] * 64 + [(256, 384), (16, 4096), (128, 128), (640, 1040), (48, 48),
                                   (1024, 16)]
    xs_cpu = [workloads.normal_bf16(r, c, 3.0, 5000 + i) for i, (r, c) in enumerate(shapes)]
    assert sum(_tiles(r, c) for r, c in shapes[:64]) == 2048
    n = len(xs_cpu)
    scales = torch.tensor([float(1 + i % 5) for i in range(n)], device="cuda")
    amax = torch.zeros(n, device="cuda")
    sinv = torch.zeros(n, device="cuda")
    outs = [torch.empty(x.numel(), dtype=torch.uint8, device="cuda") for x in xs_cpu]
    outs_t = [torch.empty(x.numel(), dtype=torch.uint8, device="cuda") for x in xs_cpu]
    ct.fp8_multi_cast_transpose([x.cuda() for x in xs_cpu], [scales[i:i + 1] for i in range(n)],
                                [amax[i:i + 1] for i in range(n)], [sinv[i:i + 1] for i in range(n)],
                                outs, outs_t, ct.E5M2)
    torch.cuda.synchronize()
    a = amax.cpu().numpy()
    for i, x in enumerate(xs_cpu):
        r, c = x.shape
        ref = oracle.cast_transpose(x, float(1 + i % 5), ct.E5M2)
        assert np.array_equal(outs[i].cpu().numpy().reshape(r, c), ref["q"]), i
        assert np.array_equal(outs_t[i].cpu().numpy().reshape(c, r), ref["qt"]), i
        assert f32_bits(a[i]) == f32_bits(ref["amax"]), i


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
@pytest.mark.parametrize("shape", [(4096, 8200), (2064, 16392), (256, 136), (1024, 1032), (16, 8),
                                   (144, 24)])
def test_cols_multiple_of_8(fmt, shape):
    """cols % 16 == 8 takes the fast kernels (the direct kernel from 2048
    tiles, the persistent one below): cast-transpose, cast only and dbias."""
    rows, cols = shape
    x_cpu = workloads.gradient_matrix("cpu", rows, cols, std=1e-2, outlier_fraction=1e-3)
    got = cast_transpose_gpu(x_cpu.cuda(), 1.75, fmt, amax_in=0.0625)
    ref = oracle.cast_transpose(x_cpu, 1.75, fmt, amax_in=0.0625)
    assert_same_cast(got, ref)
    n = rows * cols
    q = Guarded(n)
    s, a, si = scalar(1.75), scalar(0.0), scalar(0.0)
    ct.fp8_cast(x_cpu.cuda(), s, a, si, q.t, fmt)
    torch.cuda.synchronize()
    q.check()
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    q2, qt2 = Guarded(n), Guarded(n)
    db = Guarded(cols, dtype=torch.float32)
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    ct.fp8_dbias_cast_transpose(x_cpu.cuda(), scalar(1.75), scalar(0.0), scalar(0.0), q2.t, qt2.t,
                                db.t, ws, fmt)
    torch.cuda.synchronize()
    for g in (q2, qt2, db):
        g.check()
    assert np.array_equal(q2.numpy().reshape(rows, cols), ref["q"])
    assert np.array_equal(qt2.numpy().reshape(cols, rows), ref["qt"])
    assert dbias_tolerance_ok(db.numpy(), oracle.dbias(x_cpu), x_cpu)


def test_list_with_cols_multiple_of_8():
    shapes = [(1024, 1032), (4096, 4104), (16, 8), (528, 200)]
    xs_cpu = [workloads.normal_bf16(r, c, 7.0, 8100 + i) for i, (r, c) in enumerate(shapes)]
    n = len(xs_cpu)
    scales = torch.tensor([1.0, 2.0, 0.5, 4.0], device="cuda")
    amax = torch.zeros(n, device="cuda")
    sinv = torch.zeros(n, device="cuda")
    outs = [Guarded(x.numel()) for x in xs_cpu]
    outs_t = [Guarded(x.numel()) for x in xs_cpu]
    ct.fp8_multi_cast_transpose([x.cuda() for x in xs_cpu], [scales[i:i + 1] for i in range(n)],
                                [amax[i:i + 1] for i in range(n)], [sinv[i:i + 1] for i in range(n)],
                                [o.t for o in outs], [o.t for o in outs_t], ct.E4M3)
    torch.cuda.synchronize()
    a = amax.cpu().numpy()
    for i, x in enumerate(xs_cpu):
        r, c = x.shape
        outs[i].check()
        outs_t[i].check()
        ref = oracle.cast_transpose(x, float(scales[i].item()), ct.E4M3)
        assert np.array_equal(outs[i].numpy().reshape(r, c), ref["q"]), i
        assert np.array_equal(outs_t[i].numpy().reshape(c, r), ref["qt"]), i
        assert f32_bits(a[i]) == f32_bits(ref["amax"]), i


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
@pytest.mark.parametrize("shape", [(4100, 8192), (1000, 1024), (17, 8), (130, 4096), (4097, 136),
                                   (2063, 8200), (1, 512)])
def test_rows_not_multiple_of_16(fmt, shape):
    """rows % 16 != 0, cols % 8 == 0, aligned buffers: the direct kernel with
    transposed blocks at any alignment (the last one short), at every size;
    cast-transpose, cast only and dbias."""
    rows, cols = shape
    x_cpu = workloads.gradient_matrix("cpu", rows, cols, std=1e-2, outlier_fraction=1e-3)
    got = cast_transpose_gpu(x_cpu.cuda(), 3.25, fmt)
    ref = oracle.cast_transpose(x_cpu, 3.25, fmt)
    assert_same_cast(got, ref)
    n = rows * cols
    q2, qt2 = Guarded(n), Guarded(n)
    db = Guarded(cols, dtype=torch.float32)
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    ws.fill_(0x7F)
    ct.fp8_dbias_cast_transpose(x_cpu.cuda(), scalar(3.25), scalar(0.0), scalar(0.0), q2.t, qt2.t,
                                db.t, ws, fmt)
    torch.cuda.synchronize()
    for g in (q2, qt2, db):
        g.check()
    assert np.array_equal(q2.numpy().reshape(rows, cols), ref["q"])
    assert np.array_equal(qt2.numpy().reshape(cols, rows), ref["qt"])
    assert dbias_tolerance_ok(db.numpy(), oracle.dbias(x_cpu), x_cpu)
    q = Guarded(n)
    s, a, si = scalar(3.25), scalar(0.0), scalar(0.0)
    ct.fp8_cast(x_cpu.cuda(), s, a, si, q.t, fmt)
    torch.cuda.synchronize()
    q.check()
    assert np.array_equal(q.numpy().reshape(rows, cols), ref["q"])
    assert f32_bits(a.item()) == f32_bits(ref["amax"])


@pytest.mark.parametrize("d", range(1, 16))
def test_odd_rows_every_residue(d):
    """rows % 16 = d, for every d: an interior tile row stores whole aligned
    16-byte blocks of qT, the first of which starts up to 15 rows above the
    tile (rows of the tile above, loaded with it); the first and last tile
    rows are cut at the column ends.  Five tile rows, three interior; 264
    columns leave a ragged column tile.  Cast-transpose eager, with a noop
    flag 0 (E4M3) and with x_ready (E5M2); dbias; a noop flag 1 writes
    nothing."""
    rows, cols = 512 + 128 + d, 264
    x_cpu = workloads.normal_bf16(rows, cols, 20.0, 300 + d)
    ref4 = oracle.cast_transpose(x_cpu, 1.5, ct.E4M3)
    assert_same_cast(cast_transpose_gpu(x_cpu.cuda(), 1.5, ct.E4M3), ref4)
    assert_same_cast(cast_transpose_gpu(x_cpu.cuda(), 1.5, ct.E4M3, noop=scalar(0.0)), ref4)
    x = x_cpu.cuda()
    n = rows * cols
    q, qt = Guarded(n), Guarded(n)
    s, a, si = scalar(1.5), scalar(0.0), scalar(0.0)
    ct.fp8_cast_transpose(x, s, a, si, q.t, qt.t, ct.E5M2, x_ready=True)
    torch.cuda.synchronize()
    q.check()
    qt.check()
    ref5 = oracle.cast_transpose(x_cpu, 1.5, ct.E5M2)
    assert np.array_equal(q.numpy().reshape(rows, cols), ref5["q"])
    assert np.array_equal(qt.numpy().reshape(cols, rows), ref5["qt"])
    q2, qt2 = Guarded(n), Guarded(n)
    db = Guarded(cols, dtype=torch.float32)
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    ct.fp8_dbias_cast_transpose(x, scalar(1.5), scalar(0.0), scalar(0.0), q2.t, qt2.t, db.t, ws,
                                ct.E4M3)
    torch.cuda.synchronize()
    for g in (q2, qt2, db):
        g.check()
    assert np.array_equal(q2.numpy().reshape(rows, cols), ref4["q"])
    assert np.array_equal(qt2.numpy().reshape(cols, rows), ref4["qt"])
    assert dbias_tolerance_ok(db.numpy(), oracle.dbias(x_cpu), x_cpu)
    q3, qt3 = Guarded(n), Guarded(n)
    q3.t.fill_(0x5A)
    qt3.t.fill_(0x5A)
    a3 = scalar(0.0)
    ct.fp8_cast_transpose(x, scalar(1.5), a3, scalar(0.0), q3.t, qt3.t, ct.E4M3,
                          noop_flag=scalar(1.0))
    torch.cuda.synchronize()
    q3.check()
    qt3.check()
    assert (q3.numpy() == 0x5A).all() and (qt3.numpy() == 0x5A).all() and a3.item() == 0.0


@pytest.mark.parametrize("rows", [8192, 4096])
def test_default_path_sees_x_written_by_the_preceding_kernel(rows):
    """The direct kernel's first wave asks for its tiles, and the second
    wave's, to be prefetched into L2 before the wait for the preceding kernel
    (cast only and dbias, no noop flag); the persistent TMA kernel asks for
    all of its tiles.  The kernel just before each call rewrites x (a sign
    flip), eagerly and in a replayed graph: every call must see the new
    values.  8192 x 4096 is 2048 tiles (the direct kernel), 4096 x 4096 is
    1024 (the TMA kernel)."""
    cols = 4096
    x_cpu = workloads.normal_bf16(rows, cols, 1.0, 77)
    refs = [oracle.cast_transpose(x_cpu, 1.0, ct.E4M3), oracle.cast_transpose(-x_cpu, 1.0, ct.E4M3)]
    dbs = [oracle.dbias(x_cpu), oracle.dbias(-x_cpu)]
    x = x_cpu.cuda()
    qc = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    q, qt = ct.empty_outputs(x)
    db = torch.empty(cols, device="cuda")
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    s, a, si = scalar(1.0), scalar(0.0), scalar(0.0)

    def step():
        x.neg_()                                    # x := -x_cpu, then the cast only
        ct.fp8_cast(x, s, a, si, qc, ct.E4M3)
        x.neg_()                                    # x := +x_cpu, then the dbias cast-transpose
        ct.fp8_dbias_cast_transpose(x, s, a, si, q, qt, db, ws, ct.E4M3)

    for i in range(6):
        step()
        torch.cuda.synchronize()
        assert np.array_equal(qc.cpu().numpy(), refs[1]["q"]), i
        assert np.array_equal(q.cpu().numpy(), refs[0]["q"]), i
        assert np.array_equal(qt.cpu().numpy(), refs[0]["qt"]), i
        assert dbias_tolerance_ok(db.cpu().numpy(), dbs[0], x_cpu), i
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side), torch.cuda.graph(g):
        x.neg_()
        ct.fp8_cast(x, s, a, si, qc, ct.E4M3)
    torch.cuda.current_stream().wait_stream(side)
    for i in range(4):                              # x flips on every replay
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(qc.cpu().numpy(), refs[(i + 1) % 2]["q"]), i


@pytest.mark.parametrize("shape", [(8192, 4096), (4095, 4096)])
def test_x_ready_on_the_direct_kernel(shape):
    """CT_X_READY on the direct kernel loads the tiles before the wait for the
    preceding kernel (here a fill of an unrelated buffer): cast-transpose and
    dbias (CT_DBIAS_X_READY) against the oracle, eager and replayed."""
    rows, cols = shape
    x_cpu = workloads.gradient_matrix("cpu", rows, cols, std=1e-2, outlier_fraction=1e-3)
    ref = oracle.cast_transpose(x_cpu, 2.0, ct.E5M2)
    db_ref = oracle.dbias(x_cpu)
    x = x_cpu.cuda()
    q, qt = ct.empty_outputs(x)
    q2, qt2 = ct.empty_outputs(x)
    db = torch.empty(cols, device="cuda")
    ws = torch.empty(ct.dbias_workspace_size(rows, cols), dtype=torch.uint8, device="cuda")
    other = torch.empty(1 << 20, device="cuda")
    s, a, si, a2, si2 = scalar(2.0), scalar(0.0), scalar(0.0), scalar(0.0), scalar(0.0)

    def step():
        other.fill_(1.0)                            # the preceding kernel does not write x
        ct.fp8_cast_transpose(x, s, a, si, q, qt, ct.E5M2, x_ready=True)
        ct.fp8_dbias_cast_transpose(x, s, a2, si2, q2, qt2, db, ws, ct.E5M2, x_ready=True)

    def check():
        torch.cuda.synchronize()
        for qq, tt, aa, ii in ((q, qt, a, si), (q2, qt2, a2, si2)):
            assert np.array_equal(qq.cpu().numpy(), ref["q"])
            assert np.array_equal(tt.cpu().numpy(), ref["qt"])
            assert f32_bits(aa.item()) == f32_bits(ref["amax"])
            assert f32_bits(ii.item()) == f32_bits(ref["scale_inv"])
        assert dbias_tolerance_ok(db.cpu().numpy(), db_ref, x_cpu)

    step()
    check()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side), torch.cuda.graph(g):
        step()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        for t in (q, qt, q2, qt2):
            t.zero_()
        db.zero_()
        a.zero_()
        a2.zero_()
        g.replay()
        check()
