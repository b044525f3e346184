"""GPU parity of fp8_amax_and_scale_update and fp8_transpose against the
CPU oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
import oracle
from gpu_util import Guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_error():
    ct.device_error(clear=True)
    yield
    assert ct.device_error() == 0


def _history(L, n, seed):
    rng = np.random.default_rng(seed)
    h = (rng.standard_normal((L, n)) ** 2 * 10.0 ** rng.integers(-6, 4, size=(L, n))).astype(np.float32)
    # special columns: all zero, tiny (448/a overflows), Inf, NaN, fp32 subnormal,
    # a value whose scale is exactly representable
    h[:, 0] = 0.0
    h[:, 1] = 0.0
    h[0, 1] = 1e-38
    h[3 % L, 2] = np.inf
    h[L - 1, 3] = np.nan
    h[:, 4] = 0.0
    h[0, 4] = 1e-42
    h[:, 5] = 0.0
    h[L // 2, 5] = 3.5
    return h


@pytest.mark.parametrize("algo", [ct.AMAX_MAX, ct.AMAX_MOST_RECENT])
@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
@pytest.mark.parametrize("L,n,margin", [(16, 1, 0), (16, 48, 0), (1, 7, 0), (1024, 300, 3),
                                        (4, 1000, 126), (2, 8, 1), (1100, 5, 0)])
def test_update_matches_oracle(fmt, L, n, margin, algo):
    h = _history(L, max(n, 6), seed=L * 1000 + n)[:, :n].copy()
    rng = np.random.default_rng(n)
    s = (rng.random(n) * 100 + 0.01).astype(np.float32)
    si = np.zeros(n, np.float32)
    hd, sd, sid = torch.from_numpy(h).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(si).cuda()
    for step in range(3):
        ct.fp8_amax_and_scale_update_ex(hd, sd, sid, fmt, margin, amax_algo=algo)
        h, s, si = oracle.amax_and_scale_update(h, s, si, fmt, margin, algo=algo)
        torch.cuda.synchronize()
        assert np.array_equal(hd.cpu().numpy().view(np.uint32), h.view(np.uint32)), step
        assert np.array_equal(sd.cpu().numpy().view(np.uint32), s.view(np.uint32)), step
        assert np.array_equal(sid.cpu().numpy().view(np.uint32), si.view(np.uint32)), step
        # next step's amaxes
        hd[0] = torch.from_numpy(np.abs(rng.standard_normal(n)).astype(np.float32)).cuda()
        h[0] = hd[0].cpu().numpy()


TSHAPES = [(1, 1), (3, 5), (16, 16), (128, 128), (144, 272), (4096, 48), (48, 4096),
           (127, 129), (1000, 3), (2048, 2064), (8192, 12288)]


@pytest.mark.parametrize("shape", TSHAPES)
def test_transpose_matches_oracle(shape):
    rows, cols = shape
    g = torch.Generator().manual_seed(rows * 31 + cols)
    q_cpu = torch.randint(0, 256, (rows, cols), dtype=torch.uint8, generator=g)
    out = Guarded(rows * cols)
    ct.fp8_transpose(q_cpu.cuda(), out.t)
    torch.cuda.synchronize()
    out.check()
    assert np.array_equal(out.numpy().reshape(cols, rows), oracle.fp8_transpose(q_cpu.numpy()))


@pytest.mark.parametrize("shape", [(8192, 8192), (4112, 8208), (16, 4096), (8191, 8193), (4111, 3001),
                                   (17, 4095)])
def test_transpose_with_noop_flag_zero(shape):
    """With a noop flag (here 0) the transpose runs a looping first wave and
    one tile per CTA for the rest: 4096 tiles (several per looping CTA), a
    partial last tile row and column (2145 tiles), and fewer tiles than one
    wave; the aligned kernel for the first three shapes, the odd-shape kernel
    for the others."""
    rows, cols = shape
    g = torch.Generator().manual_seed(rows * 7 + cols)
    q_cpu = torch.randint(0, 256, (rows, cols), dtype=torch.uint8, generator=g)
    out = Guarded(rows * cols)
    ct.fp8_transpose(q_cpu.cuda(), out.t, noop_flag=torch.zeros(1, device="cuda"))
    torch.cuda.synchronize()
    out.check()
    assert np.array_equal(out.numpy().reshape(cols, rows), oracle.fp8_transpose(q_cpu.numpy()))


@pytest.mark.parametrize("shape", [(8192, 8192), (8191, 8193)])
def test_transpose_with_noop_flag_set_writes_nothing(shape):
    rows, cols = shape
    q = torch.randint(0, 256, (rows, cols), dtype=torch.uint8, device="cuda")
    out = Guarded(rows * cols)
    out.t.fill_(0x5A)
    ct.fp8_transpose(q, out.t, noop_flag=torch.ones(1, device="cuda"))
    torch.cuda.synchronize()
    out.check()
    assert (out.numpy() == 0x5A).all()


def test_transpose_misaligned():
    q_cpu = torch.randint(0, 256, (256, 256), dtype=torch.uint8)
    big = torch.empty(256 * 256 + 3, dtype=torch.uint8, device="cuda")
    big[3:] = q_cpu.cuda().reshape(-1)
    out = Guarded(256 * 256, offset=5)
    ct.fp8_transpose(big[3:].view(256, 256), out.t)
    torch.cuda.synchronize()
    out.check()
    assert np.array_equal(out.numpy().reshape(256, 256), oracle.fp8_transpose(q_cpu.numpy()))
