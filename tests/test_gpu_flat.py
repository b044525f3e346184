"""GPU parity of the flat cast kernel against the oracle, bit-exact.

A cast without transpose whose shape the tile kernels do not take (cols not a
multiple of 8, or q only 8-byte aligned), with x 16-byte and q 8-byte
aligned, runs as one flat array of rows * cols elements: 8-element chunks,
then the last n % 8 elements by one thread.  The cases cover every tail
length, the two ends of tiny arrays, q at an 8-byte but not 16-byte offset,
NaN and Inf in the tail (amax propagation), the noop flag, and the 8191 x
12287 matrix in full through the oracle on all host cores.  An x that is not
16-byte aligned takes the shifted flat cast: every even byte offset with
every tail length, lengths around its 31-chunk warp groups, special values
in the chunk assembled past the end of x, and the noop flag.
"""
import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
import oracle
from cast_transpose_gb300 import workloads
from gpu_util import CANARY, Guarded, f32_bits, scalar
from oracle_pool import OraclePool

pytestmark = pytest.mark.gpu

# rows * cols % 8 = 0 .. 7, and two arrays shorter than one chunk
TAILS = [(8, 5), (3, 3), (2, 5), (3, 9), (4, 5), (3, 7), (6, 5), (9, 7), (1, 1), (1, 7)]


@pytest.fixture(autouse=True)
def _no_device_error():
    ct.device_error(clear=True)
    yield
    assert ct.device_error() == 0


def _cast(x, scale, fmt, q_offset=0, amax_in=0.0, noop=None):
    rows, cols = x.shape
    q = Guarded(rows * cols, offset=q_offset)
    s, a, si = scalar(scale), scalar(amax_in), scalar(-1.0)
    ct.fp8_cast(x, s, a, si, q.t, fmt, noop_flag=noop)
    torch.cuda.synchronize()
    q.check()
    return q.numpy().reshape(rows, cols), a.item(), si.item()


def _assert_oracle(x_cpu, scale, fmt, got, amax_in=0.0):
    q, amax, sinv = got
    ref = oracle.cast_transpose(x_cpu, float(np.float32(scale)), fmt, want_qt=False, amax_in=amax_in)
    bad = np.argwhere(q != ref["q"])
    assert bad.size == 0, f"{len(bad)} FP8 bytes differ, first at {bad[:4].tolist()}"
    assert f32_bits(amax) == f32_bits(ref["amax"]), (amax, ref["amax"])
    assert f32_bits(sinv) == f32_bits(ref["scale_inv"])


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
@pytest.mark.parametrize("shape", TAILS)
def test_every_tail_length(fmt, shape):
    x_cpu = workloads.normal_bf16(*shape, 300.0, 50 + shape[0] * 16 + shape[1])
    _assert_oracle(x_cpu, 2.5, fmt, _cast(x_cpu.cuda(), 2.5, fmt))


@pytest.mark.parametrize("shape", [(64, 1000), (1000, 1037)])
def test_q_at_an_8_byte_offset(shape):
    """q 8-byte but not 16-byte aligned: the tile kernels decline it."""
    x_cpu = workloads.normal_bf16(*shape, 40.0, 61)
    _assert_oracle(x_cpu, 0.5, ct.E4M3, _cast(x_cpu.cuda(), 0.5, ct.E4M3, q_offset=8))


@pytest.mark.parametrize("where", ["tail", "chunk"])
def test_nan_and_inf(where):
    x_cpu = workloads.normal_bf16(7, 9, 3.0, 71)   # 63 elements: 7 chunks + a tail of 7
    flat = x_cpu.view(-1)
    if where == "tail":
        flat[60] = float("inf")
        flat[62] = float("nan")
    else:
        flat[3] = float("-inf")
        flat[20] = float("nan")
    _assert_oracle(x_cpu, 1.0, ct.E5M2, _cast(x_cpu.cuda(), 1.0, ct.E5M2))


def test_amax_is_max_merged():
    x_cpu = workloads.normal_bf16(9, 7, 1.0, 72)
    _assert_oracle(x_cpu, 1.0, ct.E4M3, _cast(x_cpu.cuda(), 1.0, ct.E4M3, amax_in=1e6), amax_in=1e6)


def test_noop_flag_writes_nothing():
    x = workloads.normal_bf16(333, 555, 9.0, 73, "cuda")
    q, amax, sinv = _cast(x, 1.25, ct.E4M3, amax_in=0.5, noop=scalar(1.0))
    assert np.all(q == CANARY)   # the fill Guarded starts with
    assert amax == 0.5 and sinv == -1.0


def test_ragged_8191x12287_in_full():
    """The ragged matrix of the benchmark, every byte of q against the oracle."""
    rows, cols = 8191, 12287
    x = workloads.normal_bf16(rows, cols, 1.0, 17, "cuda")
    q, amax, sinv = _cast(x, 1.0, ct.E4M3)
    with OraclePool() as pool:
        xin = pool.input_bf16(rows, cols)
        xin[:] = x.cpu().view(torch.int16).numpy().view(np.uint16)
        qv = pool.output_q(rows, cols)
        qv[:] = q
        res = pool.check_cast_transpose(rows, cols, 1.0, ct.E4M3, check_qt=False)
        del xin, qv
    assert res["bad_q"] == 0, ("FP8 data differs from the oracle", res["first_q"])
    assert f32_bits(amax) == f32_bits(res["amax"])
    assert f32_bits(sinv) == f32_bits(np.float32(1.0))


def _shifted(x_cpu, elems):
    """x on the GPU `elems` bf16 elements past a 256-byte-aligned allocation."""
    n = x_cpu.numel()
    big = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
    big[elems:elems + n] = x_cpu.reshape(-1).cuda()
    return big[elems:elems + n].view(x_cpu.shape)


@pytest.mark.parametrize("x_shift", range(1, 8))
@pytest.mark.parametrize("shape", TAILS + [(31, 8), (33, 8), (1, 248), (7, 1001), (300, 263)])
def test_shifted_x_every_offset_and_tail(shape, x_shift):
    """x 2, 4, .., 14 bytes past a 16-byte boundary (the shifted flat cast):
    every tail length, arrays shorter than one chunk, lengths around a
    31-chunk warp group, with q 8-byte aligned."""
    x_cpu = workloads.normal_bf16(*shape, 40.0, 900 + 16 * x_shift + shape[0] * 7 + shape[1])
    got = _cast(_shifted(x_cpu, x_shift), 0.375, ct.E4M3, q_offset=8 * (x_shift & 1))
    _assert_oracle(x_cpu, 0.375, ct.E4M3, got)


@pytest.mark.parametrize("x_shift", [1, 6])
def test_shifted_x_nan_and_inf_near_the_end(x_shift):
    """Special values in the last whole chunk and in the tail, reached
    through the assembled chunk past the end of x."""
    rows, cols = 37, 41
    x_cpu = workloads.normal_bf16(rows, cols, 1.0, 77 + x_shift)
    flat = x_cpu.reshape(-1)
    n = flat.numel()
    flat[n - 3] = float("inf")
    flat[(n // 8) * 8 - 2] = float("-inf")
    got = _cast(_shifted(x_cpu, x_shift), 1.0, ct.E5M2)
    _assert_oracle(x_cpu, 1.0, ct.E5M2, got)
    flat[n - 1] = float("nan")
    got = _cast(_shifted(x_cpu, x_shift), 1.0, ct.E5M2)
    _assert_oracle(x_cpu, 1.0, ct.E5M2, got)


def test_shifted_x_noop_flag_set_writes_nothing():
    x_cpu = workloads.normal_bf16(300, 263, 1.0, 5)
    q = Guarded(300 * 263)
    q.t.fill_(0x5A)
    s, a, si = scalar(1.0), scalar(0.0), scalar(-1.0)
    ct.fp8_cast(_shifted(x_cpu, 3), s, a, si, q.t, ct.E4M3, noop_flag=torch.ones(1, device="cuda"))
    torch.cuda.synchronize()
    q.check()
    assert (q.numpy() == 0x5A).all() and a.item() == 0.0 and si.item() == -1.0
