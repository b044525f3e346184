"""Pins of the oracle's fp32 -> bf16 rounding (the bf16 db output) against
values worked out by hand from the IEEE rule (round to nearest, ties to the
even significand, overflow past the largest finite bf16 to Inf) and against
torch's own CPU conversion, a library routine, on 4 M random fp32 patterns
and on every rounding boundary class."""
import numpy as np
import torch

import oracle
from cast_transpose_gb300 import workloads


def _bits(u32):
    return np.array(u32, dtype=np.uint32).view(np.float32)


# (fp32 bits, bf16 bits), each worked out by hand
HAND = [
    (0x3F800000, 0x3F80),   # 1.0
    (0x3F808000, 0x3F80),   # 1 + 2^-8: halfway between 1 (even) and 1 + 2^-7 (odd) -> even
    (0x3F818000, 0x3F82),   # 1 + 3*2^-8: halfway between 0x3F81 (odd) and 0x3F82 (even) -> even
    (0x3F808001, 0x3F81),   # just above the halfway point -> up
    (0x3F807FFF, 0x3F80),   # just below -> down
    (0xBF818000, 0xBF82),   # the same tie, negative
    (0x7F7F7FFF, 0x7F7F),   # below the overflow threshold -> the largest finite bf16
    (0x7F7F8000, 0x7F80),   # halfway between 0x7F7F (odd) and 2^128 (even) -> +Inf
    (0xFF7F8000, 0xFF80),   # the same, negative -> -Inf
    (0x80000000, 0x8000),   # -0 keeps its sign
    (0x00000001, 0x0000),   # smallest subnormal -> +0
    (0x80008000, 0x8000),   # subnormal halfway between 0 (even) and 0x0001 -> -0
    (0x00018000, 0x0002),   # subnormal halfway between 0x0001 (odd) and 0x0002 -> 0x0002
    (0x7F800000, 0x7F80),   # +Inf
    (0xFF800000, 0xFF80),   # -Inf
    (0x7FC00000, 0x7FFF),   # NaN -> canonical NaN
    (0xFFC00001, 0x7FFF),
]


def test_hand_worked():
    f = _bits([a for a, _ in HAND])
    got = oracle.f32_to_bf16(f)
    assert [int(g) for g in got] == [b for _, b in HAND]


def _torch_bf16_bits(f):
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_matches_torch_on_random_and_boundary_patterns():
    rng = np.random.default_rng(11)
    rand = rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    # every bf16 value with each low half that decides the rounding
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    edges = (hi[:, None] | lows[None, :]).reshape(-1)
    u = np.concatenate([rand, edges])
    f = u.view(np.float32)
    got = oracle.f32_to_bf16(f)
    ref = _torch_bf16_bits(f)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(got[nan] == 0x7FFF)


def test_dbias_bf16_is_the_rounded_column_sum():
    """db in bf16 equals torch's column sum in double, rounded to fp32 and then
    to bf16 by torch, on a gradient-like matrix with outliers."""
    dy = workloads.gradient_matrix("cpu", 300, 517, std=1e-2, outlier_fraction=1e-2)
    got = oracle.dbias_bf16(dy)
    ref = torch.sum(dy.double(), 0).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
