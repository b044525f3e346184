"""Pins for the oracle's cast-transpose, amax, dbias and transpose.

Each check compares the oracle with something that is not the oracle:
hand-worked fixtures (tests/golden), torch's float8 rounding and reductions
(library routines), or invariants such as transpose(transpose(q)) == q.
"""
import numpy as np
import pytest
import torch

import oracle
from cast_transpose_gb300 import workloads
from golden_io import f32_to_bf16_bits, read_cast

TORCH_FP8 = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


@pytest.mark.parametrize("name", ["cast_e4m3_2x3.txt", "cast_e5m2_4x4.txt"])
def test_hand_worked_fixture(oracle_lib, name):
    g = read_cast(name)
    bits = f32_to_bf16_bits(g["x"])
    r = oracle.cast_transpose(bits, g["scale"], g["fmt"])
    assert np.array_equal(r["q"], g["q"]), (r["q"], g["q"])
    assert np.array_equal(r["qt"], g["q"].T)
    assert r["amax"] == g["amax"]
    assert r["scale_inv"] == g["scale_inv"]


def _library_cast(x_bf16: torch.Tensor, scale: float, fmt: int) -> np.ndarray:
    """torch's float8 conversion of the fp32 product; saturation and NaN are
    filled in from their closed forms, since torch does not saturate."""
    maxval = oracle.FP8_MAX[fmt]
    maxcode = 0x7E if fmt == oracle.E4M3 else 0x7B
    p = x_bf16.float() * torch.tensor(scale, dtype=torch.float32)
    codes = p.to(TORCH_FP8[fmt]).view(torch.uint8).numpy().copy()
    pn = p.numpy()
    sat = np.abs(pn) >= maxval
    codes[sat] = np.where(pn[sat] > 0, maxcode, 0x80 | maxcode)
    codes[np.isnan(pn)] = 0x7F
    return codes


SCALES = [1.0, 2.0 ** -8, 2.0 ** 20, 3.7, 448.0 / 5.0, 2.0 ** 126, 1e-38]


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("scale", SCALES)
def test_all_bf16_patterns_against_torch(oracle_lib, fmt, scale):
    x = workloads.bf16_all_patterns()
    scale = float(np.float32(scale))
    r = oracle.cast_transpose(x, scale, fmt)
    ref = _library_cast(x, scale, fmt)
    assert np.array_equal(r["q"], ref)
    assert np.array_equal(r["qt"], ref.T)


def test_amax_matches_torch_and_merges(oracle_lib):
    x = workloads.normal_bf16(37, 53, 3.0, 11)
    ref = x.float().abs().max().item()
    assert oracle.cast_transpose(x, 1.0, oracle.E4M3)["amax"] == np.float32(ref)
    assert oracle.cast_transpose(x, 1.0, oracle.E4M3, amax_in=1e6)["amax"] == np.float32(1e6)
    assert oracle.cast_transpose(x, 1.0, oracle.E4M3, amax_in=0.5)["amax"] == np.float32(ref)
    assert oracle.amax(x) == np.float32(ref)
    assert oracle.amax(x, 7.0) == np.float32(max(ref, 7.0))
    y = x.clone()
    y[3, 4] = float("nan")
    assert np.isnan(oracle.cast_transpose(y, 1.0, oracle.E4M3)["amax"])
    y = x.clone()
    y[5, 6] = float("-inf")
    assert oracle.cast_transpose(y, 1.0, oracle.E4M3)["amax"] == np.inf


def test_scale_inv_is_correctly_rounded_reciprocal(oracle_lib):
    from fractions import Fraction
    x = workloads.normal_bf16(2, 2, 1.0, 1)
    for s in [3.0, 7.0, 448.0 / 3.0, 1e-30, 2.0 ** 100]:
        s32 = np.float32(s)
        got = oracle.cast_transpose(x, s32, oracle.E4M3)["scale_inv"]
        exact = 1 / Fraction(float(s32))
        err = abs(Fraction(float(got)) - exact)
        for nb in (np.nextafter(got, np.float32(np.inf)), np.nextafter(got, np.float32(0))):
            assert err <= abs(Fraction(float(nb)) - exact)


def test_transpose_involution_and_shape(oracle_lib):
    x = workloads.normal_bf16(33, 65, 1.0, 3)
    r = oracle.cast_transpose(x, 1.0, oracle.E4M3)
    assert r["qt"].shape == (65, 33)
    assert np.array_equal(oracle.fp8_transpose(r["q"]), r["qt"])
    assert np.array_equal(oracle.fp8_transpose(oracle.fp8_transpose(r["q"])), r["q"])
    assert np.array_equal(r["qt"], r["q"].T)


def test_transpose_random_bytes(oracle_lib):
    rng = np.random.default_rng(5)
    q = rng.integers(0, 256, size=(17, 129), dtype=np.uint8)
    assert np.array_equal(oracle.fp8_transpose(q), q.T)


@pytest.mark.parametrize("shape", [(1, 1), (1, 17), (127, 129), (512, 96)])
def test_dbias_matches_torch_double_sum(oracle_lib, shape):
    x = workloads.gradient_matrix(rows=shape[0], cols=shape[1], outlier_fraction=0.01)
    db = oracle.dbias(x)
    ref = x.double().sum(dim=0).numpy()
    col_abs = x.double().abs().sum(dim=0).numpy()
    # accumulated in double, one rounding to fp32
    assert np.all(np.abs(db.astype(np.float64) - ref) <= np.abs(ref) * 2.0 ** -24 + 1e-45)
    assert np.all(np.abs(db - ref) <= 1e-5 * col_abs + 1e-6)


def test_dbias_closed_form(oracle_lib):
    # columns of constant c sum to rows * c exactly
    x = torch.full((300, 5), 0.25, dtype=torch.bfloat16)
    x[:, 1] = -3.0
    assert list(oracle.dbias(x)) == [75.0, -900.0, 75.0, 75.0, 75.0]


def test_empty_matrix(oracle_lib):
    x = torch.zeros(0, 7, dtype=torch.bfloat16)
    r = oracle.cast_transpose(x, 1.0, oracle.E4M3, amax_in=0.0)
    assert r["q"].shape == (0, 7) and r["qt"].shape == (7, 0) and r["amax"] == 0.0
