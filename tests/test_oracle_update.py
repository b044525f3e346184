"""Pins for the oracle's delayed-scaling update (amax history -> scale).

Checked against a hand-worked sequence (tests/golden/update_e4m3_L4.txt),
exact rational arithmetic (fractions), closed forms (power-of-two rescaling,
margins) and the guard cases (amax 0, too tiny, Inf, NaN).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from golden_io import read_update


def _is_correctly_rounded(got: np.float32, exact: Fraction) -> bool:
    err = abs(Fraction(float(got)) - exact)
    up = np.nextafter(got, np.float32(np.inf))
    dn = np.nextafter(got, np.float32(-np.inf))
    return err <= abs(Fraction(float(up)) - exact) and err <= abs(Fraction(float(dn)) - exact)


def test_hand_worked_sequence(oracle_lib):
    g = read_update("update_e4m3_L4.txt")
    n = len(g["init_scale"])
    hist = np.zeros((g["L"], n), dtype=np.float32)
    scale = g["init_scale"].copy()
    sinv = (np.float32(1.0) / scale).astype(np.float32)
    for amax, want in g["steps"]:
        hist[0] = amax
        hist, scale, sinv = oracle.amax_and_scale_update(hist, scale, sinv, g["fmt"], g["margin"])
        assert np.array_equal(scale, want), (scale, want)
        for s, si in zip(scale, sinv):
            assert _is_correctly_rounded(si, 1 / Fraction(float(s)))
        assert np.all(hist[0] == 0)


def test_weight_sequence_closed_form(oracle_lib):
    """x_k = x * 2^k (k = -4..3) has amax_k = 2^k a0, an increasing sequence,
    so the window maximum is always the latest and scale_k = 2^-k * scale_0,
    with scale_0 the correctly rounded 448 / a0."""
    a0 = np.float32(0.0953125)
    L = 16
    hist = np.zeros((L, 1), dtype=np.float32)
    scale = np.ones(1, dtype=np.float32)
    sinv = np.ones(1, dtype=np.float32)
    s0 = None
    for k in range(-4, 4):
        hist[0, 0] = np.float32(a0 * np.float32(2.0 ** k))
        hist, scale, sinv = oracle.amax_and_scale_update(hist, scale, sinv, oracle.E4M3, 0)
        if s0 is None:
            s0 = scale[0] * np.float32(2.0 ** -4)
            assert _is_correctly_rounded(s0, Fraction(448) / Fraction(float(a0)))
        assert scale[0] == np.float32(s0 * np.float32(2.0 ** -k))


@pytest.mark.parametrize("margin", [0, 1, 3, 10])
def test_margin_is_power_of_two(oracle_lib, margin):
    hist = np.array([[3.3], [0.7]], dtype=np.float32)
    s = np.ones(1, np.float32)
    _, base, _ = oracle.amax_and_scale_update(hist, s, s, oracle.E5M2, 0)
    _, got, _ = oracle.amax_and_scale_update(hist, s, s, oracle.E5M2, margin)
    assert got[0] == np.float32(base[0] / np.float32(2.0 ** margin))
    assert _is_correctly_rounded(base[0], Fraction(57344) / Fraction(float(np.float32(3.3))))


@pytest.mark.parametrize("amax", [0.0, 1e-38, np.inf, np.nan])
def test_guard_keeps_scale(oracle_lib, amax):
    hist = np.array([[amax], [0.0], [0.0]], dtype=np.float32)
    s = np.array([5.0], np.float32)
    h, scale, sinv = oracle.amax_and_scale_update(hist, s, np.zeros(1, np.float32), oracle.E4M3, 0)
    assert scale[0] == 5.0 and sinv[0] == np.float32(0.2)
    assert h[0, 0] == 0.0
    assert np.array_equal(h[1], hist[0], equal_nan=True)


def test_tiny_but_finite_scale_updates(oracle_lib):
    # bf16(1e-30) as amax: 448 / a is about 4.5e32, finite, so the scale moves
    import torch
    a = np.float32(torch.tensor(1e-30).to(torch.bfloat16).float().item())
    hist = np.array([[a]], dtype=np.float32)
    s = np.ones(1, np.float32)
    _, scale, sinv = oracle.amax_and_scale_update(hist, s, s, oracle.E4M3, 0)
    assert np.isfinite(scale[0]) and scale[0] > 1e32
    assert _is_correctly_rounded(scale[0], Fraction(448) / Fraction(float(a)))


def test_window_slides_out_a_spike(oracle_lib):
    L = 5
    hist = np.zeros((L, 1), np.float32)
    s = np.ones(1, np.float32)
    si = np.ones(1, np.float32)
    scales = []
    for step in range(8):
        hist[0, 0] = 100.0 if step == 0 else 1.0
        hist, s, si = oracle.amax_and_scale_update(hist, s, si, oracle.E4M3, 0)
        scales.append(float(s[0]))
    # the spike is in the window for exactly L updates
    assert scales[:L] == [float(np.float32(448.0 / 100.0))] * L
    assert scales[L:] == [448.0] * (8 - L)


def test_nan_in_history_propagates(oracle_lib):
    hist = np.array([[1.0, 2.0], [np.nan, 3.0], [8.0, np.nan]], dtype=np.float32)
    s = np.array([1.0, 1.0], np.float32)
    h, scale, _ = oracle.amax_and_scale_update(hist, s, s, oracle.E4M3, 0)
    assert list(scale) == [1.0, 1.0]
    assert np.array_equal(h[1:], hist[:-1], equal_nan=True)


def test_most_recent_ignores_older_rows(oracle_lib):
    # rows 1..: a spike of 100 that the window maximum would use
    hist = np.array([[2.0, 0.0, np.nan], [100.0, 100.0, 1.0], [7.0, 3.0, 1.0]], dtype=np.float32)
    s = np.array([1.0, 5.0, 6.0], np.float32)
    h, scale, sinv = oracle.amax_and_scale_update(hist, s, s, oracle.E4M3, 0,
                                                  algo=oracle.AMAX_MOST_RECENT)
    assert scale[0] == np.float32(224.0)            # 448 / 2, the spike ignored
    assert scale[1] == 5.0                           # row 0 is 0: the scale stays
    assert scale[2] == 6.0                           # row 0 is NaN: the scale stays
    assert _is_correctly_rounded(sinv[0], 1 / Fraction(224))
    assert np.array_equal(h[1:], hist[:-1], equal_nan=True) and np.all(h[0] == 0)
    _, smax, _ = oracle.amax_and_scale_update(hist, s, s, oracle.E4M3, 0)
    assert smax[0] == np.float32(4.48)               # the window maximum uses the spike


def test_most_recent_equals_max_for_history_of_one(oracle_lib):
    rng = np.random.default_rng(1)
    hist = np.abs(rng.standard_normal((1, 50))).astype(np.float32)
    s = np.ones(50, np.float32)
    a = oracle.amax_and_scale_update(hist, s, s, oracle.E5M2, 3)
    b = oracle.amax_and_scale_update(hist, s, s, oracle.E5M2, 3, algo=oracle.AMAX_MOST_RECENT)
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.uint32), v.view(np.uint32))
