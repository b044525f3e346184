"""Pins for the oracle's FP8 codec, against things other than the oracle.

* decode of every code against torch's float8 dtypes (a library routine);
* encode against an exhaustive nearest-value search over the 256 decoded
  codes (ties to the even code, saturation above the largest normal);
* encode against torch's own float8 rounding wherever torch does not need to
  saturate;
* closed-form special cases (NaN, +-Inf, signed zero, round trips).
"""
import numpy as np
import pytest
import torch

import fp8_search
import oracle

FMTS = [(oracle.E4M3, torch.float8_e4m3fn, 0x7E, 448.0),
        (oracle.E5M2, torch.float8_e5m2, 0x7B, 57344.0)]


def _torch_decode(dtype):
    return torch.arange(256, dtype=torch.uint8).view(dtype).float().numpy()


@pytest.mark.parametrize("fmt,dtype,maxcode,maxval", FMTS)
def test_decode_matches_torch_float8(oracle_lib, fmt, dtype, maxcode, maxval):
    mine = oracle.fp8_decode(np.arange(256, dtype=np.uint8), fmt)
    ref = _torch_decode(dtype)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan].view(np.uint32), ref[~nan].view(np.uint32))  # signed zeros too
    assert mine[maxcode] == maxval and mine[0x80 | maxcode] == -maxval


@pytest.mark.parametrize("fmt,dtype,maxcode,maxval", FMTS)
def test_round_trip_of_every_code(oracle_lib, fmt, dtype, maxcode, maxval):
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.fp8_decode(codes, fmt)
    back = oracle.fp8_encode(vals, fmt)
    finite = np.isfinite(vals)
    assert np.array_equal(back[finite], codes[finite])
    assert np.all(back[np.isnan(vals)] == 0x7F)            # canonical NaN
    inf = np.isinf(vals)                                     # E5M2 only
    assert np.all(back[inf] == np.where(vals[inf] > 0, maxcode, 0x80 | maxcode))


def _brute_force_encode(p: np.ndarray, fmt: int, maxcode: int, maxval: float):
    """Nearest FP8 value by exhaustive search over the decoded positive codes
    (tests/fp8_search.py): independent of the oracle's binade arithmetic."""
    assert maxcode == fp8_search.MAXCODE[fmt] and maxval == fp8_search.MAXVAL[fmt]
    return fp8_search.nearest_code_by_search(p, fmt)


def _probe_values(fmt):
    rng = np.random.default_rng(7 + fmt)
    vals = []
    # every bf16 pattern, as fp32
    vals.append((np.arange(65536, dtype=np.uint32) << 16).view(np.float32))
    # random fp32 bit patterns
    vals.append(rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32))
    # every grid point, midpoints, and one fp32 ulp either side of each
    grid = oracle.fp8_decode(np.arange(256, dtype=np.uint8), fmt)
    g = np.sort(np.unique(grid[np.isfinite(grid)].astype(np.float64)))
    mids = ((g[:-1] + g[1:]) / 2).astype(np.float32)
    pts = np.concatenate([g.astype(np.float32), mids])
    vals += [pts, np.nextafter(pts, np.float32(np.inf)), np.nextafter(pts, np.float32(-np.inf))]
    return np.concatenate(vals).astype(np.float32)


@pytest.mark.parametrize("fmt,dtype,maxcode,maxval", FMTS)
def test_encode_matches_brute_force_nearest(oracle_lib, fmt, dtype, maxcode, maxval):
    p = _probe_values(fmt)
    mine = oracle.fp8_encode(p, fmt)
    ref = _brute_force_encode(p, fmt, maxcode, maxval)
    bad = np.nonzero(mine != ref)[0]
    assert bad.size == 0, [(float(p[i]), hex(mine[i]), hex(ref[i])) for i in bad[:8]]


@pytest.mark.parametrize("fmt,dtype,maxcode,maxval", FMTS)
def test_encode_matches_torch_where_no_saturation(oracle_lib, fmt, dtype, maxcode, maxval):
    p = _probe_values(fmt)
    keep = np.isfinite(p) & (np.abs(p) < maxval)
    p = p[keep]
    mine = oracle.fp8_encode(p, fmt)
    ref = torch.from_numpy(p).to(dtype).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


@pytest.mark.parametrize("fmt,dtype,maxcode,maxval", FMTS)
def test_special_values(oracle_lib, fmt, dtype, maxcode, maxval):
    p = np.array([np.nan, -np.nan, np.inf, -np.inf, 0.0, -0.0, maxval * 4, -maxval * 4,
                  np.float32(1e-45), -np.float32(1e-45)], dtype=np.float32)
    got = oracle.fp8_encode(p, fmt)
    assert list(got) == [0x7F, 0x7F, maxcode, 0x80 | maxcode, 0x00, 0x80, maxcode,
                         0x80 | maxcode, 0x00, 0x80]
