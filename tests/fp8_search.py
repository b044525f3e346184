"""FP8 encoding by exhaustive search over the decoded codes: the plain
definition of round-to-nearest with ties to even and saturation, written
independently of the oracle's binade arithmetic (the decoded grid comes from
torch's float8 dtypes, a library routine).  Used to pin the oracle's encode
(tests/test_oracle_codec*.py)."""
import numpy as np
import torch

E4M3, E5M2 = 0, 1
MAXCODE = {E4M3: 0x7E, E5M2: 0x7B}
MAXVAL = {E4M3: 448.0, E5M2: 57344.0}


def torch_decode(dtype) -> np.ndarray:
    """fp32 values of the 256 codes of a torch float8 dtype."""
    return torch.arange(256, dtype=torch.uint8).view(dtype).float().numpy()


def nearest_code_by_search(p: np.ndarray, fmt: int) -> np.ndarray:
    """FP8 code of each fp32 value in p: the nearest of the decoded positive
    codes found by search (ties to the code whose last bit is 0), +-max
    beyond the largest normal and for +-Inf, the sign bit of p, and 0x7F for
    NaN."""
    maxcode, maxval = MAXCODE[fmt], MAXVAL[fmt]
    grid_codes = np.arange(maxcode + 1, dtype=np.int64)
    grid = torch_decode(torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2)
    grid = grid[: maxcode + 1].astype(np.float64)
    assert np.all(np.diff(grid) > 0)
    with np.errstate(invalid="ignore"):      # signalling-NaN patterns among the inputs
        a = np.abs(p.astype(np.float64))
    hi = np.clip(np.searchsorted(grid, a, side="left"), 0, maxcode)
    lo = np.clip(hi - 1, 0, maxcode)
    d_lo = np.abs(a - grid[lo])
    d_hi = np.abs(grid[hi] - a)
    pick = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    pick = np.where(tie, np.where(grid_codes[lo] % 2 == 0, lo, hi), pick)
    pick = np.where(a >= maxval, maxcode, pick)
    sign = np.where(np.signbit(p), 0x80, 0)
    out = (pick | sign).astype(np.uint8)
    out[np.isnan(p)] = 0x7F
    return out
