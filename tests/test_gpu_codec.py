"""The cast kernels' FP8 conversion step on the GPU against the oracle, over
every fp32 bit pattern.

ct_fp8_convert_f32 runs the device routine that every cast kernel applies to
the product x * scale, without the scale.  All 2^32 fp32 patterns go through
it for each format, in chunks of 2^28 generated on the GPU, and every code is
compared with the oracle's encode of the same pattern (run on every host core
through tests/oracle_pool.py): finite values on and between the FP8 grid,
ties, values past the largest normal (saturation), +-Inf, every NaN payload of
either sign, signed zeros and fp32 subnormals.  Bit-exact: a conversion is an
integer decision taken in fp32 on both sides.
"""
import numpy as np
import pytest
import torch

import cast_transpose_gb300 as ct
from oracle_pool import OraclePool

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


@pytest.fixture(scope="module")
def pool():
    with OraclePool() as p:
        yield p


def _patterns(p0: int) -> torch.Tensor:
    """fp32 values with bit patterns p0 .. p0 + CHUNK - 1 (CHUNK-aligned p0,
    so a chunk never crosses the sign bit and the int32 range is contiguous)."""
    s0 = p0 if p0 < (1 << 31) else p0 - (1 << 32)
    return torch.arange(s0, s0 + CHUNK, dtype=torch.int32, device="cuda").view(torch.float32)


@pytest.mark.parametrize("fmt", [ct.E4M3, ct.E5M2])
def test_conversion_of_every_fp32_pattern(pool, fmt):
    codes = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    host = torch.from_numpy(pool.codes(CHUNK))
    bad, first = 0, None
    for p0 in range(0, 1 << 32, CHUNK):
        x = _patterns(p0)
        codes.fill_(0xA5)
        ct.fp8_convert_f32(x, codes, fmt)
        host.copy_(codes)          # synchronous device-to-host copy into shared memory
        res = pool.check_encode_patterns(p0, CHUNK, fmt)
        bad += res["bad"]
        if res["bad"] and first is None:
            first = res["first"]
        del x
    del host
    assert bad == 0, (f"{bad} codes differ from the oracle; first: pattern "
                      f"{first[0]:#010x} gave {first[1]:#04x}, oracle {first[2]:#04x}")


def test_odd_length_and_offsets():
    """n odd (the last value has no partner) and an output at an odd byte:
    every code lands where it belongs and nothing past the end is written."""
    import oracle
    vals = np.array([1.0, -1.0625, 500.0, np.nan, -0.0, 2.0 ** -10, np.inf], dtype=np.float32)
    x = torch.from_numpy(vals).cuda()
    buf = torch.full((16,), 0xA5, dtype=torch.uint8, device="cuda")
    ct.fp8_convert_f32(x, buf[3:3 + vals.size], ct.E4M3)
    got = buf.cpu().numpy()
    assert np.array_equal(got[3:3 + vals.size], oracle.fp8_encode(vals, oracle.E4M3))
    assert np.all(got[:3] == 0xA5) and np.all(got[3 + vals.size:] == 0xA5)
