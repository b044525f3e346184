"""The oracle's FP8 encode over every fp32 bit pattern (2^32 per format),
against the exhaustive nearest-code search of tests/fp8_search.py (ties to
the even code, saturation, signed zero, canonical NaN), on every host core.

Together with tests/test_gpu_codec.py (the GPU's conversion step against the
oracle over the same 2^32 patterns) this pins the conversion on every fp32
input: hardware == oracle == the definition.
"""
import pytest

import oracle
from oracle_pool import OraclePool


@pytest.fixture(scope="module")
def pool():
    with OraclePool() as p:
        yield p


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_oracle_encode_of_every_fp32_pattern(pool, fmt):
    res = pool.check_encode_against_search(0, 1 << 31, fmt)   # and each with its sign bit set
    assert res["bad"] == 0, (f"{res['bad']} patterns differ; first {res['first'][0]:#010x}: "
                             f"oracle {res['first'][1]:#04x}, search {res['first'][2]:#04x}")
