"""The parallel oracle checker (tests/oracle_pool.py) on the CPU.

The checker is what the full-size GPU parity tests rely on, so it is checked
here against the oracle's own single-process result: with the oracle's output
planted as the "device" result it must report zero differences and the same
amax; a single flipped byte of q or of qT must be found at its exact place; and
the conversion check over a range of fp32 bit patterns must agree with the
oracle's encode of the same patterns and find a planted wrong code.
"""
import numpy as np
import pytest
import torch

import oracle
from cast_transpose_gb300 import workloads
from oracle_pool import OraclePool


@pytest.fixture(scope="module")
def pool():
    with OraclePool(workers=3) as p:
        yield p


@pytest.mark.parametrize("rows,cols,fmt", [(300, 136, oracle.E4M3), (97, 33, oracle.E5M2)])
def test_pool_agrees_with_the_oracle_and_finds_planted_bytes(pool, rows, cols, fmt):
    x = workloads.normal_bf16(rows, cols, 30.0, 77)
    ref = oracle.cast_transpose(x, 1.5, fmt)
    xin = pool.input_bf16(rows, cols)
    xin[:] = x.view(torch.int16).numpy().view(np.uint16)
    q, qt = pool.output_q(rows, cols), pool.output_qt(rows, cols)
    q[:] = ref["q"]
    qt[:] = ref["qt"]
    res = pool.check_cast_transpose(rows, cols, 1.5, fmt, block_rows=41)
    assert res["bad_q"] == 0 and res["bad_qt"] == 0
    assert res["amax"].view(np.uint32) == np.float32(ref["amax"]).view(np.uint32)

    q[rows - 2, cols - 3] ^= 0x01
    qt[5, rows - 1] ^= 0x80
    res = pool.check_cast_transpose(rows, cols, 1.5, fmt, block_rows=41)
    assert res["bad_q"] == 1 and res["first_q"] == (rows - 2, cols - 3)
    assert res["bad_qt"] == 1 and res["first_qt"] == (5, rows - 1)
    del xin, q, qt


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_pool_pattern_check(pool, fmt):
    p0, n = 0x3F7F0000, 1 << 17          # patterns around 1.0 and up
    pats = np.arange(p0, p0 + n, dtype=np.uint64).astype(np.uint32)
    codes = pool.codes(n)
    codes[:] = oracle.fp8_encode(pats.view(np.float32), fmt)
    assert pool.check_encode_patterns(p0, n, fmt, chunk=5000)["bad"] == 0
    codes[1234] ^= 0x01
    res = pool.check_encode_patterns(p0, n, fmt, chunk=5000)
    assert res["bad"] == 1 and res["first"][0] == p0 + 1234
    del codes
