"""The branch-free divide and square root of the AdamW epilogues with bf16 /
8-bit moments (forge_math.cuh: sqrt_fast, rcp_refined, div_fast) give the
correctly rounded result on their whole operand ranges: every case is
enumerated on the device (forge_selftest_math) against the hardware's
correctly rounded operations. The square root: every float in
[2^-100, 2^100]; the reciprocal: every divisor in [2^-60, 2^60]; the
quotient: every pair of significands, which with the correctly rounded
reciprocal covers every exponent of the ranges (no step leaves the normal
range there, so each case scales exactly)."""

import struct

import pytest

import backward_gemm_optimizer_gb300 as F

pytestmark = pytest.mark.gpu


def bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def test_sqrt_fast_every_float_in_range():
    lo, hi = bits(2.0 ** -100), bits(2.0 ** 100)
    mism, declined = F.selftest_math(0, lo, hi - lo + 1)
    assert (mism, declined) == (0, 0)
    # zero and the values below and above the range are left to the guarded
    # functions
    assert F.selftest_math(0, 0, 1) == (0, 1)
    assert F.selftest_math(0, lo - 1000, 1000) == (0, 1000)
    assert F.selftest_math(0, hi + 1, 1000) == (0, 1000)


def test_refined_reciprocal_every_divisor_in_range():
    lo, hi = bits(2.0 ** -60), bits(2.0 ** 60)
    assert F.selftest_math(1, lo, hi - lo + 1) == (0, 0)


def test_quotient_every_pair_of_significands():
    total, chunk = 1 << 46, 1 << 41
    for first in range(0, total, chunk):
        mism, declined = F.selftest_math(2, first, chunk)
        assert (mism, declined) == (0, 0), (first, mism, declined)
