"""Exactness facts the 4-bit converters of the prefill GEMM rely on, checked
over every code on the CPU (no GPU, no library call).

The prefill converters decode 2*e2m1(q) as a bf16 pair and multiply it by
half of its block scale, rounded to bf16 once, in one packed bf16 multiply;
NVFP4's fp32 tensor scale is applied later, to the fp32 accumulators.  That
gives exactly e2m1(q) * block scale (before the tensor scale) only if

* 2*e2m1(q) is a bf16 value (for every 4-bit code),
* half of every finite block scale is a bf16 value (E8M0: a power of two;
  E4M3: four significant bits), and
* every product of the two is a bf16 value, so the multiply does not round.

Values come from the oracle's decoders (E2M1 from its bit fields, E4M3 and
E8M0 from theirs).
"""

import numpy as np

from oracle import fp4 as ofp4
from oracle import fp8 as ofp8


def _is_bf16(v: np.ndarray) -> np.ndarray:
    """True where a float64 value is exactly a (normal or zero) bf16 value."""
    v = np.asarray(v, dtype=np.float64)
    f = v.astype(np.float32)
    same = f.astype(np.float64) == v
    low = f.view(np.uint32) & np.uint32(0xFFFF)
    return same & (low == 0)


def test_bf16_check_itself():
    assert _is_bf16(np.array([0.0, 1.0, -1.5, 2.0**-126, 1.0 + 2.0**-7])).all()
    assert not _is_bf16(np.array([1.0 + 2.0**-8])).any()
    assert not _is_bf16(np.array([0.1])).any()


def test_twice_e2m1_is_bf16():
    two_v = 2.0 * ofp4.decode_e2m1(np.arange(16))
    assert _is_bf16(two_v).all()
    assert sorted(set(np.abs(two_v).tolist())) == [0.0, 1.0, 2.0, 3.0, 4.0, 6.0, 8.0, 12.0]


def test_mxfp4_products_are_exact():
    # E8M0 codes whose halves stay normal in bf16 (2^-126 and up; codes 0
    # and 1 give halves below the normal range) and whose weights stay finite
    # in bf16 and fp32 alike (6 * 2^(e - 127) < 2^128: e <= 252)
    codes = np.arange(2, 253)
    half = 0.5 * ofp4.decode_e8m0(codes)
    assert _is_bf16(half).all()
    prod = np.outer(2.0 * ofp4.decode_e2m1(np.arange(16)), half)
    assert _is_bf16(prod).all()
    assert np.array_equal(prod, np.outer(ofp4.decode_e2m1(np.arange(16)), ofp4.decode_e8m0(codes)))


def test_nvfp4_products_are_exact():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)  # 0x7F, 0xFF: NaN
    s = ofp8.decode_e4m3(codes)
    assert np.isfinite(s).all()
    half = 0.5 * s
    assert _is_bf16(half).all()
    prod = np.outer(2.0 * ofp4.decode_e2m1(np.arange(16)), half)
    assert _is_bf16(prod).all()
    assert np.array_equal(prod, np.outer(ofp4.decode_e2m1(np.arange(16)), s))
