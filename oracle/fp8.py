"""Block-FP8 expert weights: E4M3 decoding and 128x128 block dequantisation.

"Paged Experts" (SGLang docs, "Supported Configurations and Limitations")
supports block-quantised FP8 experts with a [128, 128] weight block size: each
weight is an 8-bit E4M3 code and every 128x128 block of a weight matrix has
one fp32 scale.  The dequantised weight is code_value * block_scale.

E4M3 here is the OCP "fn" variant: 1 sign bit, 4 exponent bits with bias 7,
3 mantissa bits, no infinities, only S.1111.111 is NaN, largest finite 448.
"""

from __future__ import annotations

import numpy as np


def e4m3_value(code: int) -> float:
    """Decode one E4M3 byte to its real value (NaN for the two NaN codes)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:  # subnormal: man/8 * 2^(1-7)
        return sign * (man / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """Decode an array of E4M3 codes (uint8) to float64, elementwise."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def dequant_block(codes: np.ndarray, scales: np.ndarray, block: int = 128) -> np.ndarray:
    """W[n, c] = e4m3(codes[n, c]) * scales[n // block, c // block], float64.

    ``scales`` has shape [ceil(N/block), ceil(C/block)]; a ragged last block
    uses the same scale for its partial rows/columns.
    """
    w = decode_e4m3(codes)
    n, c = w.shape
    sr = np.arange(n) // block
    sc = np.arange(c) // block
    s = np.asarray(scales, dtype=np.float64)
    if s.shape != (-(-n // block), -(-c // block)):
        raise ValueError("scale grid does not match the weight shape")
    return w * s[sr][:, sc]
