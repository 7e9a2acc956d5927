"""MXFP4 and NVFP4 expert weights: E2M1 codes with block scales.

"SGLang Paged Experts: corré MoE más grandes que tu VRAM" (blog.donweb.com),
"¿Qué es la paginación de expertos…?": the second paging change added, among
other formats, MXFP4 and NVFP4 experts.  "¿Paginar expertos afecta la
calidad…?": the MXFP4 experts of one model are padded by its kernel (a width
of 2880 becomes 2944 or 3072), and before the fix the paged copies lacked that
padding and every answer came out wrong.  The pages name the formats only;
their definitions are the public ones:

* E2M1 (a 4-bit float): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa
  bit; exponent 0 is subnormal (value m/2); no infinity or NaN.  The sixteen
  values are +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* MXFP4: every 32 consecutive weights along the input dimension share one
  E8M0 scale, an 8-bit biased exponent: value 2^(e - 127), e = 255 is NaN.
  W = e2m1(q) * 2^(e - 127).
* NVFP4: every 16 consecutive inputs share one E4M3 scale (the FP8 "fn"
  format of oracle.fp8) and the whole tensor one fp32 scale g:
  W = e2m1(q) * e4m3(s) * g.

Layout read here (the pages fix none): codes [N, K/2] bytes, input 2j in the
low nibble of byte j (as the int4 row layout); block scales [N, K/B] bytes
(B = 32 or 16), blocks in input order.  This module works on the logical
shape; the expert-row padding of the library is a storage matter and is
checked against this unpadded arithmetic.
"""

from __future__ import annotations

import numpy as np

from . import fp8 as _fp8

MX_BLOCK = 32
NV_BLOCK = 16


def e2m1_value(code: int) -> float:
    """Decode one 4-bit E2M1 code from its bit fields."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:  # subnormal: m/2 * 2^(1 - bias), bias 1
        return sign * (man / 2.0)
    return sign * (1.0 + man / 2.0) * 2.0 ** (exp - 1)


_E2M1 = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """Decode integer E2M1 codes (0..15) elementwise to float64."""
    return _E2M1[np.asarray(codes, dtype=np.int64) & 0xF]


def e8m0_value(code: int) -> float:
    """2^(code - 127); NaN for 255."""
    code = int(code) & 0xFF
    return float("nan") if code == 255 else 2.0 ** (code - 127)


_E8M0 = np.array([e8m0_value(c) for c in range(256)], dtype=np.float64)


def decode_e8m0(codes: np.ndarray) -> np.ndarray:
    return _E8M0[np.asarray(codes, dtype=np.uint8)]


def unpack_rows(codes: np.ndarray) -> np.ndarray:
    """Row-layout codes [N, K/2] (uint8) -> 4-bit codes [N, K]."""
    c = np.asarray(codes, dtype=np.uint8)
    q = np.empty((c.shape[0], 2 * c.shape[1]), dtype=np.int64)
    q[:, 0::2] = c & 0xF
    q[:, 1::2] = c >> 4
    return q


def _block_scaled(codes, block_scale_values: np.ndarray, block: int) -> np.ndarray:
    w = decode_e2m1(unpack_rows(codes))
    n, k = w.shape
    if k % block or block_scale_values.shape != (n, k // block):
        raise ValueError("scale grid does not match the weight shape")
    return w * block_scale_values[:, np.arange(k) // block]


def dequant_mx(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """MXFP4: W[n, k] = e2m1(q[n, k]) * 2^(scales[n, k // 32] - 127), float64."""
    return _block_scaled(codes, decode_e8m0(scales), MX_BLOCK)


def dequant_nv(codes: np.ndarray, scales: np.ndarray, global_scale: float) -> np.ndarray:
    """NVFP4: W[n, k] = e2m1(q[n, k]) * e4m3(scales[n, k // 16]) * g, float64."""
    g = float(np.float32(global_scale))
    return _block_scaled(codes, _fp8.decode_e4m3(scales) * g, NV_BLOCK)
