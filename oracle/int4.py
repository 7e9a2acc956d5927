"""GPTQ int4 expert weights: 4-bit codes and per-group dequantisation.

"Paged Experts" (SGLang docs), "Supported Configurations and Limitations":
GPTQ int4 experts are supported.  A GPTQ weight matrix W[N, K] (N output
rows, K inputs) is stored as 4-bit integer codes q in 0..15 with one scale
per output row and group of `group` consecutive inputs.  Symmetric GPTQ has
the zero point 8, so the dequantised weight is

    W[n, k] = (q[n, k] - 8) * s[n, k // group].

Readings (the pages name the format but not its details):
* symmetric quantisation, no zero-point tensor, group size 128, fp16 scales,
  groups in input order (no activation reordering).  This is exactly the
  pages' "2.43 MB per expert" for H = 2048, I = 768: 3*H*I/2 bytes of codes
  plus 2 bytes per (row, group) scale ("Choosing K" and the blog's
  "¿Por qué es rápido…?"): 2,359,296 + 73,728 = 2,433,024 B.

Two layouts of the same numbers appear here:
* the checkpoint layout: ``qweight`` int32 [K/8, N], the 8 codes of inputs
  8r..8r+7 of column n packed into word (r, n) from the low nibble up;
  ``scales`` [K/group, N];
* the expert-row layout the layer consumes: ``codes`` uint8 [N, K/2], byte j
  of row n holding input 2j in its low nibble and 2j+1 in its high nibble;
  ``scales`` [N, K/group].
"""

from __future__ import annotations

import numpy as np


def unpack_rows(codes: np.ndarray) -> np.ndarray:
    """Row-layout codes [N, K/2] (uint8) -> integer codes [N, K]."""
    c = np.asarray(codes, dtype=np.uint8)
    q = np.empty((c.shape[0], 2 * c.shape[1]), dtype=np.int64)
    q[:, 0::2] = c & 0xF
    q[:, 1::2] = c >> 4
    return q


def dequant_rows(codes: np.ndarray, scales: np.ndarray, group: int = 128) -> np.ndarray:
    """W[n, k] = (q[n, k] - 8) * scales[n, k // group], float64."""
    q = unpack_rows(codes).astype(np.float64) - 8.0
    n, k = q.shape
    s = np.asarray(scales, dtype=np.float64)
    if s.shape != (n, -(-k // group)):
        raise ValueError("scale grid does not match the weight shape")
    return q * s[:, np.arange(k) // group]


def unpack_gptq(qweight: np.ndarray) -> np.ndarray:
    """Checkpoint-layout qweight int32 [K/8, N] -> integer codes [K, N]."""
    w = np.asarray(qweight).astype(np.int64) & 0xFFFFFFFF
    k8, n = w.shape
    q = np.empty((8 * k8, n), dtype=np.int64)
    for i in range(8):
        q[i::8] = (w >> (4 * i)) & 0xF
    return q


def dequant_gptq(qweight: np.ndarray, scales: np.ndarray, group: int = 128) -> np.ndarray:
    """Checkpoint layout -> W[N, K] (output rows first), float64."""
    q = unpack_gptq(qweight).astype(np.float64) - 8.0
    k, n = q.shape
    s = np.asarray(scales, dtype=np.float64)
    if s.shape != (-(-k // group), n):
        raise ValueError("scale grid does not match the weight shape")
    return (q * s[np.arange(k) // group, :]).T
