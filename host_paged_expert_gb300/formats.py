"""Host-side conversion of checkpoint expert tensors into the expert-row
layout the layer consumes (the one-time repack a loader does before
pe_load_host_expert; "Paged Experts" (SGLang docs), "The K-slot table and the
host store": methods that repack their experts run the repack over the host
store, so host rows hold the layout the slots use).

GPTQ int4 checkpoints store a weight W[N, K] (N outputs, K inputs) as
``qweight`` int32 [K/8, N], the codes of inputs 8r..8r+7 of output n packed
into word (r, n) from the low nibble up, and fp16 ``scales`` [K/group, N].
The row layout is codes [N, K/2] bytes (input 2j in the low nibble of byte j)
and scales [N, K/group]: the same numbers, output-major.
"""

from __future__ import annotations

import numpy as np


def gptq_int4_to_row(qweight: np.ndarray, scales: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(qweight [K/8, N] int32, scales [K/group, N] fp16) -> (codes [N, K/2]
    uint8, scales [N, K/group] fp16).  Symmetric GPTQ only (zero point 8)."""
    w = np.ascontiguousarray(qweight).view(np.uint32)
    k8, n = w.shape
    nib = np.empty((8 * k8, n), dtype=np.uint8)
    for i in range(8):
        nib[i::8] = (w >> np.uint32(4 * i)) & np.uint32(0xF)
    nib = np.ascontiguousarray(nib.T)  # [N, K]
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return codes, np.ascontiguousarray(np.asarray(scales, dtype=np.float16).T)


def gate_up_rows(gate: tuple[np.ndarray, np.ndarray], up: tuple[np.ndarray, np.ndarray]) -> tuple[np.ndarray, np.ndarray]:
    """Stack the gate and up projections (each (codes, scales) in the row
    layout) into w13 = [gate; up] and s13, the order the layer reads."""
    return np.concatenate([gate[0], up[0]]), np.concatenate([gate[1], up[1]])
