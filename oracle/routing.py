"""Routing reference: softmax over all E experts, top-k, renormalise.

The paged layer leaves routing untouched and E-wide ("Paged Experts", SGLang
docs, "Why Paged Experts?"): every token is routed to top_k of the E experts
of the layer ("SGLang Paged Experts: corré MoE más grandes que tu VRAM",
"¿Qué es la paginación de expertos…?": 8 of 128).  The pages do not spell the
router out; the plainest reading, used here, is the usual one: p = softmax(l)
over E, keep the k largest, divide each kept p by the sum of the kept ones.

Readings where the pages are silent:
  * selection is made on the logits (softmax is strictly increasing, so the k
    largest logits are the k largest probabilities); entries are ordered by
    descending logit and equal logits go to the lower expert id first;
  * a NaN logit is treated as -inf for selection and reported through the
    returned flag;
  * a token whose logits are all NaN (all -inf) gets equal weights 1/k on the
    experts chosen by the tie rule (ids 0..k-1): the softmax is undefined there.
"""

from __future__ import annotations

import numpy as np


def softmax(logits: np.ndarray) -> np.ndarray:
    """Row-wise softmax in float64 (max subtracted for range)."""
    z = np.asarray(logits, dtype=np.float64)
    z = z - np.max(z, axis=-1, keepdims=True)
    e = np.exp(z)
    return e / np.sum(e, axis=-1, keepdims=True)


def route(logits: np.ndarray, top_k: int) -> tuple[np.ndarray, np.ndarray, bool]:
    """Route every token to its top_k experts.

    Args:
      logits: router logits, float32 [T, E].
      top_k: experts per token (1 <= top_k <= E).

    Returns:
      ids:     int32 [T, top_k], descending logit, ties to the lower id.
      weights: float64 [T, top_k], softmax over E restricted to the chosen
               experts and renormalised to sum to one.
      had_nan: True if any logit was NaN (treated as -inf).
    """
    l = np.asarray(logits, dtype=np.float32)
    T, E = l.shape
    if not 1 <= top_k <= E:
        raise ValueError("top_k out of range")
    had_nan = bool(np.isnan(l).any())
    sel = np.where(np.isnan(l), -np.inf, l).astype(np.float64)
    ids = np.empty((T, top_k), np.int32)
    expert = np.arange(E)
    for t in range(T):
        # primary key: descending logit; secondary: ascending id
        order = np.lexsort((expert, -sel[t]))
        ids[t] = order[:top_k]
    dead = np.all(np.isneginf(sel), axis=1)
    p = softmax(np.where(dead[:, None], 0.0, sel))
    kept = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    weights = kept / np.sum(kept, axis=1, keepdims=True)
    return ids, weights, had_nan
