"""Expert MLP, merged buffer, top-k sum and the whole paged layer step.

Follows "Paged Experts" (SGLang docs), "A step: waves, page-in, merge",
items 3-4, and "Correctness".  Each routed (token, expert) pair yields one
entry: the expert's gated MLP applied to the token, scaled by that pair's
router weight, with no summation over the token's experts at that point.
Whichever wave holds the expert fills the entry, once, in a single buffer
shared by all waves; each token's k entries are added afterwards.  Since no
entry depends on the wave that produced it, splitting the experts into waves
cannot change the result, and the paged layer equals the plain MoE layer
("Why Paged Experts?", "Correctness").

Readings where the pages are silent:
  * the expert MLP is the SiLU-gated one the workload description names:
    h = SiLU(x Wg^T) * (x Wu^T), y = h Wd^T, with SiLU(z) = z / (1 + e^-z);
  * the gate and up projections are stacked in one [2I, H] tensor "w13":
    rows 0..I-1 are the gate, rows I..2I-1 the up projection; "w2" is the
    [H, I] down projection;
  * the router weight multiplies the down-projection output;
  * the top-k sum adds the k entries of a token in entry order j = 0..k-1.
All arithmetic is float64; storage formats are widened exactly first.
"""

from __future__ import annotations

from typing import Callable

import numpy as np

from . import fp4 as _fp4
from . import fp8 as _fp8
from . import int4 as _int4
from .lru import ResidencySim, StepPlan
from .routing import route


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def expert_weights(row: dict, dtype: str, block: int = 128) -> tuple[np.ndarray, np.ndarray]:
    """(w13, w2) in float64 from one expert's storage-format arrays."""
    if dtype == "bf16":
        return bf16_to_f64(row["w13"]), bf16_to_f64(row["w2"])
    if dtype == "fp8":
        return (
            _fp8.dequant_block(row["w13"], row["s13"], block),
            _fp8.dequant_block(row["w2"], row["s2"], block),
        )
    if dtype == "int4":
        return (
            _int4.dequant_rows(row["w13"], row["s13"], block),
            _int4.dequant_rows(row["w2"], row["s2"], block),
        )
    if dtype == "mxfp4":
        return _fp4.dequant_mx(row["w13"], row["s13"]), _fp4.dequant_mx(row["w2"], row["s2"])
    if dtype == "nvfp4":
        return (
            _fp4.dequant_nv(row["w13"], row["s13"], row["g13"]),
            _fp4.dequant_nv(row["w2"], row["s2"], row["g2"]),
        )
    raise ValueError(f"unsupported expert dtype {dtype!r}")


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def expert_mlp(x: np.ndarray, w13: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """SiLU-gated MLP of one expert for a batch of rows x [M, H] -> [M, H]."""
    inter = w2.shape[1]
    gate = x @ w13[:inter].T
    up = x @ w13[inter:].T
    return (silu(gate) * up) @ w2.T


def topk_sum(merged: np.ndarray) -> np.ndarray:
    """out[t] = sum_j merged[t, j] in entry order j = 0..k-1."""
    acc = np.zeros((merged.shape[0], merged.shape[2]), np.float64)
    for j in range(merged.shape[1]):
        acc = acc + merged[:, j]
    return acc


ExpertFn = Callable[[int], tuple[np.ndarray, np.ndarray]]


def moe_entries(
    x: np.ndarray, ids: np.ndarray, weights: np.ndarray, experts: list[int], get_expert: ExpertFn,
    merged: np.ndarray,
) -> None:
    """Write merged[t, j] = w_tj * MLP_e(x_t) for every entry whose expert is in
    ``experts`` (batched per expert over all of that expert's tokens)."""
    for e in experts:
        t_idx, j_idx = np.nonzero(ids == e)
        if t_idx.size == 0:
            continue
        w13, w2 = get_expert(e)
        y = expert_mlp(x[t_idx], w13, w2)
        merged[t_idx, j_idx] = weights[t_idx, j_idx, None] * y


def unpaged_layer(x_bits: np.ndarray, logits: np.ndarray, top_k: int, get_expert: ExpertFn) -> np.ndarray:
    """The plain MoE layer: route, run every routed entry, top-k sum. float64 [T, H]."""
    x = bf16_to_f64(x_bits)
    ids, w, _ = route(logits, top_k)
    merged = np.zeros((x.shape[0], top_k, x.shape[1]), np.float64)
    moe_entries(x, ids, w, sorted(set(ids.reshape(-1).tolist())), get_expert, merged)
    return topk_sum(merged)


class PagedLayer:
    """One paged MoE layer: K-slot table over a host store of all E experts.

    ``get_host_expert(e)`` plays the host store; ``self.slots`` is the K-slot
    table (what each slot holds after the page-ins planned so far), and the
    MLP of an entry reads its weights from the slot its remapped id names.
    """

    def __init__(self, num_experts: int, num_slots: int, top_k: int, get_host_expert: ExpertFn):
        self.sim = ResidencySim(num_experts, num_slots)
        self.top_k = top_k
        self.host = get_host_expert
        self.slots: list = [None] * num_slots

    def step(self, x_bits: np.ndarray, logits: np.ndarray, wave_order=None):
        """Run one layer step.  Returns (out float64 [T,H], merged, plan, ids, w).

        ``wave_order``: optional list of waves (lists of experts) to compute in
        instead of the plan's own; used to check wave-split invariance.
        """
        x = bf16_to_f64(x_bits)
        ids, w, _ = route(logits, self.top_k)
        plan: StepPlan = self.sim.step(ids)
        T, H = x.shape
        merged = np.zeros((T, self.top_k, H), np.float64)
        for wi, wave in enumerate(plan.waves):
            for e, s in zip(wave.plan_expert, wave.plan_slot):
                self.slots[s] = (e, self.host(e))
            if wave_order is not None:
                continue
            mask = plan.entry_wave == wi
            for e in wave.experts:
                t_idx, j_idx = np.nonzero((ids == e) & mask)
                slot = int(plan.entry_slot[t_idx[0], j_idx[0]])
                held, (w13, w2) = self.slots[slot]
                assert held == e, "slot does not hold the routed expert"
                y = expert_mlp(x[t_idx], w13, w2)
                merged[t_idx, j_idx] = w[t_idx, j_idx, None] * y
        if wave_order is not None:
            for members in wave_order:
                moe_entries(x, ids, w, members, self.host, merged)
        return topk_sum(merged), merged, plan, ids, w
