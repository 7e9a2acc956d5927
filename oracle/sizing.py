"""Byte sizes and the miss-rate bound the pages work out by hand.

"SGLang Paged Experts: corré MoE más grandes que tu VRAM" (blog.donweb.com),
"¿Por qué es rápido si los expertos cruzan el PCIe en cada paso?": a token at
batch 1 touches layers*top_k experts; if every one missed, a token would move
layers*top_k*expert_bytes over the host link.  At a measured decode rate the
link can only have carried link_bw/tok_s bytes per token, which bounds the
fraction of expert activations that can have missed; uniform random routing
would miss 1 - K/E of them.  "Paged Experts" (SGLang docs, "Choosing K"): one
resident slot costs expert_bytes * num_moe_layers of GPU memory, so the
number of slots is what the memory left for the slot table allows (the
pages' formula itself did not survive extraction; the plainest reading is
the floor of that budget over the per-slot cost, kept within top_k..E).
"""

from __future__ import annotations


def expert_bytes(hidden: int, inter: int, dtype: str, block: int = 128) -> int:
    """Bytes of one expert: gate+up [2I, H] and down [H, I] weights, plus one
    fp32 scale per 128x128 block for block-FP8, or 4-bit codes plus one fp16
    scale per output row and 128-input group for GPTQ int4."""
    n = 3 * hidden * inter
    if dtype == "bf16":
        return 2 * n
    if dtype == "fp8":
        s13 = -(-2 * inter // block) * -(-hidden // block)
        s2 = -(-hidden // block) * -(-inter // block)
        return n + 4 * (s13 + s2)
    if dtype == "int4":  # 4-bit codes, one fp16 scale per output row and 128-input group
        s13 = 2 * inter * -(-hidden // block)
        s2 = hidden * -(-inter // block)
        return n // 2 + 2 * (s13 + s2)
    raise ValueError(dtype)


def slot_bytes(per_expert_bytes: float, num_moe_layers: int) -> float:
    """GPU memory of one resident slot across all MoE layers."""
    return per_expert_bytes * num_moe_layers


def all_miss_bytes_per_token(num_layers: int, top_k: int, per_expert_bytes: float) -> float:
    """Link bytes one batch-1 token would need if every routed expert missed."""
    return num_layers * top_k * per_expert_bytes


def max_miss_rate(link_bytes_per_s: float, tok_per_s: float, num_layers: int, top_k: int,
                  per_expert_bytes: float) -> float:
    """Largest miss fraction a measured decode rate allows over a given link."""
    return (link_bytes_per_s / tok_per_s) / all_miss_bytes_per_token(num_layers, top_k, per_expert_bytes)


def random_miss_rate(num_slots: int, num_experts: int) -> float:
    """Miss fraction of uniform random routing with K of E experts resident."""
    return 1.0 - num_slots / num_experts


def slots_for_budget(budget_bytes: float, fixed_bytes: float, per_slot_bytes: float, num_experts: int,
                     top_k: int) -> int:
    """K that a memory budget allows: floor((budget - fixed) / per_slot),
    at most E; 0 when not even top_k slots fit (the layer needs K >= top_k)."""
    if per_slot_bytes <= 0:
        raise ValueError("per-slot bytes must be positive")
    k = int((budget_bytes - fixed_bytes) // per_slot_bytes) if budget_bytes >= fixed_bytes else 0
    k = min(k, num_experts)
    return k if k >= top_k else 0
