"""Helpers shared by the GPU parity tests: build a paged stack from the seeded
generators, run the CPU oracle beside it, and compare."""

from __future__ import annotations

import numpy as np

from host_paged_expert_gb300 import synth
from oracle import mlp as omlp

# rel-L2 tolerances against the oracle: bf16 and block-FP8 as stated for the
# layer; GPTQ int4, MXFP4 and NVFP4 take the block-FP8 budget, their error
# sources being the same (exactly dequantised weights, bf16 rounding of h, of
# the output and, on the tensor cores, of each scaled weight)
REL_L2 = {"bf16": 1e-2, "fp8": 3e-2, "int4": 3e-2, "fp4": 3e-2, "mxfp4": 3e-2, "nvfp4": 3e-2}


def torch_mod():
    import torch

    return torch


def load_stack(model, weights: synth.ExpertWeights, layers=None):
    s = weights.shape
    for l in range(s.num_layers) if layers is None else layers:
        for e in range(s.num_experts):
            model.load_expert(l, e, weights.row(l, e))


def expert_fn(weights: synth.ExpertWeights, layer: int):
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = omlp.expert_weights(weights.row(layer, e), weights.shape.dtype)
        return cache[e]

    return get


def to_dev_bf16(bits: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev_f32(a: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def out_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def out_bits(t) -> np.ndarray:
    torch = torch_mod()
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def token_rel_l2(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """rel-L2 of every token (row) of a [T, H] output on its own."""
    num = np.linalg.norm(got - ref, axis=-1)
    den = np.maximum(np.linalg.norm(ref, axis=-1), 1e-300)
    return num / den


def max_token_rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    """The worst token's rel-L2: a wrong entry in one token of a long chunk
    shows here, where the whole output's norm would dilute it."""
    return float(token_rel_l2(got.reshape(-1, got.shape[-1]), ref.reshape(-1, ref.shape[-1])).max())


def check_tokens(got: np.ndarray, want: np.ndarray, tol: float, what) -> float:
    """Every token of an output within ``tol`` (rel-L2 of that token alone)
    of the oracle; prints and returns the worst token's figure."""
    worst = max_token_rel_l2(got, want)
    print(f"{what}: worst token rel-L2 {worst:.3e} (whole output {rel_l2(got, want):.3e})")
    assert worst <= tol, (what, worst)
    return worst


def check_plan(gpu: dict, plan, ids: np.ndarray, w: np.ndarray):
    """Bit-exact plan parity between the device planner and the oracle LRU."""
    assert np.array_equal(gpu["topk_id"], ids), "routed ids differ"
    assert np.allclose(gpu["topk_w"], w, rtol=2e-6, atol=1e-7), "router weights differ"
    assert gpu["num_waves"] == len(plan.waves)
    for wi, wave in enumerate(plan.waves):
        c = int(gpu["plan_count"][wi])
        assert c == wave.count, (wi, c, wave.count)
        assert gpu["plan_expert"][wi, :c].tolist() == wave.plan_expert
        assert gpu["plan_slot"][wi, :c].tolist() == wave.plan_slot
    for wi in range(len(plan.waves), gpu["plan_count"].shape[0]):
        assert gpu["plan_count"][wi] == 0
    assert np.array_equal(gpu["entry_wave"], plan.entry_wave)
    assert np.array_equal(gpu["entry_slot"], plan.entry_slot)


def check_residency(gpu: dict, sim):
    assert gpu["slot_expert"].tolist() == sim.slot_expert
    assert gpu["slot_tick"].tolist() == sim.slot_tick
    assert gpu["expert_slot"].tolist() == sim.expert_slot
    assert gpu["clock"] == sim.clock
