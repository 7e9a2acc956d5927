"""Seeded synthetic inputs for the paged MoE layer step.

This module only draws random numbers and packs them into the storage formats
the layer consumes (bf16 bit patterns, E4M3 byte codes, fp32 scales and router
logits).  It holds none of the layer's arithmetic: routing, planning, the
expert MLP and the merge live elsewhere.  Both the CUDA path and the CPU
reference draw their inputs from here, so the two always see the same bytes.

Workloads (the five shapes the layer is exercised on):

* ``tiny``        1 layer, H=256, I=128, E=16, top_k=2, K=6, bf16; 32 decode
                  steps at batch 1 plus one 64-token prefill chunk.
* ``decode48``    48 layers, H=2048, I=768, E=128, top_k=8, K=32, bf16;
                  batch-1 decode, 256 steps.
* ``graphed48``   same stack, K=64, decode batch 1/2/4/8 with an independent
                  router-bias stream per request.
* ``prefill48``   same stack, K=32, prefill chunks of 512 and 2048 tokens.
* ``fp8_48``      same stack with block-FP8 experts (E4M3, 128x128 blocks,
                  fp32 scales), K=40, decode batch 1 and 4, Zipf(1.1)
                  expert popularity on top of the drifting bias.

Router logits follow the decode recipe: a per-expert bias drawn N(0, sd=2)
that drifts by AR(1) with rho=0.9 from token to token (stationary sd kept at
2), plus fresh N(0, 1) noise per token.  Consecutive tokens therefore reuse
experts, which is the behaviour paging relies on (Paged Experts, SGLang docs,
"Why Paged Experts?").

Expert weights are N(0, 0.02) rounded to bf16.  Drawing 6144 independent
9.4 MB experts would take minutes on a CPU, so every expert is a distinct
window of one seeded pool of N(0, 0.02) values: expert ``i = layer*E + e``
starts ``i * stride`` elements into the pool.  Windows of different experts
start at different offsets, so no two experts hold the same tensor.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

# ----------------------------------------------------------------------------
# shapes


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """Static shape of one paged MoE stack."""

    num_layers: int
    num_experts: int
    top_k: int
    num_slots: int
    hidden: int
    intermediate: int
    dtype: str = "bf16"  # "bf16", "fp8" (E4M3, 128x128 blocks, fp32 scales),
    # "int4" (GPTQ: 4-bit codes, zero point 8, fp16 scale per output row and 128 inputs),
    # "mxfp4" (E2M1 codes, E8M0 scale per row and 32 inputs) or
    # "nvfp4" (E2M1 codes, E4M3 scale per row and 16 inputs, fp32 scale per tensor)
    block: int = 128

    @property
    def is_fp4(self) -> bool:
        return self.dtype in ("mxfp4", "nvfp4")

    @property
    def fp4_block(self) -> int:
        return 32 if self.dtype == "mxfp4" else 16

    def with_slots(self, k: int) -> "MoEShape":
        return dataclasses.replace(self, num_slots=k)

    # byte layout of one expert row (identical in the host store and a slot)
    @property
    def w13_elems(self) -> int:
        return 2 * self.intermediate * self.hidden

    @property
    def w2_elems(self) -> int:
        return self.hidden * self.intermediate

    @property
    def s13_shape(self) -> tuple[int, int]:
        b = self.block
        if self.is_fp4:
            return (2 * self.intermediate, self.hidden // self.fp4_block)
        if self.dtype == "int4":
            return (2 * self.intermediate, -(-self.hidden // b))
        return (-(-2 * self.intermediate // b), -(-self.hidden // b))

    @property
    def s2_shape(self) -> tuple[int, int]:
        b = self.block
        if self.is_fp4:
            return (self.hidden, self.intermediate // self.fp4_block)
        if self.dtype == "int4":
            return (self.hidden, -(-self.intermediate // b))
        return (-(-self.hidden // b), -(-self.intermediate // b))

    @property
    def expert_bytes(self) -> int:
        """Payload bytes of one expert (weights plus, for FP8 and int4, its scales)."""
        if self.dtype == "bf16":
            return 2 * (self.w13_elems + self.w2_elems)
        s13 = self.s13_shape[0] * self.s13_shape[1]
        s2 = self.s2_shape[0] * self.s2_shape[1]
        if self.is_fp4:  # codes, one byte per block scale, NVFP4 also two fp32 tensor scales
            return (self.w13_elems + self.w2_elems) // 2 + s13 + s2 + (8 if self.dtype == "nvfp4" else 0)
        if self.dtype == "int4":
            return (self.w13_elems + self.w2_elems) // 2 + 2 * (s13 + s2)
        return self.w13_elems + self.w2_elems + 4 * (s13 + s2)


TINY = MoEShape(1, 16, 2, 6, 256, 128, "bf16")
STACK48 = MoEShape(48, 128, 8, 32, 2048, 768, "bf16")
STACK48_FP8 = MoEShape(48, 128, 8, 40, 2048, 768, "fp8")
STACK48_INT4 = MoEShape(48, 128, 8, 92, 2048, 768, "int4")
STACK48_MXFP4 = MoEShape(48, 128, 8, 92, 2048, 768, "mxfp4")
STACK48_NVFP4 = MoEShape(48, 128, 8, 92, 2048, 768, "nvfp4")


# ----------------------------------------------------------------------------
# storage-format packing (inputs only)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest even) and return the uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32; exact."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _encode_e4m3(a: np.ndarray) -> np.ndarray:
    """Encode fp32 values (|a| <= 448) as OCP E4M3 byte codes (RNE).

    Uses torch's float8_e4m3fn conversion on the CPU: this is how a checkpoint
    would have been quantised, not part of the layer step.
    """
    import torch

    t = torch.from_numpy(np.clip(a, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


# ----------------------------------------------------------------------------
# expert weights


class ExpertWeights:
    """Deterministic synthetic expert weights, one window of a seeded pool each.

    ``row(layer, expert)`` returns a dict of numpy arrays in the storage
    format: bf16 experts give ``w13`` ([2I, H] uint16 bf16 bits, rows 0..I-1 the
    gate projection, rows I..2I-1 the up projection) and ``w2`` ([H, I]); FP8
    experts give E4M3 codes (uint8) for ``w13``/``w2`` plus fp32 block scales
    ``s13`` ([ceil(2I/128), ceil(H/128)]) and ``s2`` ([ceil(H/128), ceil(I/128)]);
    GPTQ int4 experts give packed 4-bit codes (uint8, [2I, H/2] and [H, I/2],
    input 2j in the low nibble of byte j) plus fp16 scales ``s13`` ([2I, H/128])
    and ``s2`` ([H, I/128]).  MXFP4 / NVFP4 experts give packed E2M1 codes in
    the same layout plus byte scale grids ``s13`` ([2I, H/32] E8M0 or
    [2I, H/16] E4M3) and ``s2``; NVFP4 also the fp32 tensor scales ``g13`` and
    ``g2``.
    """

    def __init__(self, shape: MoEShape, seed: int = 0, std: float = 0.02):
        self.shape = shape
        self.seed = seed
        n = shape.w13_elems + shape.w2_elems
        if shape.dtype == "int4" or shape.is_fp4:
            n //= 2  # two codes per byte
        n_experts = shape.num_layers * shape.num_experts
        pool = max(1 << 25, n + 64 * n_experts)
        rng = np.random.default_rng([seed, 0x5EED, 1])
        if shape.dtype == "int4":
            # codes 8 + round(N(0, 2.5)) in 0..15; with scales |N(0,1)|*0.008
            # the weights are of the 0.02 scale of the bf16 experts
            z = rng.standard_normal(2 * pool, dtype=np.float32)
            q = np.clip(np.rint(z * np.float32(2.5)) + 8, 0, 15).astype(np.uint8)
            self._pool = q[0::2] | (q[1::2] << 4)
            z = None
        elif shape.is_fp4:
            # E2M1 codes of N(0, 1.5): the nearest of the magnitudes
            # 0, .5, 1, 1.5, 2, 3, 4, 6 (ties away from zero) and the sign bit
            z = rng.standard_normal(2 * pool, dtype=np.float32) * np.float32(1.5)
            mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
            q = np.searchsorted(mids, np.abs(z), side="right").astype(np.uint8) | ((z < 0).astype(np.uint8) << 3)
            self._pool = q[0::2] | (q[1::2] << 4)
            z = None
        else:
            z = rng.standard_normal(pool, dtype=np.float32)
        if shape.dtype == "bf16":
            self._pool = f32_to_bf16_bits(z * np.float32(std))
        elif shape.dtype == "fp8":
            # E4M3 codes with sd 2; the per-block scale |N(0,1)|*0.01 brings
            # code*scale to the 0.02 scale of the bf16 experts.
            self._pool = _encode_e4m3(z * np.float32(2.0))
        self._n = n
        self._stride = ((pool - n) // n_experts) // 8 * 8
        assert self._stride >= 8

    def offset(self, layer: int, expert: int) -> int:
        return (layer * self.shape.num_experts + expert) * self._stride

    def row(self, layer: int, expert: int) -> dict[str, np.ndarray]:
        s = self.shape
        o = self.offset(layer, expert)
        win = self._pool[o : o + self._n]
        if s.dtype == "int4" or s.is_fp4:
            n13 = s.w13_elems // 2
            w13 = win[:n13].reshape(2 * s.intermediate, s.hidden // 2)
            w2 = win[n13:].reshape(s.hidden, s.intermediate // 2)
        else:
            w13 = win[: s.w13_elems].reshape(2 * s.intermediate, s.hidden)
            w2 = win[s.w13_elems :].reshape(s.hidden, s.intermediate)
        out = {"w13": w13, "w2": w2}
        if s.dtype == "fp8":
            rng = np.random.default_rng([self.seed, 0x5CA1E, layer, expert])
            out["s13"] = (np.abs(rng.standard_normal(s.s13_shape)) * 0.01).astype(np.float32)
            out["s2"] = (np.abs(rng.standard_normal(s.s2_shape)) * 0.01).astype(np.float32)
        elif s.dtype == "int4":
            rng = np.random.default_rng([self.seed, 0x5CA1E, layer, expert])
            out["s13"] = (np.abs(rng.standard_normal(s.s13_shape)) * 0.008).astype(np.float16)
            out["s2"] = (np.abs(rng.standard_normal(s.s2_shape)) * 0.008).astype(np.float16)
        elif s.dtype == "mxfp4":
            # E8M0 exponents 2^-8 .. 2^-6 per block: weights of the 0.02 scale
            rng = np.random.default_rng([self.seed, 0x5CA1E, layer, expert])
            out["s13"] = rng.integers(119, 122, size=s.s13_shape).astype(np.uint8)
            out["s2"] = rng.integers(119, 122, size=s.s2_shape).astype(np.uint8)
        elif s.dtype == "nvfp4":
            # E4M3 block scales |N(1, 0.25)| and a tensor scale near 0.015
            rng = np.random.default_rng([self.seed, 0x5CA1E, layer, expert])
            out["s13"] = _encode_e4m3(np.abs(rng.normal(1.0, 0.25, s.s13_shape)).astype(np.float32))
            out["s2"] = _encode_e4m3(np.abs(rng.normal(1.0, 0.25, s.s2_shape)).astype(np.float32))
            out["g13"] = np.float32(0.015 * (1.0 + 0.1 * rng.standard_normal()))
            out["g2"] = np.float32(0.015 * (1.0 + 0.1 * rng.standard_normal()))
        return out


# ----------------------------------------------------------------------------
# router logits and hidden states


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(list(key)))


def zipf_log_prior(num_experts: int, s: float, rng: np.random.Generator) -> np.ndarray:
    """log of a Zipf(s) popularity over a seeded random ranking of the experts."""
    ranks = rng.permutation(num_experts)
    p = 1.0 / (ranks + 1.0) ** s
    p /= p.sum()
    return np.log(p)


def decode_logits(
    num_layers: int,
    num_experts: int,
    num_steps: int,
    batch: int = 1,
    seed: int = 0,
    tag: int = 0,
    bias_sd: float = 2.0,
    rho: float = 0.9,
    zipf_s: float | None = None,
) -> np.ndarray:
    """Router logits for decode, fp32 [num_layers, num_steps, batch, E].

    Each (layer, request) has its own bias stream: b_0 ~ N(0, bias_sd^2),
    b_{t+1} = rho*b_t + sqrt(1-rho^2)*bias_sd*eps_t, and logits_t = b_t + N(0,1).
    With ``zipf_s`` the log of a per-layer Zipf(s) popularity is added.
    """
    out = np.empty((num_layers, num_steps, batch, num_experts), np.float32)
    innov = math.sqrt(1.0 - rho * rho) * bias_sd
    for l in range(num_layers):
        prior = 0.0
        if zipf_s is not None:
            prior = zipf_log_prior(num_experts, zipf_s, _rng(seed, tag, 0x21BF, l))
        for r in range(batch):
            g = _rng(seed, tag, l, r)
            b = g.normal(0.0, bias_sd, num_experts)
            eps = g.standard_normal((num_steps, num_experts))
            noise = g.standard_normal((num_steps, num_experts))
            for t in range(num_steps):
                out[l, t, r] = b + noise[t] + prior
                b = rho * b + innov * eps[t]
    return out


def prefill_logits(
    num_layers: int, num_experts: int, num_tokens: int, seed: int = 0, tag: int = 1
) -> np.ndarray:
    """Router logits for one prefill chunk, fp32 [num_layers, num_tokens, E]:
    a per-chunk bias N(0,1) per expert plus per-token N(0,1) noise."""
    out = np.empty((num_layers, num_tokens, num_experts), np.float32)
    for l in range(num_layers):
        g = _rng(seed, tag, l, num_tokens)
        bias = g.standard_normal(num_experts)
        out[l] = bias[None, :] + g.standard_normal((num_tokens, num_experts))
    return out


def hidden_states(shape: tuple[int, ...], hidden: int, seed: int = 0, tag: int = 2) -> np.ndarray:
    """N(0,1) hidden states as bf16 bits, uint16 [*shape, hidden]."""
    g = _rng(seed, tag, *shape, hidden)
    z = g.standard_normal((*shape, hidden), dtype=np.float32)
    return f32_to_bf16_bits(z)
