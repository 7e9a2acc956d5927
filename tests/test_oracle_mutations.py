"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one of them (CPU only).  A mutant is the oracle module's own
source with one edit, executed as a fresh module."""

import importlib
import inspect
import sys
import types

import pytest

import pins


def mutant(modname, old, new):
    mod = importlib.import_module(modname)
    src = inspect.getsource(mod)
    assert src.count(old) >= 1, f"mutation target not found in {modname}: {old!r}"
    m = types.ModuleType(modname + "_mutant")
    m.__package__ = "oracle"
    sys.modules[m.__name__] = m  # dataclasses look their module up here
    try:
        exec(compile(src.replace(old, new), m.__name__, "exec"), m.__dict__)
    finally:
        del sys.modules[m.__name__]
    return m


MUTANTS = [
    # routing
    ("oracle.routing", "weights = kept / np.sum(kept, axis=1, keepdims=True)", "weights = kept",
     lambda m: pins.check_route_weights(m.route)),
    ("oracle.routing", "order = np.lexsort((expert, -sel[t]))", "order = np.lexsort((-expert, -sel[t]))",
     lambda m: pins.check_route_ties(m.route)),
    ("oracle.routing", "order = np.lexsort((expert, -sel[t]))", "order = np.lexsort((expert, sel[t]))",
     lambda m: pins.check_route_brute_force(m.route)),
    # fp8
    ("oracle.fp8", "2.0 ** (exp - 7)", "2.0 ** (exp - 8)", lambda m: pins.check_e4m3_table(m.decode_e4m3)),
    ("oracle.fp8", "(man / 8.0) * 2.0 ** (1 - 7)", "(man / 8.0) * 2.0 ** (0 - 7)",
     lambda m: pins.check_e4m3_table(m.decode_e4m3)),
    ("oracle.fp8", "return w * s[sr][:, sc]", "return w * s[0, 0]",
     lambda m: pins.check_block_dequant(m.dequant_block)),
    ("oracle.fp8", "sr = np.arange(n) // block", "sr = np.arange(n) % (-(-n // block))",
     lambda m: pins.check_block_dequant(m.dequant_block)),
    # int4
    ("oracle.int4", "q[:, 0::2] = c & 0xF", "q[:, 0::2] = c >> 4",
     lambda m: pins.check_int4_values(m.dequant_rows)),
    ("oracle.int4", "q = unpack_rows(codes).astype(np.float64) - 8.0", "q = unpack_rows(codes).astype(np.float64) - 7.0",
     lambda m: pins.check_int4_values(m.dequant_rows)),
    ("oracle.int4", "return q * s[:, np.arange(k) // group]", "return q * s[:, np.arange(k) % s.shape[1]]",
     lambda m: pins.check_int4_brute_force(m.dequant_rows)),
    ("oracle.int4", "q[i::8] = (w >> (4 * i)) & 0xF", "q[i::8] = (w >> (4 * (7 - i))) & 0xF",
     lambda m: pins.check_int4_gptq_layout(m.dequant_gptq)),
    # fp4 (MXFP4, NVFP4)
    ("oracle.fp4", "q[:, 0::2] = c & 0xF", "q[:, 0::2] = c >> 4",
     lambda m: pins.check_fp4_hand_values(m.dequant_mx, m.dequant_nv)),
    ("oracle.fp4", "return sign * (1.0 + man / 2.0) * 2.0 ** (exp - 1)", "return sign * (1.0 + man / 2.0) * 2.0 ** exp",
     lambda m: pins.check_e2m1_table(m.decode_e2m1)),
    ("oracle.fp4", "return sign * (man / 2.0)", "return sign * man",
     lambda m: pins.check_e2m1_table(m.decode_e2m1)),
    ("oracle.fp4", "sign = -1.0 if code & 0x8 else 1.0", "sign = -1.0 if code & 0x1 else 1.0",
     lambda m: pins.check_e2m1_table(m.decode_e2m1)),
    ("oracle.fp4", "else 2.0 ** (code - 127)", "else 2.0 ** (code - 128)",
     lambda m: pins.check_e8m0_table(m.decode_e8m0)),
    ("oracle.fp4", "return _block_scaled(codes, decode_e8m0(scales), MX_BLOCK)",
     "return _block_scaled(codes, decode_e8m0(scales), NV_BLOCK)",
     lambda m: pins.check_fp4_brute_force(m.dequant_mx, m.dequant_nv)),
    ("oracle.fp4", "_fp8.decode_e4m3(scales) * g", "_fp8.decode_e4m3(scales)",
     lambda m: pins.check_fp4_hand_values(m.dequant_mx, m.dequant_nv)),
    ("oracle.fp4", "return w * block_scale_values[:, np.arange(k) // block]",
     "return w * block_scale_values[:, np.arange(k) % block_scale_values.shape[1]]",
     lambda m: pins.check_fp4_brute_force(m.dequant_mx, m.dequant_nv)),
    # mlp
    ("oracle.mlp", "return (silu(gate) * up) @ w2.T", "return (silu(up) * gate) @ w2.T",
     lambda m: pins.check_mlp_hand(m.expert_mlp)),
    ("oracle.mlp", "return z / (1.0 + np.exp(-z))", "return z / (1.0 + np.exp(z))",
     lambda m: pins.check_silu(m.silu)),
    ("oracle.mlp", "return (silu(gate) * up) @ w2.T", "return silu(gate) @ w2.T",
     lambda m: pins.check_mlp_brute_force(m.expert_mlp)),
    ("oracle.mlp", "return (silu(gate) * up) @ w2.T", "return (silu(gate) * up) @ w2",
     lambda m: pins.check_mlp_brute_force(m.expert_mlp)),
    ("oracle.mlp", "for j in range(merged.shape[1]):", "for j in range(merged.shape[1] - 1):",
     lambda m: pins.check_topk_sum(m.topk_sum)),
    # lru
    ("oracle.lru", "key=lambda s: (self.slot_tick[s], s),", "key=lambda s: (-self.slot_tick[s], s),",
     lambda m: pins.check_lru_hand(m.ResidencySim)),
    ("oracle.lru", "key=lambda s: (self.slot_tick[s], s),", "key=lambda s: (self.slot_tick[s], -s),",
     lambda m: pins.check_lru_hand(m.ResidencySim)),
    ("oracle.lru", "self.slot_tick[self.expert_slot[e]] = self.clock", "pass",
     lambda m: pins.check_lru_textbook(m.ResidencySim, max_e=4, max_len=3)),
    ("oracle.lru", "order = R + M", "order = M + R",
     lambda m: pins.check_lru_textbook(m.ResidencySim, max_e=4, max_len=3)),
    ("oracle.lru", "missing = sorted(e for e in members if not self.resident(e))",
     "missing = sorted((e for e in members if not self.resident(e)), reverse=True)",
     lambda m: pins.check_lru_hand(m.ResidencySim)),
    ("oracle.lru", "self.clock += 1", "self.clock += 0",
     lambda m: pins.check_lru_textbook(m.ResidencySim, max_e=4, max_len=3)),
]


@pytest.mark.parametrize("modname,old,new,check", MUTANTS, ids=[f"{m[0]}:{i}" for i, m in enumerate(MUTANTS)])
def test_pins_catch_planted_mistake(modname, old, new, check):
    m = mutant(modname, old, new)
    with pytest.raises((AssertionError, ValueError)):
        check(m)
