"""The oracle against facts fixed outside itself (CPU only)."""

import numpy as np
import pytest

import pins
from oracle import fp8, int4, lru, mlp, routing, sizing


def test_route_brute_force():
    pins.check_route_brute_force(routing.route)


def test_route_weights_closed_forms():
    pins.check_route_weights(routing.route)


def test_route_ties_lower_id_first():
    pins.check_route_ties(routing.route)


def test_route_nan_is_minus_inf_and_flagged():
    pins.check_route_nan(routing.route)


def test_softmax_matches_scipy():
    import scipy.special

    z = np.random.default_rng(0).standard_normal((7, 33)) * 10
    assert np.allclose(routing.softmax(z), scipy.special.softmax(z, axis=-1), rtol=1e-13)


def test_e4m3_table_matches_torch():
    pins.check_e4m3_table(fp8.decode_e4m3)


def test_block_dequant_scale_grid():
    pins.check_block_dequant(fp8.dequant_block)


def test_block_dequant_rejects_bad_grid():
    with pytest.raises(ValueError):
        fp8.dequant_block(np.zeros((130, 10), np.uint8), np.ones((1, 1), np.float32))


def test_mlp_hand_example():
    pins.check_mlp_hand(mlp.expert_mlp)


def test_mlp_brute_force():
    pins.check_mlp_brute_force(mlp.expert_mlp)


def test_silu_closed_form():
    pins.check_silu(mlp.silu)


def test_topk_sum_order():
    pins.check_topk_sum(mlp.topk_sum)


def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x4049, 0x7F80, 0x0001], np.uint16)
    want = [1.0, -1.0, 0.0, -0.0, 3.140625, np.inf, 2.0**-133]
    got = mlp.bf16_to_f64(bits)
    assert got.tolist() == want


def test_lru_hand_traces():
    pins.check_lru_hand(lru.ResidencySim)


def test_lru_matches_textbook_exhaustive():
    pins.check_lru_textbook(lru.ResidencySim)


def _tiny_experts(E=6, H=8, I=4, seed=0):
    rng = np.random.default_rng(seed)
    w = [(rng.standard_normal((2 * I, H)), rng.standard_normal((H, I))) for _ in range(E)]
    return lambda e: w[e]


def _bf16(x):
    from host_paged_expert_gb300.synth import f32_to_bf16_bits

    return f32_to_bf16_bits(np.asarray(x, np.float32))


def test_unpaged_layer_equals_per_token_loop():
    get = _tiny_experts()
    rng = np.random.default_rng(5)
    xb = _bf16(rng.standard_normal((9, 8)))
    logits = rng.standard_normal((9, 6)).astype(np.float32)
    out = mlp.unpaged_layer(xb, logits, 2, get)
    ref = pins.layer_brute_force(mlp.bf16_to_f64(xb), logits, 2, get, routing.route)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_paged_step_equals_unpaged_bit_exact():
    """Several waves (K=2 < distinct experts) give exactly the unpaged output."""
    get = _tiny_experts()
    rng = np.random.default_rng(6)
    layer = mlp.PagedLayer(6, 2, 3, get)
    for step in range(6):
        T = 1 + step
        xb = _bf16(rng.standard_normal((T, 8)))
        logits = (rng.standard_normal((T, 6)) * 2).astype(np.float32)
        out, merged, plan, ids, w = layer.step(xb, logits)
        assert np.array_equal(out, mlp.unpaged_layer(xb, logits, 3, get))
        assert all(len(wv.experts) <= 2 for wv in plan.waves)
        layer.sim.check_invariants()


def test_wave_split_invariance_bit_exact():
    """Any partition of the distinct experts into waves gives the same bits."""
    get = _tiny_experts(E=8)
    rng = np.random.default_rng(7)
    xb = _bf16(rng.standard_normal((12, 8)))
    logits = rng.standard_normal((12, 8)).astype(np.float32)
    ref, _, _, ids, _ = mlp.PagedLayer(8, 8, 3, get).step(xb, logits)
    distinct = sorted(set(ids.reshape(-1).tolist()))
    for trial in range(20):
        perm = rng.permutation(distinct).tolist()
        cuts = sorted(rng.choice(np.arange(1, len(perm)), size=rng.integers(0, len(perm)), replace=False).tolist())
        waves = [perm[a:b] for a, b in zip([0] + cuts, cuts + [len(perm)])]
        out, *_ = mlp.PagedLayer(8, 8, 3, get).step(xb, logits, wave_order=waves)
        assert np.array_equal(out, ref)


def test_k_equals_e_no_page_ins_after_warmup():
    rng = np.random.default_rng(8)
    E, k = 10, 3
    sim = lru.ResidencySim(E, E)
    seen = set()
    for step in range(200):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(rng.integers(1, 5))])
        plan = sim.step(ids)
        new = set(ids.reshape(-1).tolist()) - seen
        assert plan.page_ins == len(new)
        assert len(plan.waves) <= 1
        seen |= new
    assert seen == set(range(E))


def test_lru_invariants_random():
    rng = np.random.default_rng(9)
    for E, K, k in ((16, 6, 2), (32, 5, 4), (12, 12, 3), (20, 1, 1)):
        sim = lru.ResidencySim(E, K)
        for step in range(300):
            T = int(rng.integers(1, 9))
            ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
            before = [sim.resident(e) for e in range(E)]
            plan = sim.step(ids)
            D = sorted(set(ids.reshape(-1).tolist()))
            M = [e for e in D if not before[e]]
            assert plan.page_ins == len(M)
            assert sum(w.hits for w in plan.waves) == len(D) - len(M)
            assert len(plan.waves) == -(-len(D) // K)
            for wv in plan.waves:
                assert len(wv.experts) <= K
                assert wv.plan_expert == sorted(wv.plan_expert)
            # every entry's slot held its expert when its wave ran
            assert plan.entry_slot.min() >= 0 and plan.entry_slot.max() < K
            sim.check_invariants()


def test_sizes_and_miss_bounds_match_pages():
    g = pins.golden("page_numbers.json")
    m = g["model"]
    fp8_b = sizing.expert_bytes(g["fp8_expert_mb"]["hidden"], g["fp8_expert_mb"]["intermediate"], "fp8")
    assert fp8_b == 3 * 2048 * 768 + 4 * (12 * 16 + 16 * 6)
    assert round(fp8_b / 1e6, 2) == g["fp8_expert_mb"]["value"]
    L, k = m["num_layers"], m["top_k"]
    assert round(sizing.all_miss_bytes_per_token(L, k, 4.72e6) / 1e9, 2) == g["all_miss_gb_per_token"]["fp8"]
    assert round(sizing.all_miss_bytes_per_token(L, k, 2.43e6) / 1e9, 2) == g["all_miss_gb_per_token"]["int4"]
    r = g["fp8_required_link_gbs"]
    assert round(1e3 / r["tok_s"], 1) == r["ms_per_token"]
    assert round(1.81e9 / (r["ms_per_token"] * 1e-3) / 1e9) == r["value"]
    b = g["max_miss_rate_fp8"]
    bound = sizing.max_miss_rate(b["link_gbs"] * 1e9, b["tok_s"], L, k, 4.72e6)
    assert round(100 * bound) == b["bound_pct"]
    assert round(100 * sizing.random_miss_rate(b["num_slots"], m["num_experts"])) == b["random_pct"]
    b = g["max_miss_rate_int4_63"]
    assert round(100 * sizing.max_miss_rate(b["link_gbs"] * 1e9, b["tok_s"], L, k, 2.43e6)) == b["bound_pct"]
    s = g["slot_mb"]
    assert round(sizing.slot_bytes(2.43e6, L) / 1e6) == s["int4_per_slot"]
    assert round(sizing.slot_bytes(4.72e6, L) / 1e6) == s["fp8_per_slot"]


def test_slots_for_budget_closed_forms():
    # floor of the budget left after the fixed bytes over the per-slot cost
    assert sizing.slots_for_budget(1000 + 40 * 117, 1000, 117, 128, 8) == 40
    assert sizing.slots_for_budget(1000 + 40 * 117 - 1, 1000, 117, 128, 8) == 39
    assert sizing.slots_for_budget(10**12, 1000, 117, 128, 8) == 128   # never above E
    assert sizing.slots_for_budget(1000 + 7 * 117, 1000, 117, 128, 8) == 0   # below top_k: no layer
    assert sizing.slots_for_budget(500, 1000, 117, 128, 8) == 0
    with pytest.raises(ValueError):
        sizing.slots_for_budget(1, 0, 0, 4, 1)


def test_slots_for_budget_pages_example():
    g = pins.golden("page_numbers.json")["choosing_k_example"]
    slot = g["per_slot_mb"] * 1e6
    # the page's K = 92 slots at 117 MB each is 10.76 GB, inside the 0.88 x 16 GB static budget
    table = g["num_slots"] * slot
    assert round(table / 1e9, 2) == 10.76
    assert table <= g["mem_fraction_static"] * g["gpu_gb"] * 1e9
    assert sizing.slots_for_budget(table, 0, slot, g["num_experts"], 8) == g["num_slots"]
    assert sizing.slots_for_budget(table - 1, 0, slot, g["num_experts"], 8) == g["num_slots"] - 1


def test_int4_hand_values():
    pins.check_int4_values(int4.dequant_rows)


def test_int4_brute_force():
    pins.check_int4_brute_force(int4.dequant_rows)


def test_int4_checkpoint_layout():
    pins.check_int4_gptq_layout(int4.dequant_gptq)


def test_int4_rejects_bad_grid():
    with pytest.raises(ValueError):
        int4.dequant_rows(np.zeros((2, 128), np.uint8), np.ones((2, 1), np.float16))


def test_int4_expert_size_is_the_pages_2_43_mb():
    g = pins.golden("page_numbers.json")
    b = sizing.expert_bytes(2048, 768, "int4")
    assert b == 3 * 2048 * 768 // 2 + 2 * (1536 * 16 + 2048 * 6) == 2_433_024
    assert round(b / 1e6, 2) == g["int4_expert_mb"]["value"]
    m = g["model"]
    assert round(sizing.slot_bytes(b, m["num_layers"]) / 1e6) == g["slot_mb"]["int4_per_slot"]


def test_gptq_checkpoint_repack_matches_the_oracle():
    """The loader's repack of a GPTQ checkpoint tensor dequantises, in the
    row layout, to the matrix the oracle reads from the checkpoint layout."""
    from host_paged_expert_gb300 import formats

    rng = np.random.default_rng(3)
    n, k = 48, 384
    qweight = rng.integers(0, 2**32, size=(k // 8, n), dtype=np.uint64).astype(np.uint32).view(np.int32)
    scales = (rng.random((k // 128, n)) * 0.01 + 1e-3).astype(np.float16)
    codes, srow = formats.gptq_int4_to_row(qweight, scales)
    assert codes.shape == (n, k // 2) and srow.shape == (n, k // 128)
    assert np.array_equal(int4.dequant_rows(codes, srow), int4.dequant_gptq(qweight, scales))
    w13, s13 = formats.gate_up_rows((codes, srow), (codes[::-1], srow[::-1]))
    assert w13.shape == (2 * n, k // 2) and np.array_equal(w13[n:], codes[::-1]) and np.array_equal(s13[:n], srow)


def test_e2m1_table_by_hand():
    from oracle import fp4

    pins.check_e2m1_table(fp4.decode_e2m1)
    # the same values from the bit fields, one code at a time
    assert [fp4.e2m1_value(c) for c in range(16)] == pins.E2M1_BY_HAND


def test_e8m0_table_matches_torch():
    from oracle import fp4

    pins.check_e8m0_table(fp4.decode_e8m0)


def test_fp4_hand_values():
    from oracle import fp4

    pins.check_fp4_hand_values(fp4.dequant_mx, fp4.dequant_nv)


def test_fp4_brute_force():
    from oracle import fp4

    pins.check_fp4_brute_force(fp4.dequant_mx, fp4.dequant_nv)


def test_fp4_rejects_bad_grid():
    from oracle import fp4

    with pytest.raises(ValueError):
        fp4.dequant_mx(np.zeros((2, 32), np.uint8), np.zeros((2, 1), np.uint8))  # K = 64 needs 2 blocks
    with pytest.raises(ValueError):
        fp4.dequant_nv(np.zeros((2, 16), np.uint8), np.zeros((2, 1), np.uint8), 1.0)  # K = 32 needs 2 blocks
