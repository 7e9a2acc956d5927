"""GPU parity on the tiny workload (1 layer, H=256, I=128, E=16, top-2, K=6):
32 batch-1 decode steps and one 64-token prefill chunk, through the C ABI,
against the CPU oracle and against the same call with K = E."""

import numpy as np
import pytest

import gpu_util as gu
from host_paged_expert_gb300 import synth
from oracle import mlp as omlp

pytestmark = pytest.mark.gpu


def _need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from host_paged_expert_gb300 import _lib

    return _lib


@pytest.fixture(scope="module")
def tiny():
    _lib = _need_gpu()
    s = synth.TINY
    w = synth.ExpertWeights(s, seed=0)
    paged = _lib.PagedMoE(s, max_tokens=64)
    gu.load_stack(paged, w)
    unpaged = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=64, store_owner=paged)
    yield s, w, paged, unpaged
    unpaged.close()
    paged.close()


def _steps(s):
    dec = synth.decode_logits(1, s.num_experts, 32, seed=0)[0, :, 0, :]          # [32, E]
    xs = synth.hidden_states((33,), s.hidden, seed=0)                              # one per step
    pre = synth.prefill_logits(1, s.num_experts, 64, seed=0)[0]                     # [64, E]
    xp = synth.hidden_states((64,), s.hidden, seed=0, tag=3)
    steps = [(xs[t : t + 1], dec[t : t + 1]) for t in range(32)]
    steps.append((xp, pre))
    return steps


def test_tiny_decode_then_prefill(tiny):
    s, w, paged, unpaged = tiny
    get = gu.expert_fn(w, 0)
    o_paged = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, get)
    o_unpaged = omlp.PagedLayer(s.num_experts, s.num_experts, s.top_k, get)
    waves_seen = set()
    for step, (xb, lg) in enumerate(_steps(s)):
        T = xb.shape[0]
        x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
        y = paged.forward(0, x, l)
        y_ref = unpaged.forward(0, x, l)
        out, merged, plan, ids, wts = o_paged.step(xb, lg)
        _, _, plan_u, _, _ = o_unpaged.step(xb, lg)
        waves_seen.add(len(plan.waves))
        gu.check_plan(paged.read_plan(0, T), plan, ids, wts)
        gu.check_plan(unpaged.read_plan(0, T), plan_u, ids, wts)
        gu.check_residency(paged.read_residency(0), o_paged.sim)
        gu.check_residency(unpaged.read_residency(0), o_unpaged.sim)
        assert np.array_equal(gu.out_bits(y), gu.out_bits(y_ref)), f"paged != unpaged at step {step}"
        err = gu.max_token_rel_l2(gu.out_f64(y), out)
        assert err <= gu.REL_L2["bf16"], (step, err)
        # every resident slot holds its expert's host row byte for byte
        res = paged.read_residency(0)
        for slot, e in enumerate(res["slot_expert"].tolist()):
            if e >= 0:
                got = paged.read_slot(0, slot, paged.layout["payload_bytes"])
                want = paged.host_row(0, e)[: paged.layout["payload_bytes"]]
                assert np.array_equal(got, want), (step, slot, e)
    assert 1 in waves_seen and max(waves_seen) >= 2  # decode is one wave; the prefill needs more
    st = paged.stats(0)
    assert st["steps"] == 33 and st["error_word"] == 0
    assert st["bytes_paged"] == st["page_ins"] * paged.layout["payload_bytes"]


def test_tiny_stats_match_oracle_counts(tiny):
    s, w, paged, _ = tiny
    _lib = _need_gpu()
    m = _lib.PagedMoE(s, max_tokens=64, store_owner=paged)
    sim = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, gu.expert_fn(w, 0))
    hits = pins = distinct = waves = 0
    for xb, lg in _steps(s):
        m.forward(0, gu.to_dev_bf16(xb), gu.to_dev_f32(lg))
        plan = sim.sim.step(sim_route(lg, s.top_k))
        hits += plan.hits
        pins += plan.page_ins
        distinct += len(plan.distinct)
        waves += len(plan.waves)
    st = m.stats(0)
    assert (st["hits"], st["page_ins"], st["distinct"], st["waves"]) == (hits, pins, distinct, waves)
    assert st["cold_fills"] == s.num_slots
    m.close()


def sim_route(lg, k):
    from oracle.routing import route

    return route(lg, k)[0]


@pytest.mark.parametrize("T", [1, 2, 3, 4, 7, 64])
def test_multi_token_shapes(tiny, T):
    """T*top_k <= K is one fused wave; above that the wave loop and the
    separate top-k sum run.  Both equal the K = E result bit for bit."""
    s, w, paged, _ = tiny
    _lib = _need_gpu()
    a = _lib.PagedMoE(s, max_tokens=64, store_owner=paged)
    b = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=64, store_owner=paged)
    get = gu.expert_fn(w, 0)
    o = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, get)
    for rep in range(3):
        xb = synth.hidden_states((T,), s.hidden, seed=1, tag=10 + rep)
        lg = synth.prefill_logits(1, s.num_experts, T, seed=rep + 5)[0]
        x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
        ya, yb = a.forward(0, x, l), b.forward(0, x, l)
        out, _, plan, ids, wts = o.step(xb, lg)
        gu.check_plan(a.read_plan(0, T), plan, ids, wts)
        assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb))
        assert gu.max_token_rel_l2(gu.out_f64(ya), out) <= gu.REL_L2["bf16"]
    a.close()
    b.close()


def test_zero_tokens_and_range_errors(tiny):
    s, w, paged, _ = tiny
    _lib = _need_gpu()
    import torch

    x = torch.zeros((65, s.hidden), dtype=torch.bfloat16, device="cuda")
    l = torch.zeros((65, s.num_experts), dtype=torch.float32, device="cuda")
    before = paged.stats(0)["steps"]
    paged.forward(0, x[:0], l[:0])  # no-op
    assert paged.stats(0)["steps"] == before
    with pytest.raises(_lib.PEError) as ei:
        paged.forward(0, x, l)
    assert ei.value.status == _lib.PE_ERR_RANGE
    with pytest.raises(_lib.PEError) as ei:
        paged.forward(1, x[:1], l[:1])
    assert ei.value.status == _lib.PE_ERR_RANGE


def test_device_error_word(tiny):
    """NaN logits and experts that were never loaded set error bits (the
    call itself stays asynchronous and succeeds)."""
    s, w, paged, _ = tiny
    _lib = _need_gpu()
    fresh = _lib.PagedMoE(s, max_tokens=4)
    for e in range(s.num_experts):
        if e != 3:
            fresh.load_expert(0, e, w.row(0, e))
    lg = np.full((1, s.num_experts), -5.0, np.float32)
    lg[0, 5] = 1.0
    lg[0, 7] = np.nan
    lg[0, 9] = 0.5
    xb = synth.hidden_states((1,), s.hidden, seed=2)
    fresh.forward(0, gu.to_dev_bf16(xb), gu.to_dev_f32(lg))
    st = fresh.stats(0)
    assert st["error_word"] & _lib.PE_DEVERR_NAN_LOGIT
    assert not st["error_word"] & _lib.PE_DEVERR_NOT_LOADED
    assert fresh.read_plan(0, 1)["topk_id"].tolist() == [[5, 9]]
    lg2 = np.full((1, s.num_experts), -5.0, np.float32)
    lg2[0, 3] = 2.0
    fresh.forward(0, gu.to_dev_bf16(xb), gu.to_dev_f32(lg2))
    assert fresh.stats(0)["error_word"] & _lib.PE_DEVERR_NOT_LOADED
    fresh.close()


def test_scale_rows_are_paged_with_weights():
    """Changing one expert's host row changes the output after it is paged
    in again: a slot never keeps a stale piece of another expert's row."""
    _lib = _need_gpu()
    s = synth.MoEShape(1, 8, 2, 2, 256, 128, "bf16")
    w = synth.ExpertWeights(s, seed=4)
    m = _lib.PagedMoE(s, max_tokens=2)
    gu.load_stack(m, w)
    xb = synth.hidden_states((1,), s.hidden, seed=3)
    lg = np.full((1, 8), -3.0, np.float32)
    lg[0, 2], lg[0, 6] = 1.0, 0.9
    x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
    y0 = gu.out_bits(m.forward(0, x, l))
    row = w.row(0, 6)
    w2 = row["w2"].copy()
    w2[:, :] = synth.f32_to_bf16_bits(np.float32(0.5) * synth.bf16_bits_to_f32(w2))
    m.load_expert(0, 6, {"w13": row["w13"], "w2": w2})
    # evict 2 and 6 by routing elsewhere, then route back: the new row is paged in
    for other in ([0, 1], [3, 4]):
        lo = np.full((1, 8), -3.0, np.float32)
        lo[0, other] = [1.0, 0.9]
        m.forward(0, x, gu.to_dev_f32(lo))
    y1 = gu.out_bits(m.forward(0, x, l))
    assert not np.array_equal(y0, y1)
    ref = omlp.unpaged_layer(xb, lg, 2, lambda e: omlp.expert_weights(
        {"w13": row["w13"], "w2": w2} if e == 6 else w.row(0, e), "bf16"))
    got = synth.bf16_bits_to_f32(y1).astype(np.float64)
    assert gu.max_token_rel_l2(got, ref) <= 1e-2
    m.close()


def test_graph_captured_decode_matches_eager(tiny):
    """A captured decode step replays the device planner and page-in: each
    replay moves exactly the experts it plans, like the eager call."""
    s, w, paged, _ = tiny
    _lib = _need_gpu()
    import torch

    eager = _lib.PagedMoE(s, max_tokens=4, store_owner=paged)
    graphed = _lib.PagedMoE(s, max_tokens=4, store_owner=paged)
    xs = synth.hidden_states((40,), s.hidden, seed=7)
    lg = synth.decode_logits(1, s.num_experts, 40, seed=9)[0, :, 0, :]
    x_st = torch.zeros((1, s.hidden), dtype=torch.bfloat16, device="cuda")
    l_st = torch.zeros((1, s.num_experts), dtype=torch.float32, device="cuda")
    y_st = torch.zeros((1, s.hidden), dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=side):
        graphed.forward(0, x_st, l_st, y_st)
    for t in range(40):
        x, l = gu.to_dev_bf16(xs[t : t + 1]), gu.to_dev_f32(lg[t : t + 1])
        x_st.copy_(x)
        l_st.copy_(l)
        g.replay()
        ye = eager.forward(0, x, l)
        torch.cuda.synchronize()
        assert np.array_equal(gu.out_bits(y_st), gu.out_bits(ye)), t
        pg, pe_ = graphed.read_plan(0, 1), eager.read_plan(0, 1)
        for k in ("plan_expert", "plan_slot", "plan_count", "entry_slot"):
            if k == "plan_expert" or k == "plan_slot":
                c = int(pe_["plan_count"][0])
                assert np.array_equal(pg[k][0, :c], pe_[k][0, :c])
            else:
                assert np.array_equal(pg[k], pe_[k])
    assert graphed.stats(0)["page_ins"] == eager.stats(0)["page_ins"]
    eager.close()
    graphed.close()


def test_graph_captured_prefill_matches_eager(tiny):
    """A captured multi-wave prefill step (planner, align, gather, the
    pipelined page-in + GEMM step, top-k sum) replays with new chunks: every
    grid comes from shapes and every count is read on the device, so each
    replay plans, pages and computes like the eager call, bit for bit."""
    s, w, paged, _ = tiny
    _lib = _need_gpu()
    import torch

    T = 64
    eager = _lib.PagedMoE(s, max_tokens=T, store_owner=paged)
    graphed = _lib.PagedMoE(s, max_tokens=T, store_owner=paged)
    o = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, gu.expert_fn(w, 0))
    x_st = torch.zeros((T, s.hidden), dtype=torch.bfloat16, device="cuda")
    l_st = torch.zeros((T, s.num_experts), dtype=torch.float32, device="cuda")
    y_st = torch.zeros((T, s.hidden), dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=side):
        graphed.forward(0, x_st, l_st, y_st)
    for c in range(5):
        xb = synth.hidden_states((T,), s.hidden, seed=c, tag=41)
        lb = synth.prefill_logits(1, s.num_experts, T, seed=40 + c)[0]
        x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lb)
        x_st.copy_(x)
        l_st.copy_(l)
        g.replay()
        ye = eager.forward(0, x, l)
        torch.cuda.synchronize()
        assert np.array_equal(gu.out_bits(y_st), gu.out_bits(ye)), c
        out, _, plan, ids, wts = o.step(xb, lb)
        assert len(plan.waves) >= 2
        gu.check_plan(graphed.read_plan(0, T), plan, ids, wts)
        assert gu.max_token_rel_l2(gu.out_f64(ye), out) <= gu.REL_L2["bf16"], c
    assert graphed.stats(0)["page_ins"] == eager.stats(0)["page_ins"]
    assert graphed.stats(0)["error_word"] == 0
    eager.close()
    graphed.close()


@pytest.mark.parametrize("E,k,K", [(1, 1, 1), (8, 1, 3), (8, 2, 5), (9, 3, 7), (16, 2, 16)])
def test_odd_slot_and_entry_counts(E, k, K):
    """Slot and entry counts that make the fused kernel's shared-memory
    metadata block an odd number of ints; outputs still match the oracle and
    the K = E call."""
    _lib = _need_gpu()
    s = synth.MoEShape(1, E, k, K, 256, 128, "bf16")
    w = synth.ExpertWeights(s, seed=E + 10 * K)
    a = _lib.PagedMoE(s, max_tokens=7)
    gu.load_stack(a, w)
    b = _lib.PagedMoE(s.with_slots(E), max_tokens=7, store_owner=a)
    o = omlp.PagedLayer(E, K, k, gu.expert_fn(w, 0))
    for T in (1, 3, 5, 7):
        xb = synth.hidden_states((T,), s.hidden, seed=T, tag=E)
        lg = synth.prefill_logits(1, E, T, seed=T + K)[0]
        x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
        ya, yb = a.forward(0, x, l), b.forward(0, x, l)
        out, _, plan, ids, wts = o.step(xb, lg)
        gu.check_plan(a.read_plan(0, T), plan, ids, wts)
        assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb))
        assert gu.max_token_rel_l2(gu.out_f64(ya), out) <= gu.REL_L2["bf16"]
    b.close()
    a.close()


def test_prefill_runs_on_the_tensor_core_path(tiny):
    """A 64-token chunk (128 entries) takes the pipelined prefill step (one
    launch for all waves' page-ins and tcgen05 GEMMs); a decode step whose
    entries fit the slots takes the one-kernel decode path."""
    s, w, paged, _ = tiny
    _lib = _need_gpu()
    m = _lib.PagedMoE(s, max_tokens=64, store_owner=paged)
    m.profile_enable(True)
    xb = synth.hidden_states((64,), s.hidden, seed=31)
    lg = synth.prefill_logits(1, s.num_experts, 64, seed=31)[0]
    m.forward(0, gu.to_dev_bf16(xb), gu.to_dev_f32(lg))
    prof = m.profile_read()
    assert prof["prefill_step"]["launches"] == 1 and prof["prefill_align"]["launches"] == 1
    assert prof["pagein"]["launches"] == 0 and prof["gateup_pagein"]["launches"] == 0
    m.profile_enable(True)
    m.forward(0, gu.to_dev_bf16(xb[:1]), gu.to_dev_f32(lg[:1]))
    prof = m.profile_read()
    assert prof["decode_step"]["launches"] == 1 and prof["prefill_step"]["launches"] == 0
    assert prof["gateup_pagein"]["launches"] == 0 and prof["down"]["launches"] == 0
    m.close()


def test_prefill_fallback_path_for_untiled_shapes():
    """A prefill-sized step (T*top_k > 64) whose shapes do not tile for the
    tensor cores (H = 136 is not a multiple of 128, I = 72 not of 64) runs the
    plain path: per wave a page-in kernel, the weight-streaming gate/up and
    down kernels, then the top-k sum.  Plans bit-exact against the oracle,
    paged equal to K = E bit for bit, every token within 1e-2 of the oracle,
    over consecutive chunks so later waves evict earlier ones."""
    _lib = _need_gpu()
    s = synth.MoEShape(1, 16, 2, 5, 136, 72, "bf16")
    w = synth.ExpertWeights(s, seed=41)
    T = 48
    a = _lib.PagedMoE(s, max_tokens=T)
    gu.load_stack(a, w)
    b = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=T, store_owner=a)
    o = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, gu.expert_fn(w, 0))
    a.profile_enable(True)
    waves = []
    for c in range(3):
        xb = synth.hidden_states((T,), s.hidden, seed=42, tag=c)
        lg = synth.prefill_logits(1, s.num_experts, T, seed=43 + c)[0]
        x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
        ya, yb = a.forward(0, x, l), b.forward(0, x, l)
        out, _, plan, ids, wts = o.step(xb, lg)
        waves.append(len(plan.waves))
        gu.check_plan(a.read_plan(0, T), plan, ids, wts)
        gu.check_residency(a.read_residency(0), o.sim)
        assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb)), c
        gu.check_tokens(gu.out_f64(ya), out, gu.REL_L2["bf16"], ("fallback", c))
        res = a.read_residency(0)
        for slot, e in enumerate(res["slot_expert"].tolist()):
            if e >= 0:
                got = a.read_slot(0, slot, a.layout["payload_bytes"])
                assert np.array_equal(got, a.host_row(0, e)[: a.layout["payload_bytes"]]), (c, slot, e)
    prof = a.profile_read()
    assert min(waves) >= 3
    assert prof["prefill_step"]["launches"] == 0 and prof["decode_step"]["launches"] == 0
    assert prof["pagein"]["launches"] >= 3 * min(waves) and prof["gateup"]["launches"] == prof["pagein"]["launches"]
    assert prof["topk_sum"]["launches"] == 3
    assert a.stats(0)["error_word"] == 0
    b.close()
    a.close()


def test_prefill_tiles_over_128_rows():
    """Experts with more than 128 routed rows fill both 128-row halves of a
    tensor-core tile (and, past 256 rows, several tiles); results match the
    oracle and the K = E call bit for bit."""
    _lib = _need_gpu()
    s = synth.MoEShape(1, 4, 2, 2, 256, 128, "bf16")
    w = synth.ExpertWeights(s, seed=13)
    a = _lib.PagedMoE(s, max_tokens=320)
    gu.load_stack(a, w)
    b = _lib.PagedMoE(s.with_slots(4), max_tokens=320, store_owner=a)
    o = omlp.PagedLayer(4, 2, 2, gu.expert_fn(w, 0))
    for T in (70, 200, 320):
        xb = synth.hidden_states((T,), s.hidden, seed=T, tag=21)
        lg = synth.prefill_logits(1, 4, T, seed=T)[0]
        x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
        a.profile_enable(True)
        ya, yb = a.forward(0, x, l), b.forward(0, x, l)
        assert a.profile_read()["prefill_step"]["launches"] == 1
        out, _, plan, ids, wts = o.step(xb, lg)
        gu.check_plan(a.read_plan(0, T), plan, ids, wts)
        assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb)), T
        assert gu.max_token_rel_l2(gu.out_f64(ya), out) <= gu.REL_L2["bf16"], T
    b.close()
    a.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "int4"])
def test_consecutive_multiwave_prefills_keep_slots_exact(dtype):
    """Prefill steps of three waves in a row (K = 6 of 16 experts): a later
    wave's page-ins go through the staging rows while their slots are still in
    use (the second wave's fill them, the third wave's wait), and the slots'
    last occupants are copied in from there.  Every step equals K = E bit for
    bit, plans and residency equal the oracle's, and every resident slot
    holds its expert's host row byte for byte."""
    _lib = _need_gpu()
    s = synth.MoEShape(1, 16, 2, 6, 256, 256, dtype)
    w = synth.ExpertWeights(s, seed=3)
    a = _lib.PagedMoE(s, max_tokens=65)
    gu.load_stack(a, w)
    b = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=65, store_owner=a)
    o = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, gu.expert_fn(w, 0))
    waves = []
    for i, T in enumerate((64, 65, 64, 48)):
        xb = synth.hidden_states((T,), s.hidden, seed=T, tag=9 + i)
        lg = synth.prefill_logits(1, s.num_experts, T, seed=T + i)[0]
        x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
        ya, yb = a.forward(0, x, l), b.forward(0, x, l)
        out, _, plan, ids, wts = o.step(xb, lg)
        waves.append(len(plan.waves))
        gu.check_plan(a.read_plan(0, T), plan, ids, wts)
        gu.check_residency(a.read_residency(0), o.sim)
        assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb)), (dtype, i)
        assert gu.max_token_rel_l2(gu.out_f64(ya), out) <= gu.REL_L2[dtype], (dtype, i)
        for slot, e in enumerate(a.read_residency(0)["slot_expert"].tolist()):
            if e >= 0:
                got = a.read_slot(0, slot, a.layout["payload_bytes"])
                want = a.host_row(0, e)[: a.layout["payload_bytes"]]
                assert np.array_equal(got, want), (dtype, i, slot, e)
    assert max(waves) >= 3, waves
    assert a.stats(0)["error_word"] == 0
    a.close()
    b.close()
