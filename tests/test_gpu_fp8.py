"""GPU parity for block-FP8 experts (E4M3 codes, fp32 scale per 128x128
block, bf16 activations): a small stack through decode and multi-wave
prefill, the tensor-core prefill with half-block tiles, the stale-scale
regression, and the full 48-layer FP8 stack (K=40, Zipf-skewed routing) at
decode batch 1 and 4 and one 512-token prefill chunk."""

import numpy as np
import pytest

import gpu_util as gu
from host_paged_expert_gb300 import synth
from oracle import lru as olru
from oracle import mlp as omlp
from oracle.routing import route

pytestmark = pytest.mark.gpu
TOL = gu.REL_L2["fp8"]


def _need():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from host_paged_expert_gb300 import _lib

    return _lib


SMALL = synth.MoEShape(1, 16, 2, 6, 256, 256, "fp8")


def test_fp8_small_decode_and_prefill():
    _lib = _need()
    s = SMALL
    w = synth.ExpertWeights(s, seed=3)
    a = _lib.PagedMoE(s, max_tokens=64)
    gu.load_stack(a, w)
    b = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=64, store_owner=a)
    o = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, gu.expert_fn(w, 0))
    dec = synth.decode_logits(1, s.num_experts, 16, seed=4, zipf_s=1.1)[0, :, 0, :]
    xs = synth.hidden_states((16,), s.hidden, seed=4)
    steps = [(xs[t : t + 1], dec[t : t + 1]) for t in range(16)]
    for T in (3, 4, 64):
        steps.append((synth.hidden_states((T,), s.hidden, seed=T, tag=9), synth.prefill_logits(1, 16, T, seed=T)[0]))
    for xb, lg in steps:
        T = xb.shape[0]
        x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
        ya, yb = a.forward(0, x, l), b.forward(0, x, l)
        out, _, plan, ids, wts = o.step(xb, lg)
        gu.check_plan(a.read_plan(0, T), plan, ids, wts)
        gu.check_residency(a.read_residency(0), o.sim)
        assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb)), T
        err = gu.max_token_rel_l2(gu.out_f64(ya), out)
        assert err <= TOL, (T, err)
    assert a.stats(0)["error_word"] == 0
    b.close()
    a.close()


def test_fp8_prefill_tensor_core():
    """FP8 prefill on the tensor cores: each 64-row gate (and up) tile is half
    of a 128-row scale block and each 64-wide K-step half of a scale column,
    so every scale is applied to two tiles; I = 384 gives an odd number of
    scale blocks per matrix.  T = 300 and 65 give ragged row tiles; the
    pipelined tensor-core step (not the GEMV kernels) must run."""
    _lib = _need()
    s = synth.MoEShape(1, 12, 2, 4, 512, 384, "fp8")
    w = synth.ExpertWeights(s, seed=7)
    a = _lib.PagedMoE(s, max_tokens=300)
    gu.load_stack(a, w)
    b = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=300, store_owner=a)
    a.profile_enable(True)
    o = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, gu.expert_fn(w, 0))
    for T in (300, 65):
        xb = synth.hidden_states((T,), s.hidden, seed=T, tag=11)
        lg = synth.prefill_logits(1, s.num_experts, T, seed=T)[0]
        x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
        ya, yb = a.forward(0, x, l), b.forward(0, x, l)
        out, _, plan, ids, wts = o.step(xb, lg)
        assert len(plan.waves) >= 2
        gu.check_plan(a.read_plan(0, T), plan, ids, wts)
        assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb)), T
        err = gu.max_token_rel_l2(gu.out_f64(ya), out)
        assert err <= TOL, (T, err)
    prof = a.profile_read()
    assert prof["prefill_step"]["launches"] == 2
    assert prof["gateup"]["launches"] == 0
    assert a.stats(0)["error_word"] == 0
    b.close()
    a.close()


def test_fp8_scales_are_paged_with_codes():
    """Rescale one block of one expert's s13 and s2 in its host row: after the
    expert is paged in again the output follows the new scales (a slot never
    keeps another expert's or a stale scale grid)."""
    _lib = _need()
    s = synth.MoEShape(1, 8, 2, 2, 256, 256, "fp8")
    w = synth.ExpertWeights(s, seed=5)
    m = _lib.PagedMoE(s, max_tokens=2)
    gu.load_stack(m, w)
    xb = synth.hidden_states((1,), s.hidden, seed=6)
    lg = np.full((1, 8), -3.0, np.float32)
    lg[0, 1], lg[0, 5] = 1.0, 0.8
    x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
    y0 = gu.out_bits(m.forward(0, x, l))
    row = {k: v.copy() for k, v in w.row(0, 5).items()}
    row["s13"][0, 1] *= 4.0
    row["s2"][1, 0] *= 0.25
    m.load_expert(0, 5, row)
    for other in ([0, 2], [3, 4]):
        lo = np.full((1, 8), -3.0, np.float32)
        lo[0, other] = [1.0, 0.9]
        m.forward(0, x, gu.to_dev_f32(lo))
    y1 = gu.out_bits(m.forward(0, x, l))
    assert not np.array_equal(y0, y1)
    ref = omlp.unpaged_layer(xb, lg, 2, lambda e: omlp.expert_weights(row if e == 5 else w.row(0, e), "fp8"))
    assert gu.max_token_rel_l2(synth.bf16_bits_to_f32(y1).astype(np.float64), ref) <= TOL
    m.close()


@pytest.fixture(scope="module")
def fp8_stack48():
    _lib = _need()
    s = synth.STACK48_FP8
    w = synth.ExpertWeights(s, seed=0)
    owner = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=512)
    gu.load_stack(owner, w)
    yield s, w, owner
    owner.close()


@pytest.mark.parametrize("B", [1, 4])
def test_fp8_stack48_decode(fp8_stack48, B):
    from host_paged_expert_gb300 import _lib
    import torch

    s, w, owner = fp8_stack48
    L, E, k, K = s.num_layers, s.num_experts, s.top_k, s.num_slots
    S = 16
    lg = synth.decode_logits(L, E, S, batch=B, seed=0, zipf_s=1.1).transpose(1, 0, 2, 3)
    hs = synth.hidden_states((S, L, B), s.hidden, seed=0)
    model = _lib.PagedMoE(s, max_tokens=B, store_owner=owner)
    owner.reset_residency()
    sims = [olru.ResidencySim(E, K) for _ in range(L)]
    for t in range(S):
        for l in range(L):
            x, lgt = gu.to_dev_bf16(hs[t, l]), gu.to_dev_f32(lg[t, l])
            ya = model.forward(l, x, lgt)
            yb = owner.forward(l, x, lgt)
            ids, wts, _ = route(lg[t, l], k)
            gu.check_plan(model.read_plan(l, B), sims[l].step(ids), ids, wts)
            assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb)), (t, l)
            if t == S // 2 or (t, l) in ((0, 0), (S - 1, L - 1)):  # every layer of one token, per token
                want = omlp.unpaged_layer(hs[t, l], lg[t, l], k, gu.expert_fn(w, l))
                gu.check_tokens(gu.out_f64(ya), want, TOL, (B, t, l))
    torch.cuda.synchronize()
    assert model.stats(-1)["error_word"] == 0
    model.close()


def test_fp8_stack48_prefill(fp8_stack48):
    """One 512-token chunk through all 48 FP8 layers at K=40 on the
    tensor-core path: plans bit-exact, paged == K=E bit for bit, every token
    of four layers within the FP8 tolerance of the plain MoE layer."""
    from host_paged_expert_gb300 import _lib

    s, w, owner = fp8_stack48
    L, E, k, K, T = s.num_layers, s.num_experts, s.top_k, s.num_slots, 512
    lg = synth.prefill_logits(L, E, T, seed=1)
    hs = synth.hidden_states((L, T), s.hidden, seed=1, tag=5)
    model = _lib.PagedMoE(s, max_tokens=T, store_owner=owner)
    owner.reset_residency()
    model.profile_enable(True)
    sims = [olru.ResidencySim(E, K) for _ in range(L)]
    for l in range(L):
        x, lgt = gu.to_dev_bf16(hs[l]), gu.to_dev_f32(lg[l])
        ya = model.forward(l, x, lgt)
        yb = owner.forward(l, x, lgt)
        ids, wts, _ = route(lg[l], k)
        gu.check_plan(model.read_plan(l, T), sims[l].step(ids), ids, wts)
        assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb)), l
        if l in (0, 1, L // 2, L - 1):  # every token of four layers
            want = omlp.unpaged_layer(hs[l], lg[l], k, gu.expert_fn(w, l))
            gu.check_tokens(gu.out_f64(ya), want, TOL, (T, l))
    prof = model.profile_read()
    assert prof["prefill_step"]["launches"] == L
    assert model.stats(-1)["error_word"] == 0
    model.close()
