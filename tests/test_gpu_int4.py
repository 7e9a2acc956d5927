"""GPU parity for GPTQ int4 experts (4-bit codes, zero point 8, one fp16 scale
per output row and 128 inputs; bf16 activations): a small stack through the
one-kernel decode step, multi-wave decode and the tensor-core prefill; scales
paged with their codes; and the full 48-layer int4 stack at the pages' K = 92
of 128 (decode batch 1 and 4, one 512-token prefill chunk)."""

import numpy as np
import pytest

import gpu_util as gu
from host_paged_expert_gb300 import synth
from oracle import lru as olru
from oracle import mlp as omlp
from oracle.routing import route

pytestmark = pytest.mark.gpu
TOL = gu.REL_L2["int4"]


def _need():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from host_paged_expert_gb300 import _lib

    return _lib


SMALL = synth.MoEShape(1, 16, 2, 6, 256, 256, "int4")


def test_int4_small_every_path():
    """Decode (T = 1, one kernel), multi-wave decode (T = 4: 8 entries over
    6 slots, GEMV kernels) and prefill (T = 64 and 65: tensor-core step), each
    against the oracle and bit for bit against K = E."""
    _lib = _need()
    s = SMALL
    w = synth.ExpertWeights(s, seed=3)
    a = _lib.PagedMoE(s, max_tokens=65)
    gu.load_stack(a, w)
    b = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=65, store_owner=a)
    o = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, gu.expert_fn(w, 0))
    dec = synth.decode_logits(1, s.num_experts, 16, seed=4, zipf_s=1.1)[0, :, 0, :]
    xs = synth.hidden_states((16,), s.hidden, seed=4)
    steps = [(xs[t : t + 1], dec[t : t + 1]) for t in range(16)]
    for T in (3, 4, 64, 65):
        steps.append((synth.hidden_states((T,), s.hidden, seed=T, tag=9), synth.prefill_logits(1, 16, T, seed=T)[0]))
    a.profile_enable(True)
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
    prof = a.profile_read()
    assert prof["decode_step"]["launches"] >= 16
    assert prof["gateup_pagein"]["launches"] >= 2 and prof["prefill_step"]["launches"] == 2
    assert a.stats(0)["error_word"] == 0
    b.close()
    a.close()


def test_int4_scales_are_paged_with_codes():
    """Rescale one group of one expert's s13 and s2 rows in its host row:
    after the expert is paged in again the output follows the new scales."""
    _lib = _need()
    s = synth.MoEShape(1, 8, 2, 2, 256, 256, "int4")
    w = synth.ExpertWeights(s, seed=5)
    m = _lib.PagedMoE(s, max_tokens=2)
    gu.load_stack(m, w)
    xb = synth.hidden_states((1,), s.hidden, seed=6)
    lg = np.full((1, 8), -3.0, np.float32)
    lg[0, 1], lg[0, 5] = 1.0, 0.8
    x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
    y0 = gu.out_bits(m.forward(0, x, l))
    row = {k: v.copy() for k, v in w.row(0, 5).items()}
    row["s13"][3, 1] *= np.float16(4.0)
    row["s2"][7, 0] *= np.float16(0.25)
    m.load_expert(0, 5, row)
    for other in ([0, 2], [3, 4]):
        lo = np.full((1, 8), -3.0, np.float32)
        lo[0, other] = [1.0, 0.9]
        m.forward(0, x, gu.to_dev_f32(lo))
    y1 = gu.out_bits(m.forward(0, x, l))
    assert not np.array_equal(y0, y1)
    ref = omlp.unpaged_layer(xb, lg, 2, lambda e: omlp.expert_weights(row if e == 5 else w.row(0, e), "int4"))
    assert gu.max_token_rel_l2(synth.bf16_bits_to_f32(y1).astype(np.float64), ref) <= TOL
    m.close()


@pytest.fixture(scope="module")
def int4_stack48():
    _lib = _need()
    s = synth.STACK48_INT4
    w = synth.ExpertWeights(s, seed=0)
    owner = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=512)
    gu.load_stack(owner, w)
    yield s, w, owner
    owner.close()


@pytest.mark.parametrize("B", [1, 4])
def test_int4_stack48_decode(int4_stack48, B):
    from host_paged_expert_gb300 import _lib
    import torch

    s, w, owner = int4_stack48
    L, E, k, K = s.num_layers, s.num_experts, s.top_k, s.num_slots
    S = 16
    lg = synth.decode_logits(L, E, S, batch=B, seed=0).transpose(1, 0, 2, 3)
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


def test_int4_stack48_prefill(int4_stack48):
    from host_paged_expert_gb300 import _lib

    s, w, owner = int4_stack48
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
    assert model.profile_read()["prefill_step"]["launches"] == L
    assert model.stats(-1)["error_word"] == 0
    model.close()
