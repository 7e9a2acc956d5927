"""GPU parity for MXFP4 and NVFP4 experts (E2M1 codes; E8M0 scales per 32
inputs, or E4M3 scales per 16 inputs and an fp32 tensor scale; bf16
activations): a small stack through the one-kernel decode step, multi-wave
decode and the tensor-core prefill; every scale (the NVFP4 tensor scale
included) paged with its codes; the padded-width case (I = 2880, which the
kernels run as 2944) as a regression test of the padding lesson; and the full
48-layer stacks at K = 92 of 128."""

import numpy as np
import pytest

import gpu_util as gu
from host_paged_expert_gb300 import synth
from oracle import lru as olru
from oracle import mlp as omlp
from oracle.routing import route

pytestmark = pytest.mark.gpu
TOL = gu.REL_L2["fp4"]
FORMATS = ["mxfp4", "nvfp4"]


def _need():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from host_paged_expert_gb300 import _lib

    return _lib


def _run_steps(_lib, s, w, steps, max_tokens):
    a = _lib.PagedMoE(s, max_tokens=max_tokens)
    gu.load_stack(a, w)
    b = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=max_tokens, store_owner=a)
    o = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, gu.expert_fn(w, 0))
    a.profile_enable(True)
    for xb, lg in steps:
        T = xb.shape[0]
        x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
        ya, yb = a.forward(0, x, l), b.forward(0, x, l)
        out, _, plan, ids, wts = o.step(xb, lg)
        gu.check_plan(a.read_plan(0, T), plan, ids, wts)
        gu.check_residency(a.read_residency(0), o.sim)
        assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb)), T
        gu.check_tokens(gu.out_f64(ya), out, TOL, (s.dtype, T))
        # every resident slot holds its expert's host row, padding included
        res = a.read_residency(0)
        for slot, e in enumerate(res["slot_expert"].tolist()):
            if e >= 0:
                got = a.read_slot(0, slot, a.layout["payload_bytes"])
                assert np.array_equal(got, a.host_row(0, e)[: a.layout["payload_bytes"]]), (T, slot, e)
    prof = a.profile_read()
    assert a.stats(0)["error_word"] == 0
    return a, b, prof


@pytest.mark.parametrize("dtype", FORMATS)
def test_fp4_small_every_path(dtype):
    """Decode (T = 1, one kernel), multi-wave decode (T = 3, 4: more entries
    than the 6 slots, GEMV kernels) and prefill (T = 64 and 65: tensor-core
    step), each against the oracle and bit for bit against K = E."""
    _lib = _need()
    s = synth.MoEShape(1, 16, 2, 6, 256, 256, dtype)
    w = synth.ExpertWeights(s, seed=13)
    dec = synth.decode_logits(1, s.num_experts, 16, seed=4, zipf_s=1.1)[0, :, 0, :]
    xs = synth.hidden_states((16,), s.hidden, seed=4)
    steps = [(xs[t : t + 1], dec[t : t + 1]) for t in range(16)]
    for T in (3, 4, 64, 65):
        steps.append((synth.hidden_states((T,), s.hidden, seed=T, tag=9), synth.prefill_logits(1, 16, T, seed=T)[0]))
    a, b, prof = _run_steps(_lib, s, w, steps, 65)
    assert prof["decode_step"]["launches"] >= 16
    assert prof["gateup_pagein"]["launches"] >= 2 and prof["prefill_step"]["launches"] == 2
    b.close()
    a.close()


def test_mxfp4_padded_width_regression():
    """I = 2880 is not a multiple of 128: the row layout carries it padded to
    2944 (zero codes and scales), the loader writes the logical tensors into
    that padded row, and the host row, the slot and the kernels all use the
    same padded layout.  Decode, multi-wave decode and prefill all match the
    oracle on the unpadded expert and K = E bit for bit."""
    _lib = _need()
    s = synth.MoEShape(1, 8, 2, 3, 256, 2880, "mxfp4")
    Ip = 2944
    w = synth.ExpertWeights(s, seed=17)
    m = _lib.PagedMoE(s, max_tokens=40)
    lay = m.layout
    assert lay["w13_bytes"] == 2 * Ip * s.hidden // 2 and lay["w2_bytes"] == s.hidden * Ip // 2
    assert lay["s13_bytes"] == 2 * Ip * s.hidden // 32 and lay["s2_bytes"] == s.hidden * Ip // 32
    gu.load_stack(m, w)
    row = m.host_row(0, 5)
    w13p = row[lay["w13_offset"] : lay["w13_offset"] + lay["w13_bytes"]].reshape(2 * Ip, s.hidden // 2)
    w2p = row[lay["w2_offset"] : lay["w2_offset"] + lay["w2_bytes"]].reshape(s.hidden, Ip // 2)
    src = w.row(0, 5)
    assert np.array_equal(w13p[: s.intermediate], src["w13"][: s.intermediate])
    assert np.array_equal(w13p[Ip : Ip + s.intermediate], src["w13"][s.intermediate :])
    assert not w13p[s.intermediate : Ip].any() and not w13p[Ip + s.intermediate :].any()
    assert np.array_equal(w2p[:, : s.intermediate // 2], src["w2"]) and not w2p[:, s.intermediate // 2 :].any()
    m.close()
    dec = synth.decode_logits(1, s.num_experts, 6, seed=18)[0, :, 0, :]
    xs = synth.hidden_states((6,), s.hidden, seed=18)
    steps = [(xs[t : t + 1], dec[t : t + 1]) for t in range(6)]
    for T in (3, 40):
        steps.append((synth.hidden_states((T,), s.hidden, seed=T, tag=19), synth.prefill_logits(1, 8, T, seed=T)[0]))
    a, b, prof = _run_steps(_lib, s, w, steps, 40)
    assert prof["gateup_pagein"]["launches"] >= 6 and prof["prefill_step"]["launches"] == 1
    b.close()
    a.close()


@pytest.mark.parametrize("dtype", FORMATS)
def test_fp4_scales_are_paged_with_codes(dtype):
    """Change one block scale of s13 and of s2 (and, for NVFP4, both tensor
    scales) of one expert in its host row: once the expert is paged in again
    the output follows the new scales."""
    _lib = _need()
    s = synth.MoEShape(1, 8, 2, 2, 256, 256, dtype)
    w = synth.ExpertWeights(s, seed=5)
    m = _lib.PagedMoE(s, max_tokens=2)
    gu.load_stack(m, w)
    xb = synth.hidden_states((1,), s.hidden, seed=6)
    lg = np.full((1, 8), -3.0, np.float32)
    lg[0, 1], lg[0, 5] = 1.0, 0.8
    x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
    y0 = gu.out_bits(m.forward(0, x, l))
    row = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in w.row(0, 5).items()}
    if dtype == "mxfp4":
        row["s13"][3, 1] += 2  # x4
        row["s2"][7, 0] -= 2   # x1/4
    else:
        row["s13"][3, 1] = 0x48  # E4M3 4.0
        row["s2"][7, 0] = 0x30   # E4M3 0.5
        row["g13"] = np.float32(row["g13"] * 2)
        row["g2"] = np.float32(row["g2"] * 0.5)
    m.load_expert(0, 5, row)
    for other in ([0, 2], [3, 4]):
        lo = np.full((1, 8), -3.0, np.float32)
        lo[0, other] = [1.0, 0.9]
        m.forward(0, x, gu.to_dev_f32(lo))
    y1 = gu.out_bits(m.forward(0, x, l))
    assert not np.array_equal(y0, y1)
    ref = omlp.unpaged_layer(xb, lg, 2, lambda e: omlp.expert_weights(row if e == 5 else w.row(0, e), dtype))
    gu.check_tokens(synth.bf16_bits_to_f32(y1).astype(np.float64), ref, TOL, (dtype, "rescaled"))
    m.close()


STACKS = {"mxfp4": synth.STACK48_MXFP4, "nvfp4": synth.STACK48_NVFP4}


@pytest.fixture(scope="module", params=FORMATS)
def fp4_stack48(request):
    _lib = _need()
    s = STACKS[request.param]
    w = synth.ExpertWeights(s, seed=0)
    owner = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=512)
    gu.load_stack(owner, w)
    yield s, w, owner
    owner.close()


def test_fp4_stack48_decode_and_prefill(fp4_stack48):
    """The 48-layer FP4 stack at K = 92: 12 batch-1 decode tokens (every plan
    bit-exact, paged == K = E every layer-step, every layer of one token
    against the oracle) and one 512-token prefill chunk on the tensor-core
    path (four layers against the oracle, token by token)."""
    from host_paged_expert_gb300 import _lib

    s, w, owner = fp4_stack48
    L, E, k, K = s.num_layers, s.num_experts, s.top_k, s.num_slots
    S = 12
    lg = synth.decode_logits(L, E, S, batch=1, seed=0).transpose(1, 0, 2, 3)
    hs = synth.hidden_states((S, L, 1), s.hidden, seed=0)
    model = _lib.PagedMoE(s, max_tokens=512, store_owner=owner)
    owner.reset_residency()
    sims = [olru.ResidencySim(E, K) for _ in range(L)]
    for t in range(S):
        for l in range(L):
            x, lgt = gu.to_dev_bf16(hs[t, l]), gu.to_dev_f32(lg[t, l])
            ya, yb = model.forward(l, x, lgt), owner.forward(l, x, lgt)
            ids, wts, _ = route(lg[t, l], k)
            gu.check_plan(model.read_plan(l, 1), sims[l].step(ids), ids, wts)
            assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb)), (t, l)
            if t == S // 2:
                want = omlp.unpaged_layer(hs[t, l], lg[t, l], k, gu.expert_fn(w, l))
                gu.check_tokens(gu.out_f64(ya), want, TOL, (s.dtype, t, l))
    T = 512
    lgp = synth.prefill_logits(L, E, T, seed=1)
    hp = synth.hidden_states((L, T), s.hidden, seed=1, tag=5)
    model.profile_enable(True)
    for l in range(L):
        x, lgt = gu.to_dev_bf16(hp[l]), gu.to_dev_f32(lgp[l])
        ya, yb = model.forward(l, x, lgt), owner.forward(l, x, lgt)
        ids, wts, _ = route(lgp[l], k)
        gu.check_plan(model.read_plan(l, T), sims[l].step(ids), ids, wts)
        assert np.array_equal(gu.out_bits(ya), gu.out_bits(yb)), l
        if l in (0, 1, L // 2, L - 1):
            want = omlp.unpaged_layer(hp[l], lgp[l], k, gu.expert_fn(w, l))
            gu.check_tokens(gu.out_f64(ya), want, TOL, (s.dtype, T, l))
    assert model.profile_read()["prefill_step"]["launches"] == L
    assert model.stats(-1)["error_word"] == 0
    model.close()
