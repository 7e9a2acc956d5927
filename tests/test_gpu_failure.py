"""Failure detection on the GPU without a fault: every kind of bounded wait the
kernels use (the prefill step's counter wait, its mbarrier waits, the decode
step's phase wait) is run on a condition that never becomes true; each must
give up, record the timeout bit in its error word and return, and the context
must stay usable for a normal forward afterwards."""

import numpy as np
import pytest

import gpu_util as gu
from host_paged_expert_gb300 import synth
from oracle import mlp as omlp

pytestmark = pytest.mark.gpu

PE_DEVERR_TIMEOUT = 0x8  # include/pe.h


def test_bounded_waits_give_up_and_report():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from host_paged_expert_gb300 import _lib

    words = _lib.selftest_bounded_waits(1 << 15)
    assert words == [PE_DEVERR_TIMEOUT] * 3, [hex(w) for w in words]
    # the context is intact: a decode and a prefill step still match the oracle
    s = synth.TINY
    w = synth.ExpertWeights(s, seed=2)
    m = _lib.PagedMoE(s, max_tokens=64)
    gu.load_stack(m, w)
    o = omlp.PagedLayer(s.num_experts, s.num_slots, s.top_k, gu.expert_fn(w, 0))
    for T in (1, 64):
        xb = synth.hidden_states((T,), s.hidden, seed=T, tag=3)
        lg = synth.prefill_logits(1, s.num_experts, T, seed=T)[0]
        y = m.forward(0, gu.to_dev_bf16(xb), gu.to_dev_f32(lg))
        out, _, plan, ids, wts = o.step(xb, lg)
        gu.check_plan(m.read_plan(0, T), plan, ids, wts)
        assert gu.max_token_rel_l2(gu.out_f64(y), out) <= gu.REL_L2["bf16"], T
    assert m.stats(0)["error_word"] == 0
    m.close()
