"""pe_expert_mlp_noalloc: the expert MLP for callers that cannot allocate.

Some callers cannot allocate device memory where they need the computation
(code that may only use buffers a framework hands it, or a path that must
not synchronise the device by calling cudaMalloc).  This entry point keeps
its scratch in a static device array instead.  It is checked here, through
the C ABI, against pe_forward on a one-expert layer (E = K = top_k = 1, so the
router weight is exactly 1 and the layer output is that expert's MLP), on two
calls in a row: bit for bit up to 64 tokens, within the bf16 tolerance above
that; and against the oracle's expert MLP.  Its size limit is checked too.
This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest

import gpu_util as gu
from host_paged_expert_gb300 import synth
from oracle import mlp as omlp

pytestmark = pytest.mark.gpu


def _load():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from host_paged_expert_gb300 import _lib

    return _lib


def _call(L, w13, w2, x, out, T, H, I, stream):
    return L.pe_expert_mlp_noalloc(ctypes.c_void_p(w13.data_ptr()), ctypes.c_void_p(w2.data_ptr()),
                                   ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(out.data_ptr()), T, H, I,
                                   ctypes.c_void_p(stream))


def _one_expert(max_tokens):
    from host_paged_expert_gb300 import _lib

    s = synth.MoEShape(1, 1, 1, 1, 256, 128, "bf16")
    w = synth.ExpertWeights(s, seed=21)
    row = w.row(0, 0)
    model = _lib.PagedMoE(s, max_tokens=max_tokens)
    model.load_expert(0, 0, row)
    return s, row, model


def _oracle(row, xb):
    w13, w2 = omlp.expert_weights(row, "bf16")
    return omlp.expert_mlp(omlp.bf16_to_f64(xb), w13, w2)


@pytest.mark.parametrize("sizes", [(5, 8), (64, 64)])
def test_noalloc_mlp_matches_forward_twice(sizes):
    """Up to 64 tokens pe_forward serves a one-expert layer with its GEMV
    decode kernels, whose arithmetic the no-alloc kernels share: bit-equal
    results on two calls in a row, and within the bf16 tolerance of the
    oracle's expert MLP."""
    _lib = _load()
    import torch

    L = _lib.lib()
    s, row, model = _one_expert(64)
    w13 = gu.to_dev_bf16(row["w13"])
    w2 = gu.to_dev_bf16(row["w2"])
    stream = torch.cuda.current_stream().cuda_stream
    for call, T in enumerate(sizes):
        xb = synth.hidden_states((T,), s.hidden, seed=22, tag=call)
        x = gu.to_dev_bf16(xb)
        ref = model.forward(0, x, torch.zeros((T, 1), dtype=torch.float32, device="cuda"))
        out = torch.full_like(x, float("nan"))
        st = _call(L, w13, w2, x, out, T, s.hidden, s.intermediate, stream)
        assert st == _lib.PE_OK, L.pe_last_error(None)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (call, T)
        got = gu.out_f64(out)
        assert np.isfinite(got).all()
        worst = gu.max_token_rel_l2(got, _oracle(row, xb))
        assert worst <= gu.REL_L2["bf16"], (call, T, worst)
    model.close()


def test_noalloc_mlp_above_64_tokens_within_tolerance():
    """Above 64 tokens pe_forward takes its tensor-core path, which rounds
    differently: there the two entry points agree within the bf16 tolerance,
    per token, and both stay within it of the oracle."""
    _lib = _load()
    import torch

    L = _lib.lib()
    T = 100
    s, row, model = _one_expert(T)
    w13 = gu.to_dev_bf16(row["w13"])
    w2 = gu.to_dev_bf16(row["w2"])
    xb = synth.hidden_states((T,), s.hidden, seed=23)
    x = gu.to_dev_bf16(xb)
    ref = model.forward(0, x, torch.zeros((T, 1), dtype=torch.float32, device="cuda"))
    out = torch.full_like(x, float("nan"))
    st = _call(L, w13, w2, x, out, T, s.hidden, s.intermediate, torch.cuda.current_stream().cuda_stream)
    assert st == _lib.PE_OK, L.pe_last_error(None)
    torch.cuda.synchronize()
    got, fwd, want = gu.out_f64(out), gu.out_f64(ref), _oracle(row, xb)
    assert np.isfinite(got).all()
    assert gu.max_token_rel_l2(got, fwd) <= gu.REL_L2["bf16"]
    assert gu.max_token_rel_l2(got, want) <= gu.REL_L2["bf16"]
    assert gu.max_token_rel_l2(fwd, want) <= gu.REL_L2["bf16"]
    model.close()


def test_noalloc_rejects_sizes_beyond_scratch():
    _lib = _load()
    import torch

    L = _lib.lib()
    H, I = 256, 1024
    T = (1 << 20) // (4 * I) + 1  # one token more than the scratch holds
    w13 = torch.zeros((2 * I, H), dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros((H, I), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(x)
    st = _call(L, w13, w2, x, out, T, H, I, torch.cuda.current_stream().cuda_stream)
    assert st == _lib.PE_ERR_RANGE
    assert b"PE_NOALLOC_SCRATCH_BYTES" in L.pe_last_error(None)
    assert _call(L, w13, w2, x, out, T - 1, H, I, torch.cuda.current_stream().cuda_stream) == _lib.PE_OK
    torch.cuda.synchronize()
