"""pe_create_external on the GPU: a host store in a shared mapping, filled
through one handle (filled = 0) and read by another created on the same
mapping with filled = 1, as each replica process would.  The reading handle
matches a handle with its own pinned store bit for bit, over decode steps and
a multi-wave prefill chunk, and flags no unloaded expert."""

import os
import tempfile

import numpy as np
import pytest

import gpu_util as gu
from host_paged_expert_gb300 import synth

pytestmark = pytest.mark.gpu


def test_external_shared_store_matches_private_store():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from host_paged_expert_gb300 import _lib, shared_store

    s = synth.TINY
    w = synth.ExpertWeights(s, seed=0)
    base = "/dev/shm" if os.access("/dev/shm", os.W_OK) else None
    d = tempfile.mkdtemp(dir=base)
    store = shared_store.SharedHostStore(os.path.join(d, "store"), _lib.host_store_bytes(s), create=True)
    try:
        filler = _lib.PagedMoE(s, max_tokens=64, host_store=store, filled=False)
        gu.load_stack(filler, w)
        reader = _lib.PagedMoE(s, max_tokens=64, host_store=store, filled=True)
        private = _lib.PagedMoE(s, max_tokens=64)
        gu.load_stack(private, w)
        dec = synth.decode_logits(1, s.num_experts, 8, seed=3)[0, :, 0, :]
        xs = synth.hidden_states((8,), s.hidden, seed=3)
        steps = [(xs[t : t + 1], dec[t : t + 1]) for t in range(8)]
        steps.append((synth.hidden_states((64,), s.hidden, seed=3, tag=3), synth.prefill_logits(1, 16, 64, seed=3)[0]))
        for xb, lg in steps:
            x, l = gu.to_dev_bf16(xb), gu.to_dev_f32(lg)
            assert np.array_equal(gu.out_bits(reader.forward(0, x, l)), gu.out_bits(private.forward(0, x, l)))
        assert reader.stats(0)["error_word"] == 0 and reader.stats(0)["page_ins"] > 0
        # the reader's host rows are the filler's bytes, at the same address
        assert reader.host_row(0, 3).ctypes.data == filler.host_row(0, 3).ctypes.data
        for m in (reader, private, filler):
            m.close()
    finally:
        store.close()
        os.rmdir(d)
