"""Seeded input generators: determinism, formats and distributions (CPU)."""

import numpy as np
import torch

from host_paged_expert_gb300 import synth


def test_bf16_rounding_matches_torch():
    z = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 7
    z[:4] = [0.0, -0.0, 1e-40, 3.0e38]
    ours = synth.f32_to_bf16_bits(z)
    ref = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_bits_to_f32(ours), torch.from_numpy(z).to(torch.bfloat16).float().numpy())


def test_expert_weights_deterministic_and_distinct():
    s = synth.TINY
    a = synth.ExpertWeights(s, seed=0)
    b = synth.ExpertWeights(s, seed=0)
    r0, r1 = a.row(0, 3), b.row(0, 3)
    assert np.array_equal(r0["w13"], r1["w13"]) and np.array_equal(r0["w2"], r1["w2"])
    assert r0["w13"].shape == (2 * s.intermediate, s.hidden) and r0["w2"].shape == (s.hidden, s.intermediate)
    rows = [a.row(0, e)["w13"] for e in range(s.num_experts)]
    for i in range(len(rows)):
        for j in range(i + 1, len(rows)):
            assert not np.array_equal(rows[i], rows[j])
    w = synth.bf16_bits_to_f32(r0["w13"])
    assert abs(w.std() - 0.02) < 0.002 and abs(w.mean()) < 0.002


def test_fp8_expert_rows():
    s = synth.MoEShape(1, 4, 2, 2, 256, 192, "fp8")
    r = synth.ExpertWeights(s).row(0, 1)
    assert r["w13"].dtype == np.uint8 and r["w13"].shape == (384, 256)
    assert r["s13"].shape == (3, 2) and r["s2"].shape == (2, 2)
    assert not np.any((r["w13"] & 0x7F) == 0x7F)  # no NaN codes
    assert np.all(r["s13"] > 0)
    assert s.expert_bytes == 3 * 256 * 192 + 4 * (6 + 4)


def test_decode_logits_drift():
    lg = synth.decode_logits(2, 64, 400, batch=2, seed=0)
    assert lg.shape == (2, 400, 2, 64) and lg.dtype == np.float32
    assert np.array_equal(lg, synth.decode_logits(2, 64, 400, batch=2, seed=0))
    # requests have independent bias streams
    assert not np.allclose(lg[0, :, 0], lg[0, :, 1])
    # total sd = sqrt(2^2 + 1) and consecutive tokens are correlated
    x = lg[:, :, 0, :]
    assert abs(x.std() - np.sqrt(5)) < 0.3
    c = np.corrcoef(x[:, 1:].reshape(-1), x[:, :-1].reshape(-1))[0, 1]
    assert 0.6 < c < 0.85  # 0.9 * 4 / 5 = 0.72


def test_zipf_prior_and_prefill():
    lg = synth.decode_logits(1, 32, 10, zipf_s=1.1)
    assert np.isfinite(lg).all()
    p = synth.prefill_logits(3, 128, 64)
    assert p.shape == (3, 64, 128)
    h = synth.hidden_states((2, 3), 16)
    assert h.shape == (2, 3, 16) and h.dtype == np.uint16


def test_fp4_expert_rows():
    """MXFP4 / NVFP4 rows: packed E2M1 codes in the int4 layout covering all
    sixteen codes, byte scale grids of the format's block, NVFP4 tensor
    scales, and distinct experts."""
    for dt, blk in (("mxfp4", 32), ("nvfp4", 16)):
        s = synth.MoEShape(2, 4, 2, 2, 256, 384, dt)
        w = synth.ExpertWeights(s, seed=1)
        r = w.row(1, 2)
        assert r["w13"].shape == (2 * 384, 128) and r["w2"].shape == (256, 192)
        assert r["s13"].shape == (2 * 384, 256 // blk) and r["s2"].shape == (256, 384 // blk)
        assert r["w13"].dtype == np.uint8 and r["s13"].dtype == np.uint8
        codes = np.concatenate([r["w13"].ravel() & 0xF, r["w13"].ravel() >> 4])
        assert set(np.unique(codes).tolist()) == set(range(16))
        if dt == "nvfp4":
            assert r["g13"].dtype == np.float32 and 0.005 < float(r["g13"]) < 0.03
        assert not np.array_equal(r["w13"], w.row(1, 3)["w13"])
        assert s.expert_bytes == 3 * 256 * 384 // 2 + (2 * 384 * 256 + 256 * 384) // blk + (8 if dt == "nvfp4" else 0)
