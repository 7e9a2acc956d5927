"""Checks that tie the CPU oracle to facts fixed outside itself.

Each ``check_*`` takes the oracle piece it checks as an argument, so the
mutation tests can hand it a deliberately broken copy and confirm the check
fails.  Sources of truth: the pages' printed numbers (tests/golden), closed
forms, library routines (scipy, torch's float8 decoding), brute force on tiny
inputs, and a second LRU model written differently (lru_textbook).
"""

from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import scipy.special

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- routing


def check_route_brute_force(route, seed=0):
    """The chosen set maximises the sum of logits over all C(E,k) subsets
    (softmax is increasing, so top-k probabilities = top-k logits), entries are
    in descending logit order and the weights are the softmax over E
    renormalised on the chosen set."""
    rng = np.random.default_rng(seed)
    for E in (3, 5, 8):
        for k in range(1, min(E, 4) + 1):
            logits = rng.standard_normal((6, E)).astype(np.float32)
            ids, w, nan = route(logits, k)
            assert not nan
            for t in range(logits.shape[0]):
                best = max(itertools.combinations(range(E), k),
                           key=lambda c: sum(float(logits[t, i]) for i in c))
                assert set(ids[t].tolist()) == set(best), (E, k, t)
                vals = logits[t, ids[t]]
                assert np.all(vals[:-1] >= vals[1:])
                p = scipy.special.softmax(logits[t].astype(np.float64))
                ref = p[ids[t]] / p[ids[t]].sum()
                assert np.allclose(w[t], ref, rtol=1e-12, atol=0), (w[t], ref)


def check_route_weights(route):
    """Weights sum to one; top-1 gets exactly 1; for top-2 the first weight is
    the logistic of the logit gap (closed form); weights do not depend on the
    logits of experts that were not chosen."""
    rng = np.random.default_rng(1)
    logits = (rng.standard_normal((16, 12)) * 3).astype(np.float32)
    for k in (1, 2, 5):
        ids, w, _ = route(logits, k)
        assert np.allclose(w.sum(1), 1.0, atol=1e-12)
        if k == 1:
            assert np.all(w == 1.0)
        if k == 2:
            l0 = logits[np.arange(16), ids[:, 0]].astype(np.float64)
            l1 = logits[np.arange(16), ids[:, 1]].astype(np.float64)
            assert np.allclose(w[:, 0], scipy.special.expit(l0 - l1), rtol=1e-12)
        lower = logits.copy()
        for t in range(16):
            others = np.setdiff1d(np.arange(12), ids[t])
            lower[t, others] -= 5.0
        ids2, w2, _ = route(lower, k)
        assert np.array_equal(ids, ids2)
        assert np.allclose(w, w2, rtol=1e-12)


def check_route_ties(route):
    """Equal logits go to the lower expert id first."""
    logits = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]], np.float32)
    ids, _, _ = route(logits, 2)
    assert ids.tolist() == [[1, 2]]
    ids, _, _ = route(logits, 4)
    assert ids.tolist() == [[1, 2, 4, 3]]
    ids, w, _ = route(np.zeros((1, 6), np.float32), 3)
    assert ids.tolist() == [[0, 1, 2]] and np.allclose(w, 1 / 3)


def check_route_nan(route):
    logits = np.array([[0.5, np.nan, 2.0, -1.0]], np.float32)
    ids, w, nan = route(logits, 2)
    assert nan
    assert ids.tolist() == [[2, 0]]
    assert np.allclose(w[0], scipy.special.softmax([2.0, 0.5]), rtol=1e-12)
    # every logit NaN: tie rule picks ids 0..k-1 with equal weights
    ids, w, nan = route(np.full((1, 5), np.nan, np.float32), 3)
    assert nan and ids.tolist() == [[0, 1, 2]]
    assert np.all(w == 1.0 / 3.0)


# ---------------------------------------------------------------- fp8


def check_e4m3_table(decode_e4m3):
    """Every code decodes as torch's float8_e4m3fn does, plus named values."""
    import torch

    codes = np.arange(256, dtype=np.uint8)
    ours = decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    named = {0x7E: 448.0, 0xFE: -448.0, 0x38: 1.0, 0xB8: -1.0, 0x01: 2.0**-9,
             0x08: 2.0**-6, 0x07: 7 * 2.0**-9, 0x40: 2.0, 0x3C: 1.5}
    for c, v in named.items():
        assert ours[c] == v, (hex(c), ours[c], v)


def check_block_dequant(dequant_block):
    """Codes of 1.0 times a distinct scale per block reproduce the scale grid
    expanded over 128x128 blocks, including a ragged last block."""
    n, c = 200, 300
    codes = np.full((n, c), 0x38, np.uint8)
    scales = (np.arange(2 * 3, dtype=np.float32).reshape(2, 3) + 1) * 0.25
    w = dequant_block(codes, scales)
    for r in (0, 127, 128, 199):
        for q in (0, 127, 128, 255, 256, 299):
            assert w[r, q] == scales[r // 128, q // 128], (r, q)
    codes2 = codes.copy()
    codes2[5, 7] = 0xC0  # -2.0
    w2 = dequant_block(codes2, scales)
    assert w2[5, 7] == -2.0 * scales[0, 0]


# ---------------------------------------------------------------- mlp


def check_mlp_hand(expert_mlp):
    """H = I = 1 written out by hand: y = wd * silu(wg x) * (wu x)."""
    x = np.array([[2.0]])
    w13 = np.array([[0.5], [3.0]])  # row 0 gate, row 1 up
    w2 = np.array([[-1.5]])
    g, u = 1.0, 6.0
    ref = -1.5 * (g * scipy.special.expit(g)) * u
    y = expert_mlp(x, w13, w2)
    assert y.shape == (1, 1)
    assert math.isclose(float(y[0, 0]), ref, rel_tol=1e-14)


def check_mlp_brute_force(expert_mlp, seed=2):
    """Pure-Python loops over every index equal the batched form; shapes are
    all different so a transposed operand cannot pass."""
    rng = np.random.default_rng(seed)
    M, H, I = 3, 5, 4
    x = rng.standard_normal((M, H))
    w13 = rng.standard_normal((2 * I, H))
    w2 = rng.standard_normal((H, I))
    y = expert_mlp(x, w13, w2)
    assert y.shape == (M, H)
    for m in range(M):
        for o in range(H):
            acc = 0.0
            for i in range(I):
                g = sum(x[m, c] * w13[i, c] for c in range(H))
                u = sum(x[m, c] * w13[I + i, c] for c in range(H))
                acc += w2[o, i] * (g / (1.0 + math.exp(-g))) * u
            assert math.isclose(float(y[m, o]), acc, rel_tol=1e-10, abs_tol=1e-12)


def check_silu(silu):
    z = np.linspace(-30, 30, 121)
    assert np.allclose(silu(z), z * scipy.special.expit(z), rtol=1e-13, atol=1e-300)
    assert silu(np.array([0.0]))[0] == 0.0


def check_topk_sum(topk_sum):
    rng = np.random.default_rng(3)
    merged = rng.standard_normal((4, 3, 6))
    out = topk_sum(merged)
    assert out.shape == (4, 6)
    ref = (merged[:, 0] + merged[:, 1]) + merged[:, 2]
    assert np.array_equal(out, ref)


def layer_brute_force(x, logits, top_k, get_expert, route):
    """Per-token, per-entry loop of the plain MoE layer."""
    ids, w, _ = route(logits, top_k)
    out = np.zeros_like(x)
    for t in range(x.shape[0]):
        for j in range(top_k):
            w13, w2 = get_expert(int(ids[t, j]))
            inter = w2.shape[1]
            g = w13[:inter] @ x[t]
            u = w13[inter:] @ x[t]
            h = g / (1 + np.exp(-g)) * u
            out[t] += w[t, j] * (w2 @ h)
    return out


# ---------------------------------------------------------------- lru


def lru_hand_traces():
    """Traces worked out by hand from the LRU rules: (E, K, steps, expected)
    where expected per step is a list of waves (plan pairs, hits)."""
    return [
        # cold fills go to empty slots in slot order; then the oldest slot
        # (lowest tick, then lowest slot) is the victim; a slot touched by a
        # hit and a slot filled in the same wave tie, and the lower slot goes.
        (4, 2, [[0, 1], [2], [1, 3], [0]],
         [[([(0, 0), (1, 1)], 0)],
          [([(2, 0)], 0)],
          [([(3, 0)], 1)],
          [([(0, 0)], 0)]]),
        # three distinct experts, two slots: two waves; wave 2 evicts the
        # oldest slot, which holds an expert of wave 1.
        (4, 2, [[2, 0, 1], [1]],
         [[([(0, 0), (1, 1)], 0), ([(2, 0)], 0)],
          [([], 1)]]),
        # hits refresh a slot's tick, so the victim is the least recently
        # used slot, not the lowest one.
        (5, 3, [[0, 1, 2], [0], [1], [3], [4]],
         [[([(0, 0), (1, 1), (2, 2)], 0)],
          [([], 1)],
          [([], 1)],
          [([(3, 2)], 0)],
          [([(4, 0)], 0)]]),
        # resident experts go first and are never evicted by their own wave;
        # the second wave may evict what the first one just paged in.
        (6, 3, [[0, 1, 2], [5, 2, 4, 3]],
         [[([(0, 0), (1, 1), (2, 2)], 0)],
          [([(3, 0), (4, 1)], 1), ([(5, 0)], 0)]]),
    ]


def check_lru_hand(sim_cls):
    for E, K, steps, expected in lru_hand_traces():
        sim = sim_cls(E, K)
        for ids, exp_waves in zip(steps, expected):
            plan = sim.step(np.array([ids]))
            got = [(list(zip(w.plan_expert, w.plan_slot)), w.hits) for w in plan.waves]
            assert got == exp_waves, (E, K, ids, got, exp_waves)
            sim.check_invariants()


def check_lru_textbook(sim_cls, max_e=5, max_len=3):
    """Exhaustive: every sequence of routed sets (size 1..3) of length
    ``max_len`` over E experts, for every K, plans like the recency-list LRU."""
    from lru_textbook import TextbookLRU

    for E in range(2, max_e + 1):
        sets = [c for r in range(1, min(3, E) + 1) for c in itertools.combinations(range(E), r)]
        for K in range(1, min(4, E) + 1):
            for seq in itertools.product(sets, repeat=max_len):
                a = sim_cls(E, K)
                b = TextbookLRU(E, K)
                for routed in seq:
                    plan = a.step(np.array([list(routed)]))
                    ref = b.step(routed)
                    got = [(w.experts, list(zip(w.plan_expert, w.plan_slot)), w.hits)
                           for w in plan.waves]
                    assert got == [(m, c, h) for m, c, h in ref], (E, K, seq, got, ref)
                    res = {e: s for e, s in enumerate(a.expert_slot) if s >= 0}
                    assert res == b.resident_map()


# ---------------------------------------------------------------- int4


def _pack_rows_by_hand(q):
    """Integer codes [N, K] -> row-layout bytes, written as plain loops."""
    n, k = len(q), len(q[0])
    out = np.zeros((n, k // 2), dtype=np.uint8)
    for r in range(n):
        for j in range(k // 2):
            out[r, j] = int(q[r][2 * j]) | (int(q[r][2 * j + 1]) << 4)
    return out


def _pack_gptq_by_hand(q):
    """Integer codes [N, K] -> checkpoint qweight int32 [K/8, N], by loops."""
    n, k = len(q), len(q[0])
    out = np.zeros((k // 8, n), dtype=np.uint32)
    for c in range(n):
        for r in range(k // 8):
            word = 0
            for i in range(8):
                word |= int(q[c][8 * r + i]) << (4 * i)
            out[r, c] = word
    return out.view(np.int32)


def check_int4_values(dequant_rows):
    """Hand values: a byte 0x9F holds 15 (low) and 9 (high), i.e. +7 and +1
    around the zero point 8; every code 8 dequantises to 0; codes 0..15 give
    -8..7 times the scale."""
    codes = np.array([[0x9F] + [0x88] * 63], dtype=np.uint8)  # one row, K = 128
    w = dequant_rows(codes, np.array([[0.5]], dtype=np.float16))
    assert w.shape == (1, 128)
    assert w[0, 0] == 3.5 and w[0, 1] == 0.5 and not w[0, 2:].any()
    q = np.tile(np.arange(16), 8).reshape(1, 128)  # K = 128: 0..15 eight times
    w = dequant_rows(_pack_rows_by_hand(q), np.array([[0.25]], dtype=np.float16))
    assert np.array_equal(w[0, :16], (np.arange(16) - 8) * 0.25)


def check_int4_brute_force(dequant_rows, seed=0):
    """Plain loops over (n, k) with the group index written out, on
    non-square shapes with more than one group."""
    rng = np.random.default_rng(seed)
    for n, k in ((3, 256), (5, 384)):
        q = rng.integers(0, 16, size=(n, k))
        s = (rng.random((n, k // 128)) + 0.1).astype(np.float16)
        w = dequant_rows(_pack_rows_by_hand(q), s)
        for r in range(n):
            for c in range(k):
                assert w[r, c] == (q[r, c] - 8) * float(s[r, c // 128]), (r, c)


def check_int4_gptq_layout(dequant_gptq, seed=1):
    """The checkpoint layout (8 codes per int32 along the input, scales
    [K/128, N]) dequantises to the same matrix as loops over the codes."""
    rng = np.random.default_rng(seed)
    n, k = 6, 256
    q = rng.integers(0, 16, size=(n, k))
    s = (rng.random((n, k // 128)) + 0.1).astype(np.float16)
    w = dequant_gptq(_pack_gptq_by_hand(q), np.ascontiguousarray(s.T))
    assert w.shape == (n, k)
    for r in range(n):
        for c in range(k):
            assert w[r, c] == (q[r, c] - 8) * float(s[r, c // 128]), (r, c)


# ---------------------------------------------------------------- fp4 (MXFP4, NVFP4)

# The sixteen E2M1 values, typed from the format's published value list
# (positive codes 0..7, then the same magnitudes negated).
E2M1_BY_HAND = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def check_e2m1_table(decode_e2m1):
    got = decode_e2m1(np.arange(16))
    assert got.tolist() == E2M1_BY_HAND
    assert np.signbit(got[8]) and not np.signbit(got[0])


def check_e8m0_table(decode_e8m0):
    """Every E8M0 code against torch's float8_e8m0fnu decoding."""
    import torch

    want = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = decode_e8m0(np.arange(256, dtype=np.uint8))
    assert np.isnan(got[255]) and np.isnan(want[255])
    assert np.array_equal(got[:255], want[:255])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127


def _pack_fp4_by_hand(q):
    """4-bit codes [N, K] -> row bytes [N, K/2], input 2j in the low nibble."""
    n, k = len(q), len(q[0])
    out = np.zeros((n, k // 2), dtype=np.uint8)
    for r in range(n):
        for j in range(k // 2):
            out[r, j] = int(q[r][2 * j]) | (int(q[r][2 * j + 1]) << 4)
    return out


def check_fp4_hand_values(dequant_mx, dequant_nv):
    """A byte 0x9F holds code 15 (-6) in its low nibble and code 9 (-0.5) in
    its high one.  MX scale code 126 halves; NV: an E4M3 block scale of 2.0
    (code 0x40) times a global scale of 0.25."""
    codes = np.array([[0x9F] + [0x00] * 15], dtype=np.uint8)  # one row, K = 32
    w = dequant_mx(codes, np.array([[126]], dtype=np.uint8))
    assert w.shape == (1, 32)
    assert w[0, 0] == -3.0 and w[0, 1] == -0.25 and not w[0, 2:].any()
    w = dequant_nv(codes, np.array([[0x40, 0x38]], dtype=np.uint8), 0.25)  # 2.0 and 1.0
    assert w[0, 0] == -3.0 and w[0, 1] == -0.25 and not w[0, 2:16].any()


def check_fp4_brute_force(dequant_mx, dequant_nv, seed=3):
    """Plain loops over (n, k) with each block index written out, on
    non-square shapes with several blocks per row; the NV global scale is an
    fp32 value."""
    from oracle.fp8 import e4m3_value

    rng = np.random.default_rng(seed)
    for n, k in ((3, 64), (5, 96)):
        q = rng.integers(0, 16, size=(n, k))
        packed = _pack_fp4_by_hand(q)
        smx = rng.integers(118, 134, size=(n, k // 32)).astype(np.uint8)
        w = dequant_mx(packed, smx)
        for r in range(n):
            for c in range(k):
                assert w[r, c] == E2M1_BY_HAND[q[r, c]] * 2.0 ** (int(smx[r, c // 32]) - 127), (r, c)
        snv = rng.integers(0x20, 0x58, size=(n, k // 16)).astype(np.uint8)
        g = float(np.float32(0.0123))
        w = dequant_nv(packed, snv, g)
        for r in range(n):
            for c in range(k):
                assert w[r, c] == E2M1_BY_HAND[q[r, c]] * e4m3_value(snv[r, c // 16]) * g, (r, c)
