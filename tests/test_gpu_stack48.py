"""GPU parity at full size: the 48-layer bf16 stack (H=2048, I=768, E=128,
top-8, 9.4 MB experts, 58 GB pinned host store), decoded the way bench.py
times it (one CUDA graph per token over the 48 layers).

* every plan of every layer-step (page-in experts, slots, counts, slot remap,
  routed ids) is bit-exact against the oracle's LRU simulator;
* the output of every layer-step equals the same call on a K = E handle bit
  for bit;
* sampled layer-steps (every layer of one decode token; four layers of each
  prefill chunk) match the oracle's plain MoE layer token by token: each
  token's rel-L2 is within 1e-2.
Covers the K=32 batch-1 decode workload and the K=64 graph-captured decode at
batch 1, 2, 4 and 8 (= K // top_k) with one router-bias stream per request.
"""

import numpy as np
import pytest

import gpu_util as gu
from host_paged_expert_gb300 import synth
from oracle import lru as olru
from oracle import mlp as omlp
from oracle.routing import route

pytestmark = pytest.mark.gpu

STEPS = 24


@pytest.fixture(scope="module")
def stack48():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from host_paged_expert_gb300 import _lib

    s = synth.STACK48
    w = synth.ExpertWeights(s, seed=0)
    owner = _lib.PagedMoE(s.with_slots(s.num_experts), max_tokens=2048)  # K = E: the unpaged reference
    gu.load_stack(owner, w)
    yield s, w, owner
    owner.close()


def _run(model, lg, hs, B):
    """Graph-replayed decode over the stack; returns outputs [S, L, B, H] bits
    and every layer-step's plan."""
    import torch

    L, H, E = model.shape.num_layers, model.shape.hidden, model.shape.num_experts
    stream = torch.cuda.Stream()
    x_st = torch.zeros((L, B, H), dtype=torch.bfloat16, device="cuda")
    l_st = torch.zeros((L, B, E), dtype=torch.float32, device="cuda")
    y_st = torch.zeros((L, B, H), dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for l in range(L):
            model.forward(l, x_st[l], l_st[l], y_st[l])
    outs, plans = [], []
    for t in range(lg.shape[0]):
        x_st.copy_(gu.to_dev_bf16(hs[t]))
        l_st.copy_(gu.to_dev_f32(lg[t]))
        g.replay()
        torch.cuda.synchronize()
        outs.append(gu.out_bits(y_st))
        plans.append([model.read_plan(l, B) for l in range(L)])
    return np.stack(outs), plans


def _eager(model, lg, hs, B):
    import torch

    L = model.shape.num_layers
    outs = []
    for t in range(lg.shape[0]):
        ys = []
        for l in range(L):
            ys.append(gu.out_bits(model.forward(l, gu.to_dev_bf16(hs[t, l]), gu.to_dev_f32(lg[t, l]))))
        outs.append(np.stack(ys))
    torch.cuda.synchronize()
    return np.stack(outs)


@pytest.mark.parametrize("K,B", [(32, 1), (64, 1), (64, 2), (64, 4), (64, 8)])
def test_stack48_decode(stack48, K, B):
    from host_paged_expert_gb300 import _lib

    s, w, owner = stack48
    L, E, k = s.num_layers, s.num_experts, s.top_k
    lg = synth.decode_logits(L, E, STEPS, batch=B, seed=0).transpose(1, 0, 2, 3)  # [S, L, B, E]
    hs = synth.hidden_states((STEPS, L, B), s.hidden, seed=0)
    model = _lib.PagedMoE(s.with_slots(K), max_tokens=B, store_owner=owner)
    owner.reset_residency()
    got, plans = _run(model, lg, hs, B)
    ref = _eager(owner, lg, hs, B)
    assert np.array_equal(got, ref), "paged output differs from K = E"
    sims = [olru.ResidencySim(E, K) for _ in range(L)]
    for t in range(STEPS):
        for l in range(L):
            ids, wts, _ = route(lg[t, l], k)
            plan = sims[l].step(ids)
            gu.check_plan(plans[t][l], plan, ids, wts)
    for l in (0, L // 2, L - 1):
        gu.check_residency(model.read_residency(l), sims[l])
    st = model.stats(-1)
    assert st["error_word"] == 0 and st["steps"] == STEPS * L
    # sampled values against the plain MoE layer, token by token: every layer
    # of one token, and the first and last layer-steps
    samples = [(STEPS // 2, l) for l in range(L)] + [(0, 0), (STEPS - 1, L - 1)]
    worst = 0.0
    for t, l in samples:
        want = omlp.unpaged_layer(hs[t, l], lg[t, l], k, gu.expert_fn(w, l))
        have = synth.bf16_bits_to_f32(got[t, l]).astype(np.float64)
        worst = max(worst, gu.check_tokens(have, want, gu.REL_L2["bf16"], (K, B, t, l)))
    print(f"K={K} B={B}: worst token rel-L2 over {len(samples)} layer-steps {worst:.3e}")
    model.close()


@pytest.mark.parametrize("T", [512, 2048])
def test_stack48_prefill(stack48, T):
    """One prefill chunk through all 48 layers at K=32: routing covers about
    100-128 experts per layer, so each layer-step runs 4 waves through the
    pipelined prefill step; plans bit-exact, paged == K=E bit for bit, every
    token of four layers within 1e-2 of the plain MoE layer."""
    from host_paged_expert_gb300 import _lib

    s, w, owner = stack48
    L, E, k, K = s.num_layers, s.num_experts, s.top_k, 32
    lg = synth.prefill_logits(L, E, T, seed=0)           # [L, T, E]
    hs = synth.hidden_states((L, T), s.hidden, seed=0, tag=5)
    model = _lib.PagedMoE(s.with_slots(K), max_tokens=T, store_owner=owner)
    owner.reset_residency()
    model.profile_enable(True)
    sims = [olru.ResidencySim(E, K) for _ in range(L)]
    waves = []
    for l in range(L):
        x, lgt = gu.to_dev_bf16(hs[l]), gu.to_dev_f32(lg[l])
        ya = model.forward(l, x, lgt)
        yb = owner.forward(l, x, lgt)
        ids, wts, _ = route(lg[l], k)
        plan = sims[l].step(ids)
        waves.append(len(plan.waves))
        gu.check_plan(model.read_plan(l, T), plan, ids, wts)
        got = gu.out_bits(ya)
        assert np.array_equal(got, gu.out_bits(yb)), l
        if l in (0, 1, L // 2, L - 1):  # every token of four layers against the plain MoE layer
            want = omlp.unpaged_layer(hs[l], lg[l], k, gu.expert_fn(w, l))
            gu.check_tokens(synth.bf16_bits_to_f32(got).astype(np.float64), want, gu.REL_L2["bf16"], (T, l))
    assert min(waves) >= 3
    prof = model.profile_read()
    assert prof["prefill_step"]["launches"] == L and prof["pagein"]["launches"] == 0
    assert model.stats(-1)["error_word"] == 0
    model.close()
