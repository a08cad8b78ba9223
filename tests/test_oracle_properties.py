"""Properties of the oracle's plan on arbitrary small shapes (CPU only).

Hypothesis draws the shape -- R ranks, L experts per rank, K experts per token
(up to E), S tokens per rank, training or inference with any slot count the
mode allows, either planner policy -- and a routing with K distinct experts
per token, and checks what Theorem 1 and the buffer contract fix for any valid
plan (Kimi K3 模型结构（8）, section 定理 1; Moonshot AI 开源 MoonEP, contract
paragraph): every rank computes exactly S*K copies, at most R-1 fills, every
receiving rank's copies come from one source rank and at most E/R of its
experts, destinations are a bijection and every copy lands in its expert's
group; and the send-once route entries decode back to the destinations with
one payload-carrying entry per (token, destination rank) (section 在线规划、
零拷贝、静态 shape).  On the tiniest draws the planner's largest per-rank
redundant count is compared with the exact minimax found by brute force.
On the same draws the plan-driven layer (permute, grouped GEMM over the
[E+B, H, H'] rows, combine, reduce_grad) is checked against its plan-free
definitions: a plan changes where a copy is computed, never its result.
"""
import numpy as np
import pytest

from oracle import layer, planner, theory
from oracle.planner import Dims
from tests.invariants import check_plan_arrays

try:
    import hypothesis as hyp
    import hypothesis.strategies as st
except ImportError:  # the property test needs hypothesis; everything else runs without
    hyp = st = None


def _case(draw):
    R = draw(st.integers(1, 6))
    L = draw(st.integers(1, 4))
    E = R * L
    K = draw(st.integers(1, min(E, 4)))
    S = draw(st.integers(1, 12))
    mode = draw(st.integers(0, 1))
    B = draw(st.integers(L, L + 2)) if mode == 0 else draw(st.integers(0, L))
    policy = draw(st.integers(0, 1))
    # per token: K distinct experts, drawn as a random permutation prefix;
    # a popularity skew makes fills likely
    skew = draw(st.floats(0.0, 3.0))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    p = (np.arange(E) + 1.0) ** -skew
    p = p[rng.permutation(E)]
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=K, replace=False, p=p) for _ in range(R * S)])
    return Dims(R=R, E=E, B=B, K=K, S=S, mode=mode, policy=policy), idx.reshape(R, S, K)


def _check(case):
    d, idx = case
    fp = planner.full_plan(idx, d)
    check_plan_arrays(idx, d.R, d.E, d.B, d.K, d.S, d.mode, T=fp["T"], n_fills=fp["n_fills"],
                      fills=fp["fills"], keep=fp["keep"], slot_expert=fp["slot_expert"],
                      n_recv=fp["n_recv"], src=fp["src"], cu_seqlens=fp["cu_seqlens"],
                      dst=fp["dst"], inverse=fp["inverse"], gidx=fp["gidx"])
    # the fills never exceed the proof's bounds
    assert fp["n_fills"] <= max(d.R - 1, 0)
    assert int(fp["n_recv"].max(initial=0)) <= d.L
    # inference: experts beyond the slots run from their home rows on the receiver
    p = fp["plan"]
    for u in range(d.R):
        assert len(p.overflow[u]) == max(0, int(p.n_recv[u]) - d.B)
    # send-once route entries
    enc = planner.route_encoding(fp["dst"], d).reshape(-1, d.K)
    dst = fp["dst"].reshape(-1, d.K)
    dec = np.where(enc >= 0, enc, -enc - 1)
    assert np.array_equal(dec, dst % d.C)
    for t in range(dst.shape[0]):
        ranks = dst[t] // d.C
        assert sorted(ranks[enc[t] >= 0].tolist()) == sorted(set(ranks.tolist()))
    # exact minimax on the tiniest draws
    if d.R <= 3 and d.L <= 2 and d.mode == 0:
        m, _ = theory.min_max_redundant(fp["T"], d.R, d.C, m_max=d.L)
        assert m is not None and m <= int(fp["n_recv"].max(initial=0))


def _check_layer(case):
    """Whatever the plan, the plan-driven layer equals the plan-free one: the
    grouped GEMM over each rank's buffer gives every copy bf16(x W_e), the
    combine equals the per-copy definition, and reduce_grad conserves the sum
    of home and slot gradients (small integers, so exactly)."""
    d0, idx = case
    rng = np.random.default_rng(int(idx.sum()) + d0.R)
    d = Dims(R=d0.R, E=d0.E, B=d0.B, K=d0.K, S=d0.S, H=8, Hp=5, mode=d0.mode, policy=d0.policy)
    x = layer.to_bf16(rng.integers(-3, 4, size=(d.R, d.S, d.H)).astype(np.float64))
    w = layer.to_bf16(rng.integers(-3, 4, size=(d.E, d.H, d.Hp)).astype(np.float64))
    gates = rng.random((d.R, d.S, d.K)).astype(np.float32)
    fp = planner.full_plan(idx, d)
    y_rows = layer.grouped_gemm_rows(layer.permute(x, fp["dst"], d), fp["plan"], w)
    per_e = layer.expert_outputs(x, w, idx, d)
    dst = fp["dst"].reshape(-1)
    for e, (cids, yb) in per_e.items():
        assert np.array_equal(y_rows[dst[cids]], yb)
    assert np.array_equal(layer.combine(y_rows, fp["dst"], gates, d),
                          layer.combine_from_copies(per_e, gates, d))
    if d.B:
        gh = rng.integers(-9, 10, size=(d.E, 2, 3)).astype(np.float32)
        gs = rng.integers(-9, 10, size=(d.R, d.B, 2, 3)).astype(np.float32)
        gs[fp["slot_expert"] < 0] = 0.0
        total = gh.astype(np.float64).sum() + gs.astype(np.float64).sum()
        layer.reduce_grad(gh, gs, fp["plan"])
        assert np.all(gs == 0.0) and gh.astype(np.float64).sum() == total


if hyp is not None:
    @hyp.settings(max_examples=400, deadline=None)
    @hyp.given(st.composite(_case)())
    def test_plan_properties_on_arbitrary_small_shapes(case):
        _check(case)

    @hyp.settings(max_examples=150, deadline=None)
    @hyp.given(st.composite(_case)())
    def test_layer_is_plan_independent_on_arbitrary_small_shapes(case):
        _check_layer(case)
else:
    def test_plan_properties_on_arbitrary_small_shapes():
        pytest.skip("hypothesis is not installed")

    def test_layer_is_plan_independent_on_arbitrary_small_shapes():
        pytest.skip("hypothesis is not installed")
