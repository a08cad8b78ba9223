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
"""
import numpy as np
import pytest

from oracle import planner, theory
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


if hyp is not None:
    @hyp.settings(max_examples=400, deadline=None)
    @hyp.given(st.composite(_case)())
    def test_plan_properties_on_arbitrary_small_shapes(case):
        _check(case)
else:
    def test_plan_properties_on_arbitrary_small_shapes():
        pytest.skip("hypothesis is not installed")
