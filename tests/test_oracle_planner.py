"""The planner oracle pinned to what the pages and mathematics fix (CPU only)."""
import json
import os

import numpy as np
import pytest

from oracle import planner, theory
from oracle.planner import Dims
from perfectly_balanced_token_gb300 import synthetic as syn
from tests.invariants import check_plan_arrays

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _full(idx, d):
    fp = planner.full_plan(idx, d)
    check_plan_arrays(idx, d.R, d.E, d.B, d.K, d.S, d.mode, T=fp["T"],
                      n_fills=fp["n_fills"], fills=fp["fills"], keep=fp["keep"],
                      slot_expert=fp["slot_expert"], n_recv=fp["n_recv"],
                      src=fp["src"], cu_seqlens=fp["cu_seqlens"], dst=fp["dst"],
                      inverse=fp["inverse"], gidx=fp["gidx"])
    return fp


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "hand_plans.json")))["cases"],
                         ids=lambda c: c["name"])
def test_hand_worked_plans(case):
    d = Dims(**case["dims"])
    idx = np.asarray(case["idx"], dtype=np.int64)
    fp = _full(idx, d)
    assert fp["T"].tolist() == case["T"]
    assert fp["load"].tolist() == case["load"]
    assert fp["fills"][:fp["n_fills"]].tolist() == case["fills"]
    assert fp["keep"].tolist() == case["keep"]
    assert fp["slot_expert"].tolist() == case["slot_expert"]
    assert fp["src"].tolist() == case["src"]
    assert fp["cu_seqlens"].tolist() == case["cu_seqlens"]
    assert fp["dst"].reshape(-1).tolist() == case["dst"]
    assert fp["inverse"].tolist() == case["inverse"]


THM2 = json.load(open(os.path.join(GOLD, "theorem2.json")))


@pytest.mark.parametrize("case", THM2["cases"], ids=lambda c: c["name"])
def test_theorem2_worst_case(case):
    R, E, K, S = case["R"], case["E"], case["K"], case["S"]
    d = Dims(R=R, E=E, B=E // R, K=K, S=S)
    rt = syn.round_robin_routing(R, S, K, E, first=E // R)
    counts, T, load = planner.histogram(rt.idx, d)
    assert load.tolist() == case["loads"]
    assert theory.theorem2_bound(R, E) == case["bound"]
    p = planner.build_plan(rt.idx, d)
    assert [[f.u, f.o, f.d] for f in p.fills] == case["fills"]
    assert p.n_recv.tolist() == case["redundant_per_rank"]
    # rank 0 reaches the bound: the construction is tight on this input
    assert p.n_recv[0] == case["bound"]
    # and no plan at all can do better for rank 0 (per-expert supply bound)
    assert theory.rank_lower_bound(d.C, int(load[0]), int(T.max())) == case["bound"]


def test_slot_budget_table():
    tab = THM2["slot_budget_table"]
    for R, want in tab["R_to_slots"].items():
        assert Dims(R=int(R), E=tab["E"], B=want, K=16, S=1).L == want


def test_demo_bound_from_first_page():
    # E=8, R=4: ceil(8*3/16) = 2, the demo's worst-case button
    assert theory.theorem2_bound(4, 8) == 2


def test_global_ordinal_matches_stable_sort():
    rt = syn.zipf_bias_routing(4, 64, 2, 8, seed=3)
    d = Dims(R=4, E=8, B=2, K=2, S=64)
    q = planner.global_ordinals(rt.idx, d).reshape(-1)
    flat = rt.idx.reshape(-1)
    order = np.argsort(flat, kind="stable")
    start = np.searchsorted(flat[order], np.arange(8))
    want = np.empty_like(q)
    want[order] = np.arange(flat.size) - start[flat[order]]
    assert np.array_equal(q, want)


def test_balanced_routing_is_a_stable_counting_sort():
    R, E, K, S = 8, 64, 4, 256
    rt = syn.round_robin_routing(R, S, K, E)
    d = Dims(R=R, E=E, B=8, K=K, S=S)
    fp = _full(rt.idx, d)
    assert fp["n_fills"] == 0 and np.all(fp["slot_expert"] < 0)
    assert np.array_equal(fp["inverse"], np.argsort(rt.idx.reshape(-1), kind="stable"))


def test_single_hot_rank_chains_fills():
    # every copy goes to rank 0's experts: R-1 fills, each from a different donor
    R, E, K, S = 4, 16, 2, 64
    L = E // R
    c = np.arange(R * S * K).reshape(R, S, K)
    idx = (c % L).astype(np.int32)  # experts 0..L-1 only (rank 0)
    d = Dims(R=R, E=E, B=L, K=K, S=S)
    fp = _full(idx, d)
    assert fp["n_fills"] == R - 1
    assert fp["src"].tolist() == [-1, 0, 0, 0]


SHAPES = [  # (R, E, B, K, S) of every workload, plus small random variants
    (4, 8, 2, 2, 16), (8, 64, 8, 4, 1024), (8, 384, 48, 8, 8192),
    (64, 896, 14, 16, 1024), (3, 6, 2, 2, 8), (5, 10, 2, 3, 7),
]


@pytest.mark.parametrize("shape", SHAPES[:2] + SHAPES[4:])
@pytest.mark.parametrize("seed", range(6))
def test_theorem1_invariants_random(shape, seed):
    R, E, B, K, S = shape
    d = Dims(R=R, E=E, B=B, K=K, S=S)
    for rt in (syn.zipf_bias_routing(R, S, K, E, seed=seed),
               syn.gumbel_topk_routing(R, S, K, E, alpha=0.5 * seed, seed=seed)):
        _full(rt.idx, d)


@pytest.mark.parametrize("shape", SHAPES[2:4], ids=["pages", "k3"])
def test_theorem1_invariants_large(shape):
    R, E, B, K, S = shape
    d = Dims(R=R, E=E, B=B, K=K, S=S)
    for alpha in (0.3, 1.5):
        rt = syn.gumbel_topk_routing(R, S, K, E, alpha=alpha, seed=1)
        p = planner.build_plan(rt.idx, d)
        assert len(p.fills) <= R - 1
        assert np.all(p.cu_seqlens[:, -1] == d.C)
        assert np.all(p.n_recv <= d.L)
    _full(rt.idx, d)  # full destination check once per shape


@pytest.mark.parametrize("seed", range(4))
def test_inference_overflow_invariants(seed):
    R, E, K, S = 4, 16, 2, 64
    rt = syn.round_robin_routing(R, S, K, E, first=E // R, seed=seed)
    for B in (0, 1, 2):
        d = Dims(R=R, E=E, B=B, K=K, S=S, mode=1)
        fp = _full(rt.idx, d)
        p = fp["plan"]
        for u in range(R):
            assert len(p.overflow[u]) == max(0, p.n_recv[u] - B)


def test_routing_is_validated():
    d = Dims(R=2, E=4, B=2, K=2, S=3)
    with pytest.raises(planner.RoutingError):
        planner.check_routing(syn.bad_routing_out_of_range(2, 3, 2, 4), d)
    with pytest.raises(planner.RoutingError):
        planner.check_routing(syn.bad_routing_duplicate(2, 3, 2, 4), d)
    with pytest.raises(ValueError):
        planner.build_plan(syn.round_robin_routing(2, 3, 2, 4).idx, Dims(R=2, E=4, B=1, K=2, S=3))


def test_brute_force_tiny_adversarial_minimum_is_the_bound():
    R, E, K, S = 4, 8, 2, 16
    d = Dims(R=R, E=E, B=2, K=K, S=S)
    rt = syn.round_robin_routing(R, S, K, E, first=2)
    _, T, _ = planner.histogram(rt.idx, d)
    m, witness = theory.min_max_redundant(T, R, d.C, m_max=2)
    assert m == 2 == theory.theorem2_bound(R, E)
    assert max(planner.build_plan(rt.idx, d).n_recv) == m


@pytest.mark.parametrize("seed", range(8))
def test_brute_force_bounds_the_planner(seed):
    R, E, K, S = 3, 6, 2, 8
    d = Dims(R=R, E=E, B=2, K=K, S=S)
    rt = syn.gumbel_topk_routing(R, S, K, E, alpha=1.0 + seed * 0.5, seed=seed)
    _, T, _ = planner.histogram(rt.idx, d)
    m, _ = theory.min_max_redundant(T, R, d.C, m_max=d.L)
    got = int(max(planner.build_plan(rt.idx, d).n_recv))
    assert m is not None and m <= got <= d.L


def test_max_flow_hand_case():
    # two ranks, experts 0,1 home to rank 0 with 3+3 copies, rank 1's experts
    # empty, C = 3: rank 1 must import 3 copies; allowing expert 0 suffices.
    T = np.array([3, 3, 0, 0])
    assert not theory.feasible(T, 2, 3, [[], []])
    assert theory.feasible(T, 2, 3, [[], [0]])
    assert theory.min_max_redundant(T, 2, 3, 2)[0] == 1


def test_maxvio():
    assert theory.maxvio(np.array([2, 2, 2, 2]), 8, 4) == 0.0
    assert theory.maxvio(np.array([3, 1, 0, 0]), 4, 4) == 2.0


def test_generator_skew_agrees_with_oracle_maxvio():
    rt = syn.tune_alpha(8, 1024, 4, 64, target=1.0, seed=0)
    _, T, _ = planner.histogram(rt.idx, Dims(R=8, E=64, B=8, K=4, S=1024))
    v = theory.maxvio(T, 8 * 1024 * 4, 64)
    assert v == pytest.approx(syn.input_skew(rt.idx, 64))
    assert abs(v - 1.0) <= 0.05


def test_route_encoding_hand_case():
    case = json.load(open(os.path.join(GOLD, "hand_plans.json")))["route_cases"][0]
    R, S, K, C, owner = case["R"], case["S"], case["K"], case["C"], case["owner"]
    d = Dims(R=R, E=R, B=1, K=K, S=S)
    assert d.C == C
    dst = np.zeros((R, S, K), dtype=np.int64)
    for r in range(R):
        for s in range(S):
            dst[r, s] = r * C + s * K + np.arange(K)  # stays on its own rank
    dst[owner, 0] = [u * C + o for u, o in zip(case["dst_rank"], case["offset"])]
    enc = planner.route_encoding(dst, d)
    assert enc[owner, 0].tolist() == case["route"]
    # a token whose K entries share one rank carries its payload in entry 0 only
    assert enc[owner, 1, 0] >= 0 and np.all(enc[owner, 1, 1:] < 0)
    traffic = planner.link_traffic(dst, d, payload_bytes=7168)
    assert traffic["remote_entries"] == case["remote_entries"]
    assert traffic["remote_pairs"] == case["remote_pairs"]
    assert traffic["send_once_bytes"] == 2 * 7168 + 5 * 4
    assert traffic["per_entry_bytes"] == 5 * (7168 + 4)


@pytest.mark.parametrize("seed", range(3))
def test_route_encoding_invariants(seed):
    R, E, B, K, S = 8, 64, 8, 4, 256
    d = Dims(R=R, E=E, B=B, K=K, S=S)
    rt = syn.gumbel_topk_routing(R, S, K, E, alpha=1.0 + seed, seed=seed)
    fp = planner.full_plan(rt.idx, d)
    enc = planner.route_encoding(fp["dst"], d).reshape(-1, K)
    dst = fp["dst"].reshape(-1, K)
    for t in range(dst.shape[0]):
        ranks = dst[t] // d.C
        nonneg = enc[t] >= 0
        # exactly one payload-carrying entry per distinct destination rank, the first
        assert sorted(ranks[nonneg].tolist()) == sorted(set(ranks.tolist()))
        assert nonneg[0]
        # decoding recovers every offset
        dec = np.where(enc[t] >= 0, enc[t], -enc[t] - 1)
        assert np.array_equal(dec, dst[t] % d.C)
    tr = planner.link_traffic(fp["dst"], d, payload_bytes=2 * 64)
    assert tr["send_once_bytes"] <= tr["per_entry_bytes"]
    assert tr["remote_pairs"] <= tr["remote_entries"]


# ---- the largest-first policy --------------------------------------------------

def _min_items_covering(sizes, need):
    """Fewest items whose sizes sum to at least `need` (brute force)."""
    from itertools import combinations
    for k in range(len(sizes) + 1):
        if any(sum(c) >= need for c in combinations(sizes, k)):
            return k
    return None


@pytest.mark.parametrize("seed", range(10))
def test_largest_first_each_fill_uses_the_fewest_experts(seed):
    R, E, K, S = 4, 24, 3, 40
    d = Dims(R=R, E=E, B=E // R, K=K, S=S, policy=1)
    rt = syn.gumbel_topk_routing(R, S, K, E, alpha=1.5 + 0.2 * seed, seed=seed)
    _, T, _ = planner.histogram(rt.idx, d)
    fills, _ = planner.constructive_plan(T, d)
    # replay: before each fill, the donor's remaining copies per expert
    remaining = [int(x) for x in T]
    for f in fills:
        sizes = [remaining[e] for e in range(f.o * d.L, (f.o + 1) * d.L) if remaining[e] > 0]
        assert len(f.pieces) == _min_items_covering(sizes, f.d)
        for e, lo, hi in f.pieces:
            remaining[e] -= hi - lo
    _full(rt.idx, d)  # and Theorem 1's invariants still hold


@pytest.mark.parametrize("seed", range(8))
def test_largest_first_against_brute_force_and_constructive(seed):
    R, E, K, S = 3, 6, 2, 8
    d0 = Dims(R=R, E=E, B=2, K=K, S=S)
    d1 = Dims(R=R, E=E, B=2, K=K, S=S, policy=1)
    rt = syn.gumbel_topk_routing(R, S, K, E, alpha=1.0 + seed * 0.5, seed=seed)
    _, T, _ = planner.histogram(rt.idx, d0)
    m, _ = theory.min_max_redundant(T, R, d0.C, m_max=d0.L)
    got1 = int(max(planner.build_plan(rt.idx, d1).n_recv))
    assert m <= got1 <= d0.L


def test_largest_first_is_never_worse_in_total_over_a_sweep():
    R, E, B, K, S = 8, 64, 8, 4, 512
    tot0 = tot1 = 0
    for seed, alpha in enumerate((0.5, 1.0, 1.5, 2.0, 3.0)):
        rt = syn.gumbel_topk_routing(R, S, K, E, alpha=alpha, seed=seed)
        p0 = planner.build_plan(rt.idx, Dims(R=R, E=E, B=B, K=K, S=S))
        p1 = planner.build_plan(rt.idx, Dims(R=R, E=E, B=B, K=K, S=S, policy=1))
        assert len(p1.fills) <= R - 1 and max(p1.n_recv) <= E // R
        tot0 += int(p0.n_recv.sum())
        tot1 += int(p1.n_recv.sum())
    assert tot1 <= tot0


def test_largest_first_on_the_theorem2_case_reaches_the_bound():
    R, E, K, S = 8, 384, 8, 8192
    d = Dims(R=R, E=E, B=E // R, K=K, S=S, policy=1)
    rt = syn.round_robin_routing(R, S, K, E, first=E // R)
    p = planner.build_plan(rt.idx, d)
    # rank 0 owns nothing, so any plan gives it >= ceil(E(R-1)/R^2) = 42 experts
    assert p.n_recv[0] >= theory.theorem2_bound(R, E)
    assert max(p.n_recv) <= E // R


def test_largest_first_reaches_the_exact_minimax_on_a_seeded_sweep():
    # [Equilibrage] "La planification en ligne": the online planner is fast and
    # close to the exact optimum. Against the brute-force minimax (max-flow over
    # every choice of remote experts) on 240 skewed small instances, the
    # largest-first policy reaches the optimum every time, while the plain
    # policy is above it on a large share: a change that made the two policies
    # pair alike would fail here.
    above0 = n = 0
    for (R, E, K, S) in ((2, 6, 2, 12), (3, 6, 2, 8), (4, 8, 4, 8), (4, 12, 2, 8)):
        for seed in range(60):
            rt = syn.gumbel_topk_routing(R, S, K, E, alpha=0.5 + (seed % 12) * 0.35, seed=seed)
            d0 = Dims(R=R, E=E, B=E // R, K=K, S=S)
            _, T, _ = planner.histogram(rt.idx, d0)
            m, _ = theory.min_max_redundant(T, R, d0.C, m_max=d0.L)
            got0 = int(max(planner.build_plan(rt.idx, d0).n_recv))
            got1 = int(max(planner.build_plan(rt.idx, Dims(R=R, E=E, B=E // R, K=K, S=S,
                                                           policy=1)).n_recv))
            assert got1 == m, (R, E, K, S, seed)
            assert m <= got0 <= d0.L
            above0 += got0 > m
            n += 1
    assert n == 240 and above0 >= n // 4


def test_largest_first_is_a_heuristic_not_the_exact_minimax():
    # one instance (six ranks) where the largest-first pairing needs one more
    # redundant expert on some rank than the exact minimax: the policy is a
    # heuristic, as the pages describe their planner
    R, E, K, S = 6, 12, 2, 6
    rt = syn.gumbel_topk_routing(R, S, K, E, alpha=0.5, seed=12)
    d = Dims(R=R, E=E, B=E // R, K=K, S=S, policy=1)
    _, T, _ = planner.histogram(rt.idx, d)
    assert T.tolist() == [8, 10, 4, 3, 11, 5, 4, 10, 5, 11, 1, 0]
    m, _ = theory.min_max_redundant(T, R, d.C, m_max=1)
    assert m == 1
    assert planner.build_plan(rt.idx, d).n_recv.tolist() == [1, 1, 1, 0, 1, 2]
