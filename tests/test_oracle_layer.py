"""The layer oracle (bf16, GEMM, combine, permute, prefetch, reduce) pinned on CPU."""
import os

import numpy as np

from oracle import layer, planner
from oracle.planner import Dims
from perfectly_balanced_token_gb300 import synthetic as syn

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bits(vals):
    return layer.f32_bits_to_bf16_rne(np.asarray(vals, np.float32).view(np.uint32))


def test_bf16_rne_hand_patterns():
    rows = [ln.split() for ln in open(os.path.join(GOLD, "bf16_rne.txt"))
            if ln.strip() and not ln.startswith("#")]
    src = np.array([int(r[0], 16) for r in rows], dtype=np.uint32)
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint16)
    assert np.array_equal(layer.f32_bits_to_bf16_rne(src), want)


def test_bf16_roundtrip_exact_values():
    v = np.array([0.0, 1.0, -2.5, 0.15625, 65280.0, -1.0 / 64])
    assert np.array_equal(layer.bf16_to_f64(layer.to_bf16(v)), v)


def test_gemm_one_hot_rows_pick_weight_rows():
    # x rows one-hot on h -> Y row is row h of W_e (not a column): H != H'
    d = Dims(R=1, E=2, B=2, K=1, S=4, H=4, Hp=3)
    x = np.zeros((1, 4, 4))
    for s in range(4):
        x[0, s, (s + 1) % 4] = 1.0
    w = np.arange(2 * 4 * 3, dtype=np.float64).reshape(2, 4, 3) - 7
    idx = np.array([[[0], [1], [1], [0]]])
    out = layer.expert_outputs(layer.to_bf16(x), layer.to_bf16(w), idx, d)
    for e in (0, 1):
        cids, yb = out[e]
        for c, y in zip(cids, layer.bf16_to_f64(yb)):
            assert np.array_equal(y, w[e, (c + 1) % 4])


def test_gemm_small_integer_closed_form():
    # x all ones: Y = column sums of W (exact in bf16 for small integers)
    d = Dims(R=2, E=2, B=1, K=1, S=2, H=8, Hp=16)
    rng = np.random.default_rng(0)
    w = rng.integers(-4, 5, size=(2, 8, 16)).astype(np.float64)
    x = np.ones((2, 2, 8))
    idx = np.array([[[0], [1]], [[1], [0]]])
    out = layer.expert_outputs(layer.to_bf16(x), layer.to_bf16(w), idx, d)
    for e in (0, 1):
        for y in layer.bf16_to_f64(out[e][1]):
            assert np.array_equal(y, w[e].sum(axis=0))


def _small_case(seed=0, R=4, E=8, B=2, K=2, S=16, H=64, Hp=32, mode=0):
    d = Dims(R=R, E=E, B=B, K=K, S=S, H=H, Hp=Hp, mode=mode)
    rt = syn.zipf_bias_routing(R, S, K, E, seed=seed)
    x = syn.bf16_bits(syn.normal_bf16((R, S, H), 1.0, seed + 1))
    w = syn.bf16_bits(syn.normal_bf16((E, H, Hp), 0.02, seed + 2))
    return d, rt, x, w


def test_plan_driven_gemm_equals_per_expert_definition():
    d, rt, x, w = _small_case()
    fp = planner.full_plan(rt.idx, d)
    recv = layer.permute(x, fp["dst"], d)
    y_rows = layer.grouped_gemm_rows(recv, fp["plan"], w)
    per_e = layer.expert_outputs(x, w, rt.idx, d)
    dst = fp["dst"].reshape(-1)
    for e, (cids, yb) in per_e.items():
        assert np.array_equal(y_rows[dst[cids]], yb)


def test_permute_places_each_token_row():
    d, rt, x, _ = _small_case(seed=5)
    fp = planner.full_plan(rt.idx, d)
    recv = layer.permute(x, fp["dst"], d)
    xs = x.reshape(-1, d.H)
    for c in range(d.N):
        assert np.array_equal(recv[fp["dst"].reshape(-1)[c]], xs[c // d.K])


def test_combine_one_hot_gates_and_plan_independence():
    d, rt, x, w = _small_case(seed=2)
    fp = planner.full_plan(rt.idx, d)
    per_e = layer.expert_outputs(x, w, rt.idx, d)
    y_rows = layer.grouped_gemm_rows(layer.permute(x, fp["dst"], d), fp["plan"], w)
    gates = np.zeros((d.R, d.S, d.K), np.float32)
    gates[..., 1] = 1.0
    out = layer.combine(y_rows, fp["dst"], gates, d)
    dst = fp["dst"].reshape(d.R * d.S, d.K)
    assert np.array_equal(out, y_rows[dst[:, 1]])
    # with the routing's own gates, plan-driven == plan-free formulation
    a = layer.combine(y_rows, fp["dst"], rt.gates, d)
    b = layer.combine_from_copies(per_e, rt.gates, d)
    assert np.array_equal(a, b)


def test_combine_exact_weighted_sum():
    d = Dims(R=1, E=2, B=1, K=2, S=1, H=1, Hp=4)
    y = layer.to_bf16(np.array([[1.0, 2.0, -4.0, 8.0], [3.0, 6.0, 4.0, 0.0]]))
    out = layer.combine(y, np.array([[[1, 0]]]), np.array([[[0.25, 0.75]]]), d)
    assert np.array_equal(layer.bf16_to_f64(out[0]), [0.75 * 1 + 0.25 * 3, 0.75 * 2 + 0.25 * 6,
                                                      0.75 * -4 + 0.25 * 4, 6.0])


def test_prefetch_and_reduce_grad_conservation():
    R, E, K, S = 4, 8, 2, 16
    d = Dims(R=R, E=E, B=2, K=K, S=S, H=4, Hp=8)
    rt = syn.round_robin_routing(R, S, K, E, first=2)
    p = planner.build_plan(rt.idx, d)
    w = np.arange(E * 4 * 8, dtype=np.uint16).reshape(E, 4, 8)
    ws = layer.prefetch(w, p)
    for u in range(R):
        for j in range(d.B):
            e = p.slot_expert[u, j]
            assert np.array_equal(ws[u, j], w[e] if e >= 0 else np.zeros_like(w[0]))
    rng = np.random.default_rng(0)
    gh = rng.integers(-50, 50, size=(E, 4, 8)).astype(np.float32)
    gs = rng.integers(-50, 50, size=(R, d.B, 4, 8)).astype(np.float32)
    occupied = p.slot_expert >= 0
    gs[~occupied] = 0.0
    total = gh.astype(np.float64).sum() + gs.astype(np.float64).sum()
    want = gh.copy()
    for u in range(R):
        for j in range(d.B):
            if occupied[u, j]:
                want[p.slot_expert[u, j]] += gs[u, j]
    layer.reduce_grad(gh, gs, p)
    assert np.array_equal(gh, want)
    assert np.all(gs == 0.0)
    assert gh.astype(np.float64).sum() == total


def test_reduce_grad_leaves_unoccupied_slots_alone():
    d = Dims(R=2, E=4, B=2, K=1, S=5)
    idx = np.array([[[0], [1], [0], [0], [0]], [[0], [1], [2], [3], [0]]])
    p = planner.build_plan(idx, d)
    gh = np.ones((4, 2, 2), np.float32)
    gs = np.full((2, 2, 2, 2), 7.0, np.float32)
    layer.reduce_grad(gh, gs, p)
    assert np.all(gs[0] == 7.0)        # rank 0 holds no slots
    assert np.all(gs[1] == 0.0)        # rank 1 slots hold e1, e0: consumed
    assert np.all(gh[0] == 8.0) and np.all(gh[1] == 8.0) and np.all(gh[2:] == 1.0)
