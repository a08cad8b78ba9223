"""The backward oracle pinned by closed forms and the adjoint identity (CPU)."""
import numpy as np
import pytest

from oracle import layer, planner
from oracle.planner import Dims
from perfectly_balanced_token_gb300 import synthetic as syn


def _ints(rng, shape, lo=-2, hi=3):
    return rng.integers(lo, hi, size=shape).astype(np.float64)


def test_one_hot_dy_picks_weight_columns():
    # forward: one-hot x picks a ROW of W; backward: one-hot dY picks a COLUMN
    d = Dims(R=1, E=1, B=1, K=1, S=3, H=4, Hp=5)
    w = np.arange(20, dtype=np.float64).reshape(1, 4, 5) - 9
    dy = np.zeros((3, 5))
    for s in range(3):
        dy[s, (2 * s + 1) % 5] = 1.0
    out = layer.expert_backward(layer.to_bf16(np.zeros((1, 3, 4))), layer.to_bf16(w),
                                np.zeros((1, 3, 1), dtype=np.int64), layer.to_bf16(dy), d)
    cids, drecv, _ = out[0]
    for c, row in zip(cids, layer.bf16_to_f64(drecv)):
        assert np.array_equal(row, w[0, :, (2 * c + 1) % 5])


def test_single_copy_weight_gradient_is_an_outer_product():
    d = Dims(R=1, E=2, B=2, K=1, S=2, H=3, Hp=4)
    x = np.array([[[1.0, -2.0, 3.0], [0.0, 1.0, 0.0]]])
    dy = np.array([[2.0, 0.0, -1.0, 1.0], [1.0, 1.0, 1.0, 1.0]])
    idx = np.array([[[0], [1]]])
    out = layer.expert_backward(layer.to_bf16(x), layer.to_bf16(np.ones((2, 3, 4))), idx,
                                layer.to_bf16(dy), d)
    assert np.array_equal(out[0][2], np.outer(x[0, 0], dy[0]))
    assert np.array_equal(out[1][2], np.outer(x[0, 1], dy[1]))


def test_adjoint_identity_exact_on_small_integers():
    # <dY, X W> = <X^T dY, W> = <dY W^T, X>, exact for small integers
    rng = np.random.default_rng(0)
    d = Dims(R=2, E=4, B=2, K=2, S=6, H=8, Hp=6)
    rt = syn.round_robin_routing(d.R, d.S, d.K, d.E, first=0)
    x = _ints(rng, (d.R, d.S, d.H), -1, 2)
    w = _ints(rng, (d.E, d.H, d.Hp), -1, 2)
    dy = _ints(rng, (d.N, d.Hp), -1, 2)
    xb, wb, dyb = layer.to_bf16(x), layer.to_bf16(w), layer.to_bf16(dy)
    fwd = layer.expert_outputs(xb, wb, rt.idx, d)
    bwd = layer.expert_backward(xb, wb, rt.idx, dyb, d)
    lhs = sum(np.sum(layer.bf16_to_f64(fwd[e][1]) * dy[fwd[e][0]]) for e in range(d.E))
    mid = sum(np.sum(bwd[e][2] * w[e]) for e in range(d.E))
    xs = x.reshape(-1, d.H)
    rhs = sum(np.sum(layer.bf16_to_f64(bwd[e][1]) * xs[bwd[e][0] // d.K]) for e in range(d.E))
    assert lhs == mid == rhs


def test_combine_backward_closed_forms():
    d = Dims(R=1, E=2, B=1, K=2, S=1, H=1, Hp=3)
    y = layer.to_bf16(np.array([[1.0, 2.0, 3.0], [4.0, 0.0, -1.0]]))
    dout = layer.to_bf16(np.array([[1.0, -1.0, 2.0]]))
    dy, dg = layer.combine_backward(y, dout, np.array([[[0.5, 0.25]]]), d)
    assert np.array_equal(layer.bf16_to_f64(dy), [[0.5, -0.5, 1.0], [0.25, -0.25, 0.5]])
    assert np.array_equal(dg.reshape(-1), [1 - 2 + 6, 4 + 0 - 2])


def test_dispatch_backward_sums_copies():
    d = Dims(R=1, E=2, B=1, K=2, S=2, H=2, Hp=1)
    r = layer.to_bf16(np.array([[1.0, 2.0], [3.0, -4.0], [0.5, 0.5], [0.25, 1.0]]))
    assert np.array_equal(layer.bf16_to_f64(layer.dispatch_backward(r, d)),
                          [[4.0, -2.0], [0.75, 1.5]])


@pytest.mark.parametrize("policy", [0, 1])
def test_grouped_weight_gradient_reduces_to_the_dense_one(policy):
    # per-group partial sums (what the grouped GEMM writes into home rows and
    # slots) fold back, via the slot table, into the plan-free per-expert sums
    d = Dims(R=4, E=8, B=2, K=2, S=16, H=6, Hp=5, policy=policy)
    rt = syn.zipf_bias_routing(d.R, d.S, d.K, d.E, seed=2)
    rng = np.random.default_rng(1)
    xb = layer.to_bf16(_ints(rng, (d.R, d.S, d.H)))
    dyb = layer.to_bf16(_ints(rng, (d.N, d.Hp)))
    fp = planner.full_plan(rt.idx, d)
    parts = layer.dw_by_group(xb, rt.idx, dyb, fp["plan"], fp["dst"])
    dense = layer.expert_backward(xb, layer.to_bf16(np.zeros((d.E, d.H, d.Hp))), rt.idx, dyb, d)
    folded = {e: np.zeros((d.H, d.Hp)) for e in range(d.E)}
    for (u, g), dw in parts.items():
        e = g if g < d.E else int(fp["slot_expert"][u, g - d.E])
        folded[e] += dw
    for e in range(d.E):
        assert np.array_equal(folded[e], dense[e][2])


def test_row_range_weight_gradient_matches_token_form():
    d = Dims(R=4, E=8, B=2, K=2, S=16, H=6, Hp=5)
    rt = syn.zipf_bias_routing(d.R, d.S, d.K, d.E, seed=4)
    rng = np.random.default_rng(3)
    xb = layer.to_bf16(_ints(rng, (d.R, d.S, d.H)))
    dyb = layer.to_bf16(_ints(rng, (d.N, d.Hp)))
    fp = planner.full_plan(rt.idx, d)
    dy_rows = np.zeros((d.N, d.Hp), dtype=np.uint16)
    dy_rows[fp["dst"].reshape(-1)] = dyb
    a = layer.grouped_gemm_dw_rows(layer.permute(xb, fp["dst"], d), dy_rows, fp["plan"])
    b = layer.dw_by_group(xb, rt.idx, dyb, fp["plan"], fp["dst"])
    assert a.keys() == b.keys()
    for k in a:
        assert np.array_equal(a[k], b[k])
