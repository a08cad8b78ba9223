"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of an oracle module -- a wrong
tie-break, a dropped term, a wrong sign, index or offset, a transposed operand
-- installs the copy's functions in place of the real ones for the duration of
the test, and runs the pins named for it: at least one of them must fail.  A
pin that still passes on every planted mistake it is meant to catch pins
nothing.  The real oracle is restored after every case (pytest's monkeypatch).

Nothing here touches the CUDA path: the mistakes are planted in the oracle,
and the pins are the oracle's own CPU tests.
"""
import inspect
import json
import os
import types

import pytest

from oracle import layer, planner, theory
from tests import test_oracle_backward as tb
from tests import test_oracle_layer as tl
from tests import test_oracle_planner as tp

MODULES = {"planner": planner, "layer": layer, "theory": theory}
GOLD = os.path.join(os.path.dirname(__file__), "golden")
HAND = {c["name"]: c for c in json.load(open(os.path.join(GOLD, "hand_plans.json")))["cases"]}
THM2 = {c["name"]: c for c in tp.THM2["cases"]}


def _hand(*names):
    names = names or tuple(HAND)
    return [lambda n=n: tp.test_hand_worked_plans(HAND[n]) for n in names]


def _seeds(fn, seeds):
    return [lambda s=s: fn(s) for s in seeds]


# (id, module, [(text in the module, planted text)], pins)
MUTANTS = [
    # ---- planner: which copies move, in which order, from which rank ----
    ("moves-lowest-ordinals", "planner",
     [("f.pieces.append((e, left - t, left))",
       "f.pieces.append((e, migrated[e], migrated[e] + t))")],
     _hand()),
    ("ascending-expert-cursor", "planner",
     [("cursor = {h: (h + 1) * L - 1 for h in over}", "cursor = {h: h * L for h in over}"),
      ("cursor[o] = e - 1", "cursor[o] = e + 1"),
      ("assert cursor[o] >= o * L", "assert cursor[o] < (o + 1) * L")],
     _hand()),
    ("largest-id-underloaded-rank", "planner",
     [("u, o = under[0], over[0]", "u, o = under[-1], over[0]")],
     _hand("r4e4k1s4-two-under")),
    ("largest-id-overloaded-rank", "planner",
     [("u, o = under[0], over[0]", "u, o = under[0], over[-1]")],
     _hand("r4e4k1s4-two-over")),
    ("fill-size-from-donor-surplus", "planner",
     [("f = Fill(u=u, o=o, d=C - load[u])", "f = Fill(u=u, o=o, d=load[o] - C)")],
     _hand()),
    ("drained-donor-not-requeued", "planner",
     [("insort(under, o)", "pass")],
     [lambda: tp.test_theorem2_worst_case(THM2["tiny"]),
      *_seeds(lambda s: tp.test_theorem1_invariants_random((5, 10, 2, 3, 7), s), range(6))]),
    ("kept-copies-not-reduced", "planner",
     [("keep = T - migrated", "keep = T")],
     _hand()),
    ("overflow-takes-a-slot", "planner",
     [("if j < d.B:", "if j <= d.B:")],
     _hand("r2e4k1s5-infer-overflow") + _seeds(tp.test_inference_overflow_invariants, range(4))),
    ("ordinals-in-token-major-order", "planner",
     [("for e in idx.reshape(-1).tolist():", "for e in idx.transpose(1, 0, 2).reshape(-1).tolist():")],
     [tp.test_global_ordinal_matches_stable_sort]),
    ("group-rows-reversed", "planner",
     [("dst[c] = u * d.C + cu[u][g] + (q - lo)", "dst[c] = u * d.C + cu[u][g + 1] - 1 - (q - lo)")],
     _hand() + [tp.test_balanced_routing_is_a_stable_counting_sort]),
    # ---- planner: send-once route encoding and its traffic count ----
    ("route-minus-offset-without-one", "planner",
     [("out[t, k] = -off - 1 if u in seen else off", "out[t, k] = -off if u in seen else off")],
     [tp.test_route_encoding_hand_case, *_seeds(tp.test_route_encoding_invariants, range(3))]),
    ("route-rank-never-remembered", "planner",
     [("seen.add(u)", "pass")],
     [tp.test_route_encoding_hand_case]),
    ("traffic-counts-local-entries", "planner",
     [("remote = [u for u in ranks if u != r]", "remote = ranks")],
     [tp.test_route_encoding_hand_case]),
    # ---- planner: the largest-first policy ----
    ("largest-first-smallest-surplus", "planner",
     [("o = max(over, key=lambda h: (load[h] - C, -h))", "o = min(over, key=lambda h: (load[h] - C, h))")],
     _hand("r4e4k1s6-largest-first-pairing")),
    ("largest-first-smallest-deficit", "planner",
     [("u = min(under, key=lambda h: (load[h] - C, h))", "u = max(under, key=lambda h: (load[h] - C, -h))")],
     _hand("r4e4k1s6-largest-first-pairing")),
    ("largest-first-u-by-smallest-id", "planner",
     [("u = min(under, key=lambda h: (load[h] - C, h))", "u = under[0]")],
     _hand("r4e4k1s6-largest-first-pairing")),
    ("largest-first-o-by-smallest-id", "planner",
     [("o = max(over, key=lambda h: (load[h] - C, -h))", "o = over[0]")],
     _hand("r4e4k1s6-largest-first-pairing")),
    ("largest-first-deficit-ties-to-largest-id", "planner",
     [("u = min(under, key=lambda h: (load[h] - C, h))", "u = min(under, key=lambda h: (load[h] - C, -h))")],
     _hand("r4e4k1s5-largest-first-ties")),
    ("largest-first-surplus-ties-to-largest-id", "planner",
     [("o = max(over, key=lambda h: (load[h] - C, -h))", "o = max(over, key=lambda h: (load[h] - C, h))")],
     _hand("r4e4k1s5-largest-first-ties")),
    ("largest-first-expert-ties-to-lowest-id", "planner",
     [("left, e = max(cand)", "left, e = max(cand, key=lambda c: (c[0], -c[1]))")],
     _hand("r3e6k1s8-largest-first-expert-choice")),
    ("largest-first-takes-highest-id", "planner",
     [("left, e = max(cand)", "left, e = max(cand, key=lambda c: (c[0] > 0, c[1]))")],
     _seeds(tp.test_largest_first_each_fill_uses_the_fewest_experts, range(10))),
    # ---- theory ----
    ("theorem2-bound-floor", "theory",
     [("return -(-E * (R - 1) // (R * R))", "return E * (R - 1) // (R * R)")],
     [tp.test_demo_bound_from_first_page]),
    ("maxvio-without-minus-one", "theory",
     [("return float(np.max(T) / (N / E) - 1.0)", "return float(np.max(T) / (N / E))")],
     [tp.test_maxvio]),
    ("flow-rank-capacity-unbounded", "theory",
     [("cap[1 + E + r][t] = C", "cap[1 + E + r][t] = big")],
     [tp.test_max_flow_hand_case]),
    ("flow-home-edge-by-modulo", "theory",
     [("cap[1 + e][1 + E + e // L] = big", "cap[1 + e][1 + E + e % R] = big")],
     [tp.test_max_flow_hand_case, tp.test_brute_force_tiny_adversarial_minimum_is_the_bound]),
    # ---- layer: bf16 rounding ----
    ("bf16-truncation", "layer",
     [("rounded = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)", "rounded = u >> np.uint32(16)")],
     [tl.test_bf16_rne_hand_patterns]),
    ("bf16-ties-away-from-zero", "layer",
     [("(u + np.uint32(0x7FFF) + lsb)", "(u + np.uint32(0x8000))")],
     [tl.test_bf16_rne_hand_patterns]),
    ("bf16-nan-not-quieted", "layer",
     [("nan_bits = (u >> np.uint32(16)) | np.uint32(0x0040)", "nan_bits = u >> np.uint32(16)")],
     [tl.test_bf16_rne_hand_patterns]),
    # ---- layer: GEMM, permute, combine, prefetch, reduce_grad ----
    ("weight-read-transposed", "layer",
     [("y = a @ bf16_to_f64(w)", "y = a @ bf16_to_f64(w).reshape(d.Hp, d.H).T")],
     [tl.test_gemm_one_hot_rows_pick_weight_rows]),
    ("slot-weight-by-slot-index", "layer",
     [("w = w_home_bits[plan.slot_expert[u, g - d.E]]", "w = w_home_bits[g - d.E]")],
     [tl.test_plan_driven_gemm_equals_per_expert_definition]),
    ("permute-copy-to-token-k-major", "layer",
     [("tok = np.arange(d.N) // d.K\n    recv[", "tok = np.arange(d.N) % (d.R * d.S)\n    recv[")],
     [tl.test_permute_places_each_token_row]),
    ("combine-drops-first-term", "layer",
     [("    for k in range(d.K):\n        acc += g2[tok, k]", "    for k in range(1, d.K):\n        acc += g2[tok, k]")],
     [tl.test_combine_exact_weighted_sum]),
    ("combine-gates-reversed", "layer",
     [("acc += g2[tok, k][:, None]", "acc += g2[tok, d.K - 1 - k][:, None]")],
     [tl.test_combine_exact_weighted_sum]),
    ("prefetch-row-by-slot-index", "layer",
     [("out[u, j] = w_home_bits[e]", "out[u, j] = w_home_bits[j]")],
     [tl.test_prefetch_and_reduce_grad_conservation]),
    ("slots-not-zeroed", "layer",
     [("g_slot[u, j] = 0.0", "pass")],
     [tl.test_prefetch_and_reduce_grad_conservation]),
    ("every-slot-reduced-into-every-expert", "layer",
     [("if plan.slot_expert[u, j] == e:", "if plan.slot_expert[u, j] >= 0:")],
     [tl.test_prefetch_and_reduce_grad_conservation]),
    # ---- layer: backward ----
    ("combine-backward-drops-gate", "layer",
     [("dy = to_bf16(g[:, None] * dout[tok])", "dy = to_bf16(dout[tok])")],
     [tb.test_combine_backward_closed_forms]),
    ("gate-gradient-sign", "layer",
     [("dg = np.einsum(", "dg = -np.einsum(")],
     [tb.test_combine_backward_closed_forms]),
    ("input-gradient-weight-not-transposed", "layer",
     [("drecv = to_bf16(dyc[cids] @ w.T)", "drecv = to_bf16(dyc[cids] @ w.reshape(d.Hp, d.H))")],
     [tb.test_one_hot_dy_picks_weight_columns]),
    ("weight-gradient-token-index", "layer",
     [("dw = xs[cids // d.K].T @ dyc[cids]", "dw = xs[cids % (d.R * d.S)].T @ dyc[cids]")],
     [tb.test_adjoint_identity_exact_on_small_integers]),
    ("dispatch-backward-drops-a-copy", "layer",
     [("return to_bf16(r.sum(axis=1))", "return to_bf16(r[:, 1:].sum(axis=1))")],
     [tb.test_dispatch_backward_sums_copies]),
    ("group-gradient-rows-without-rank-offset", "layer",
     [("rows = set(range(u * d.C + a0, u * d.C + a1))", "rows = set(range(a0, a1))")],
     [lambda: tb.test_grouped_weight_gradient_reduces_to_the_dense_one(0)]),
    ("row-range-gradient-without-rank-offset", "layer",
     [("rows = slice(u * d.C + a0, u * d.C + a1)", "rows = slice(a0, a1)")],
     [tb.test_row_range_weight_gradient_matches_token_form]),
]


def _plant(monkeypatch, modname, edits):
    """Install the module's functions, recompiled from its source with `edits`."""
    mod = MODULES[modname]
    src = inspect.getsource(mod)
    for old, new in edits:
        assert src.count(old) == 1, f"{modname}: the text to mutate is not unique: {old!r}"
        src = src.replace(old, new)
    ns = {"__name__": mod.__name__, "__package__": "oracle"}
    exec(compile(src, f"<{modname} with a planted mistake>", "exec"), ns)
    for name, obj in ns.items():
        if isinstance(obj, types.FunctionType) and obj.__module__ == mod.__name__:
            monkeypatch.setattr(mod, name, obj)


def _first_failure(pins):
    for pin in pins:
        try:
            pin()
        except Exception as exc:  # an assertion, or the mistake breaking a shape or index
            return exc
    return None


@pytest.mark.parametrize("mid,modname,edits,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(monkeypatch, mid, modname, edits, pins):
    _plant(monkeypatch, modname, edits)
    assert _first_failure(pins) is not None, f"no pin caught the planted mistake {mid}"


def test_unplanted_copy_passes_the_same_pins(monkeypatch):
    # the recompiled copy itself (no edit) is not what makes the pins fail
    for modname in MODULES:
        _plant(monkeypatch, modname, [])
    for _, _, _, pins in MUTANTS:
        assert _first_failure(pins) is None
