"""CUDA path vs CPU oracle, element by element, through the C ABI.

Plans, cu_seqlens, destinations and the inverse permutation must be
bit-exact; the dispatch buffer and the prefetched slots are byte copies and
must be bit-exact; GEMM and combine outputs must be within 1e-2 absolute +
2e-2 relative of the oracle (bf16 values, fp32 accumulation); reduce_grad
adds fp32 values in the oracle's order and must be bit-exact.
"""
import numpy as np
import pytest
import torch

import perfectly_balanced_token_gb300 as mx
from oracle import layer as olayer
from oracle import planner as oplanner
from perfectly_balanced_token_gb300 import synthetic as syn
from tests import gpu_harness as gh
from tests.invariants import check_plan_arrays

pytestmark = pytest.mark.gpu

W = syn.Workload


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gh.ensure_library()


# (workload, routing recipe) covering several GEMM column tiles (BN 64/128/256),
# ragged row tails, tiles straddling ranks, K=1, R=1, E=R, inference overflow
CASES = [
    ("tiny", syn.TINY, lambda w: syn.routing_for(w)),
    ("tiny-adversarial", syn.TINY, lambda w: syn.round_robin_routing(w.R, w.S, w.K, w.E, first=2)),
    ("r8e64-maxvio0", syn.SMALL, lambda w: syn.routing_for(w, 0.0)),
    ("r8e64-maxvio1", syn.SMALL, lambda w: syn.routing_for(w, 1.0)),
    ("r8e64-maxvio5", syn.SMALL, lambda w: syn.routing_for(w, 5.0)),
    ("r1-single-rank", W("r1", R=1, E=4, B=4, K=2, S=37, H=64, Hp=64),
     lambda w: syn.zipf_bias_routing(w.R, w.S, w.K, w.E, seed=4)),
    ("r4-e4-k1-bn64", W("e=r", R=4, E=4, B=1, K=1, S=300, H=128, Hp=192),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=2.0, seed=5)),
    ("r5-e20-ragged", W("ragged", R=5, E=20, B=4, K=3, S=171, H=192, Hp=320),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.3, seed=6)),
    ("infer-b1-overflow", W("infer1", R=4, E=16, B=1, K=2, S=200, H=128, Hp=256, mode=1),
     lambda w: syn.round_robin_routing(w.R, w.S, w.K, w.E, first=4)),
    ("infer-b0", W("infer0", R=4, E=16, B=0, K=2, S=96, H=64, Hp=128, mode=1),
     lambda w: syn.round_robin_routing(w.R, w.S, w.K, w.E, first=4)),
    ("hot-rank-chain", W("chain", R=8, E=32, B=4, K=2, S=256, H=128, Hp=256),
     lambda w: syn.Routing(((np.arange(w.R * w.S * w.K).reshape(w.R, w.S, w.K)) % 4).astype(np.int32),
                           np.full((w.R, w.S, w.K), 0.5, np.float32))),
    # C*R/E >= 4096: the GEMM runs 256-row work tiles (two accumulators)
    ("m256-bn256", W("m256", R=2, E=4, B=2, K=2, S=4096, H=128, Hp=256),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.5, seed=7)),
    ("m256-bn64-ragged", W("m256b", R=4, E=8, B=2, K=2, S=8192, H=64, Hp=192),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=2.5, seed=8)),
    ("m256-infer-b0", W("m256i", R=2, E=4, B=0, K=1, S=9000, H=64, Hp=128, mode=1),
     lambda w: syn.round_robin_routing(w.R, w.S, w.K, w.E, first=2)),
    # several 256-wide column tiles with ragged groups of a few 128-row tiles,
    # groups mostly under one tile, and inference overflow
    ("bn256-ragged", W("bn256r", R=4, E=12, B=3, K=3, S=700, H=192, Hp=512),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.2, seed=9)),
    ("bn256-small-groups", W("bn256s", R=8, E=64, B=8, K=2, S=200, H=64, Hp=512),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=0.8, seed=10)),
    ("bn256-infer-overflow", W("bn256i", R=4, E=16, B=1, K=2, S=300, H=128, Hp=1024, mode=1),
     lambda w: syn.round_robin_routing(w.R, w.S, w.K, w.E, first=4)),
    # the small recipe's literal form, raw Zipf samples as the bias: every
    # token on the same two experts
    ("tiny-raw-zipf-bias", syn.TINY, lambda w: syn.zipf_sample_bias_routing(w.R, w.S, w.K, w.E, 0)),
]


@pytest.mark.parametrize("name,w,mk", CASES, ids=[c[0] for c in CASES])
def test_layer_parity(name, w, mk):
    _layer_parity(name, w, mk(w), 0)


# the GEMM work-tile height fixed either way (the plan and every output must
# not depend on it)
FIXED_ROWS_CASES = [c for c in CASES if c[0] in (
    "r8e64-maxvio1", "r5-e20-ragged", "infer-b1-overflow", "m256-bn256", "m256-bn64-ragged",
    "bn256-ragged")]


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("name,w,mk", FIXED_ROWS_CASES, ids=[c[0] for c in FIXED_ROWS_CASES])
def test_layer_parity_fixed_tile_rows(name, w, mk, rows):
    run = _layer_parity(name, w, mk(w), rows)
    assert int(run.ws.tables()["counters"][7]) == rows


def _cost_model():
    """Coefficients of the GEMM tile-height cost model, read from its header."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(mx.__file__), "csrc", "gemm_cost.cuh")).read()
    return {k: float(v) for k, v in re.findall(r"constexpr float (kCost\w+) = ([-0-9.e+]+)f;", src)}


@pytest.mark.parametrize("name,w,mk", CASES, ids=[c[0] for c in CASES])
def test_tile_rows_follow_the_cost_model(name, w, mk):
    """With the height left to the plan, the planner's choice equals the cost
    model evaluated on the plan's own group sizes (from cu_seqlens)."""
    rt = mk(w)
    run = gh.Run(w, rt)
    tabs = run.plan()
    rows = np.diff(tabs["cu_seqlens"].astype(np.int64), axis=1).reshape(-1)
    rows = rows[rows > 0]
    rem = rows % 256
    n128 = np.sum((rows + 127) // 128)
    n256f = np.sum(rows // 256 + (rem > 128))
    n256h = np.sum((rem > 0) & (rem <= 128))
    c = _cost_model()
    waves = float(n128) * (w.Hp / 256.0) / 152.0
    t128 = c["kCostA128"] * n128 + c["kCostG128"] * rows.size + c["kCostW128"] * n128 * waves
    t256 = (c["kCostA256Full"] * n256f + c["kCostA256Half"] * n256h + c["kCostG256"] * rows.size
            + c["kCostW256"] * n256f * waves)
    want = 256 if t256 < t128 else 128
    if abs(float(t256) - float(t128)) <= 1e-4 * float(t128):  # a tie up to rounding: either
        want = int(tabs["counters"][7])
    assert int(tabs["counters"][7]) == want
    assert int(tabs["counters"][1]) == (n128 if want == 128 else n256f + n256h)


def _layer_parity(name, w, rt, gemm_rows):
    od = gh.odims(w)
    fp = oplanner.full_plan(rt.idx, od)
    run = gh.Run(w, rt, gemm_rows=gemm_rows)
    run.forward()

    # plan: bit-exact, and Theorem 1 invariants on the GPU's own tables
    tabs = run.ws.tables()
    gh.compare_plan(tabs, fp, od)
    check_plan_arrays(rt.idx, w.R, w.E, w.B, w.K, w.S, w.mode, T=tabs["T"],
                      n_fills=int(tabs["counters"][0]), fills=tabs["fills"], keep=tabs["keep"],
                      slot_expert=tabs["slot_expert"], n_recv=tabs["n_recv"], src=tabs["src"],
                      cu_seqlens=tabs["cu_seqlens"], dst=tabs["dst"], inverse=tabs["inverse"],
                      gidx=tabs["gidx"])

    x_bits = gh.host_bits(run.x)
    w_bits = gh.host_bits(run.w_home)
    # dispatch: byte-exact copy of every token row to every destination
    recv_want = olayer.permute(x_bits, fp["dst"], od)
    assert np.array_equal(gh.host_bits(run.recv).reshape(w.N, w.H), recv_want)
    # prefetch: occupied slots hold their expert's weights; empty slots untouched
    if w.B:
        ws = gh.host_bits(run.w_slot).reshape(w.R, w.B, w.H, w.Hp)
        want = olayer.prefetch(w_bits, fp["plan"])
        occ = fp["slot_expert"] >= 0
        assert np.array_equal(ws[occ], want[occ])
        assert np.all(ws[~occ] == 0x7F7F)
    # GEMM: each copy's output row against the per-expert definition
    per_e = olayer.expert_outputs(x_bits, w_bits, rt.idx, od)
    y = gh.bf16_to_np(run.y).reshape(w.N, w.Hp)
    dst = fp["dst"].reshape(-1)
    for e, (cids, yb) in per_e.items():
        if cids.size:
            gh.assert_close(y[dst[cids]], gh.bits_to_np(yb), f"{name} Y expert {e}")
    # combine: against the plan-free definition
    out_want = olayer.combine_from_copies(per_e, rt.gates, od)
    gh.assert_close(gh.bf16_to_np(run.out).reshape(w.R * w.S, w.Hp), gh.bits_to_np(out_want),
                    f"{name} combine")
    run.check_all_guards()
    return run


# the largest sizes the planner accepts: E = 4096 (its shared-memory
# histograms), R = 1024 (the most ranks the parallel-fill path takes) and
# R = 2048 (past it: the one-warp fill loop), each under both planner policies
MAX_CASES = [
    ("max-e4096", W("maxE", R=8, E=4096, B=512, K=8, S=256, H=64, Hp=64),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.2, seed=14)),
    ("max-r1024", W("maxR1k", R=1024, E=4096, B=4, K=2, S=8, H=64, Hp=64),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.5, seed=15)),
    ("max-r2048", W("maxR2k", R=2048, E=4096, B=2, K=2, S=4, H=64, Hp=64),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.5, seed=16)),
]


@pytest.mark.parametrize("policy", [0, 1])
@pytest.mark.parametrize("name,w,mk", MAX_CASES, ids=[c[0] for c in MAX_CASES])
def test_maximum_sizes(name, w, mk, policy):
    """Plan tables and route entries bit-exact, dispatch byte-exact, GEMM and
    combine within tolerance, at the planner's size limits."""
    rt = mk(w)
    od = gh.odims(w, policy)
    fp = oplanner.full_plan(rt.idx, od)
    assert fp["n_fills"] > 0
    run = gh.Run(w, rt, policy=policy)
    run.forward()
    tabs = run.ws.tables()
    gh.compare_plan(tabs, fp, od)
    assert np.array_equal(tabs["route"], oplanner.route_encoding(fp["dst"], od))
    x_bits, w_bits = gh.host_bits(run.x), gh.host_bits(run.w_home)
    assert np.array_equal(gh.host_bits(run.recv).reshape(w.N, w.H),
                          olayer.permute(x_bits, fp["dst"], od))
    per_e = olayer.expert_outputs(x_bits, w_bits, rt.idx, od)
    y = gh.bf16_to_np(run.y).reshape(w.N, w.Hp)
    dst = fp["dst"].reshape(-1)
    for e, (cids, yb) in per_e.items():
        if cids.size:
            gh.assert_close(y[dst[cids]], gh.bits_to_np(yb), f"{name} Y expert {e}")
    out_want = olayer.combine_from_copies(per_e, rt.gates, od)
    gh.assert_close(gh.bf16_to_np(run.out).reshape(w.R * w.S, w.Hp), gh.bits_to_np(out_want),
                    f"{name} combine")
    run.check_all_guards()


@pytest.mark.parametrize("name,w,mk", CASES[:6], ids=[c[0] for c in CASES[:6]])
def test_gemm_isolated_synthetic_rows(name, w, mk):
    """GEMM on a synthetic receive buffer (not produced by dispatch)."""
    rt = mk(w)
    od = gh.odims(w)
    fp = oplanner.full_plan(rt.idx, od)
    run = gh.Run(w, rt)
    run.plan()
    recv = syn.normal_bf16((w.N, w.H), 1.0, 77).cuda()
    mx.moonep_prefetch_weights(run.d, run.ws.buf, run.w_home, run.w_slot)
    mx.moonep_grouped_gemm(run.d, run.ws.buf, recv.view(-1), run.w_home, run.w_slot, run.y)
    want = olayer.grouped_gemm_rows(gh.host_bits(recv), fp["plan"], gh.host_bits(run.w_home))
    gh.assert_close(gh.bf16_to_np(run.y).reshape(w.N, w.Hp), gh.bits_to_np(want), f"{name} gemm")


@pytest.mark.parametrize("name,w,mk", CASES[:6], ids=[c[0] for c in CASES[:6]])
def test_combine_isolated_synthetic_outputs(name, w, mk):
    rt = mk(w)
    od = gh.odims(w)
    fp = oplanner.full_plan(rt.idx, od)
    run = gh.Run(w, rt)
    run.plan()
    y = syn.normal_bf16((w.N, w.Hp), 1.0, 78).cuda()
    mx.moonep_combine(run.d, run.ws.buf, y.view(-1), run.gates, run.out)
    want = olayer.combine(gh.host_bits(y), fp["dst"], rt.gates, od)
    gh.assert_close(gh.bf16_to_np(run.out).reshape(w.R * w.S, w.Hp), gh.bits_to_np(want),
                    f"{name} combine")


@pytest.mark.parametrize("name,w,mk", [c for c in CASES if c[1].B > 0],
                         ids=[c[0] for c in CASES if c[1].B > 0])
def test_reduce_grad_parity(name, w, mk):
    rt = mk(w)
    od = gh.odims(w)
    fp = oplanner.full_plan(rt.idx, od)
    run = gh.Run(w, rt)
    run.plan()
    hh = w.H * w.Hp
    g_home = syn.normal_f32((w.E, w.H, w.Hp), 1.0, 90).cuda()
    g_slot = syn.normal_f32((w.R, w.B, w.H, w.Hp), 1.0, 91).cuda()
    occ = torch.from_numpy(fp["slot_expert"] >= 0).cuda()
    g_slot[~occ] = 7.0  # sentinel: unoccupied slots must stay untouched
    gh_host, gs_host = g_home.cpu().numpy().copy(), g_slot.cpu().numpy().copy()
    mx.moonep_reduce_grad(run.d, run.ws.buf, g_home.view(-1), g_slot.view(-1))
    olayer.reduce_grad(gh_host, gs_host, fp["plan"])
    assert np.array_equal(g_home.cpu().numpy(), gh_host)
    assert np.array_equal(g_slot.cpu().numpy(), gs_host)
    assert bool((g_slot[occ] == 0).all()) and bool((g_slot[~occ] == 7.0).all())
    assert hh > 0


def test_determinism_two_runs():
    w = syn.SMALL
    rt = syn.routing_for(w, 5.0)
    a, b = gh.Run(w, rt), gh.Run(w, rt)
    a.forward()
    b.forward()
    # every table is identical; the workspace's tail (the GEMMs' tensor-map
    # copies) holds the addresses of each run's own buffers
    tables = a.ws.buf.numel() - mx.GEMM_SCRATCH_BYTES
    assert tables > 0 and torch.equal(a.ws.buf[:tables], b.ws.buf[:tables])
    assert torch.equal(a.y, b.y) and torch.equal(a.out, b.out)


def test_workspace_reuse_across_routings():
    """A second plan in the same workspace fully replaces the first."""
    w = syn.SMALL
    r1, r2 = syn.routing_for(w, 5.0), syn.routing_for(w, 0.0)
    run = gh.Run(w, r1)
    run.plan()
    run.idx.copy_(torch.from_numpy(r2.idx))
    tabs = run.plan()
    gh.compare_plan(tabs, oplanner.full_plan(r2.idx, gh.odims(w)), gh.odims(w))


@pytest.mark.parametrize("bad", ["range", "duplicate"])
def test_bad_routing_sets_status_and_writes_nothing(bad):
    w = syn.TINY
    f = syn.bad_routing_out_of_range if bad == "range" else syn.bad_routing_duplicate
    rt = syn.Routing(f(w.R, w.S, w.K, w.E), np.full((w.R, w.S, w.K), 0.5, np.float32))
    run = gh.Run(w, rt)
    run.forward()  # every call after the plan sees the status and returns
    st = mx.moonep_read_status(run.d, run.ws.buf)
    assert st & mx._lib.ERR_ROUTING
    for t in (run.recv, run.y, run.out):
        assert bool((t.view(torch.int16) == 0x7F7F).all())
    if w.B:
        assert bool((run.w_slot.view(torch.int16) == 0x7F7F).all())


@pytest.mark.parametrize("name,w,mk", CASES, ids=[c[0] for c in CASES])
def test_send_once_route_and_dispatch(name, w, mk):
    """Route entries and link counters bit-exact with the oracle's encoding;
    the two-pass send-once dispatch fills recv exactly like the fused one and
    delivers every entry's weight to its row."""
    rt = mk(w)
    od = gh.odims(w)
    fp = oplanner.full_plan(rt.idx, od)
    run = gh.Run(w, rt)
    tabs = run.plan()
    assert np.array_equal(tabs["route"], oplanner.route_encoding(fp["dst"], od))
    traffic = oplanner.link_traffic(fp["dst"], od, payload_bytes=2 * w.H)
    assert int(tabs["counters"][4]) == traffic["remote_entries"]
    assert int(tabs["counters"][5]) == traffic["remote_pairs"]
    recv_w = torch.full((w.N,), -1.0, dtype=torch.float32, device="cuda")
    mx.moonep_dispatch_send_once(run.d, run.ws.buf, run.x, run.gates, run.recv, recv_w)
    torch.cuda.synchronize()
    want = olayer.permute(gh.host_bits(run.x), fp["dst"], od)
    assert np.array_equal(gh.host_bits(run.recv).reshape(w.N, w.H), want)
    got_w = recv_w.cpu().numpy()
    assert np.array_equal(got_w[fp["dst"].reshape(-1)], rt.gates.reshape(-1))
    run.check_all_guards()


@pytest.mark.parametrize("name,w,mk", CASES, ids=[c[0] for c in CASES])
def test_largest_first_policy_parity(name, w, mk):
    """Planner policy 1 (largest first): tables bit-exact with the oracle's,
    Theorem 1 invariants on the GPU's own tables, and the layer outputs still
    equal the plan-free definitions."""
    rt = mk(w)
    od = gh.odims(w, policy=1)
    fp = oplanner.full_plan(rt.idx, od)
    run = gh.Run(w, rt, policy=1)
    run.forward()
    tabs = run.ws.tables()
    gh.compare_plan(tabs, fp, od)
    check_plan_arrays(rt.idx, w.R, w.E, w.B, w.K, w.S, w.mode, T=tabs["T"],
                      n_fills=int(tabs["counters"][0]), fills=tabs["fills"], keep=tabs["keep"],
                      slot_expert=tabs["slot_expert"], n_recv=tabs["n_recv"], src=tabs["src"],
                      cu_seqlens=tabs["cu_seqlens"], dst=tabs["dst"], inverse=tabs["inverse"],
                      gidx=tabs["gidx"])
    x_bits, w_bits = gh.host_bits(run.x), gh.host_bits(run.w_home)
    per_e = olayer.expert_outputs(x_bits, w_bits, rt.idx, od)
    out_want = olayer.combine_from_copies(per_e, rt.gates, od)
    gh.assert_close(gh.bf16_to_np(run.out).reshape(w.R * w.S, w.Hp), gh.bits_to_np(out_want),
                    f"{name} combine (policy 1)")
    run.check_all_guards()


@pytest.mark.parametrize("rows", [128, 256])
def test_gemm_launches_repeated_on_one_plan(rows):
    """The GEMM kernels claim their work items from counters in the plan
    workspace, which each launch's last CTA resets for the next: repeated
    launches on one plan compute the same output, and two weight-gradient
    launches add exactly twice."""
    w = syn.SMALL
    rt = syn.routing_for(w, 5.0)
    od = gh.odims(w)
    fp = oplanner.full_plan(rt.idx, od)
    run = gh.Run(w, rt, gemm_rows=rows)
    run.plan()
    mx.moonep_prefetch_weights(run.d, run.ws.buf, run.w_home, run.w_slot)
    recv = syn.normal_bf16((w.N, w.H), 1.0, 77).cuda()
    outs = []
    for _ in range(3):
        run.y.zero_()
        mx.moonep_grouped_gemm(run.d, run.ws.buf, recv.view(-1), run.w_home, run.w_slot, run.y)
        outs.append(run.y.clone())
    assert mx.moonep_read_status(run.d, run.ws.buf) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    want = olayer.grouped_gemm_rows(gh.host_bits(recv), fp["plan"], gh.host_bits(run.w_home))
    gh.assert_close(gh.bf16_to_np(outs[2]).reshape(w.N, w.Hp), gh.bits_to_np(want), "repeated gemm")
    # the input gradient runs the same kernels, claiming from the same counters
    dy = syn.normal_bf16((w.N, w.Hp), 1.0, 78).cuda()
    drecv = [torch.zeros(w.N * w.H, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    for dr in drecv:
        mx.moonep_grouped_gemm_dx(run.d, run.ws.buf, dy.view(-1), run.w_home, run.w_slot, dr)
    assert torch.equal(drecv[0], drecv[1])
    # weight gradient twice into zeroed gradients: exactly twice one launch (x + x is exact)
    g1 = [torch.zeros(n, dtype=torch.float32, device="cuda")
          for n in (w.E * w.H * w.Hp, w.R * w.B * w.H * w.Hp)]
    g2 = [torch.zeros_like(t) for t in g1]
    mx.moonep_grouped_gemm_dw(run.d, run.ws.buf, recv.view(-1), dy.view(-1), g1[0], g1[1])
    for _ in range(2):
        mx.moonep_grouped_gemm_dw(run.d, run.ws.buf, recv.view(-1), dy.view(-1), g2[0], g2[1])
    assert mx.moonep_read_status(run.d, run.ws.buf) == 0
    assert torch.equal(g2[0], 2 * g1[0]) and torch.equal(g2[1], 2 * g1[1])
    assert bool(g1[0].abs().sum() > 0)
