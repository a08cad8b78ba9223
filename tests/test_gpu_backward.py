"""Backward of the layer on the GPU vs the oracle, through the C ABI.

Each kernel is checked in isolation on synthetic inputs (combine backward,
input-gradient GEMM, weight-gradient GEMM, dispatch backward), then the whole
training step is checked against plan-free definitions: after
moonep_grouped_gemm_dw and moonep_reduce_grad every home gradient row equals
its initial value plus X_e^T dY_e over all copies of e, whatever the plan, and
the token gradient equals sum_k bf16(dY_k W_k^T).  Tolerance 1e-2 + 2e-2|x|.
"""
import numpy as np
import pytest
import torch

import perfectly_balanced_token_gb300 as mx
from oracle import layer as olayer
from oracle import planner as oplanner
from perfectly_balanced_token_gb300 import synthetic as syn
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu
W = syn.Workload

CASES = [  # H % 128 == 0 for the weight gradient
    ("r8e64-maxvio1", syn.SMALL, lambda w: syn.routing_for(w, 1.0), 0),
    ("r8e64-maxvio5-largest-first", syn.SMALL, lambda w: syn.routing_for(w, 5.0), 1),
    ("r4-e4-k1-bn64", W("e=r", R=4, E=4, B=1, K=1, S=300, H=128, Hp=192),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=2.0, seed=5), 0),
    ("hot-rank-chain", W("chain", R=8, E=32, B=4, K=2, S=256, H=128, Hp=256),
     lambda w: syn.Routing(((np.arange(w.R * w.S * w.K).reshape(w.R, w.S, w.K)) % 4).astype(np.int32),
                           np.full((w.R, w.S, w.K), 0.5, np.float32)), 0),
    ("m256-bn256", W("m256", R=2, E=4, B=2, K=2, S=4096, H=128, Hp=256),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.5, seed=7), 0),
    ("ragged-h256", W("ragged256", R=5, E=20, B=4, K=3, S=171, H=256, Hp=320),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.3, seed=6), 0),
    # ragged groups with several 256-wide column tiles in both directions, and
    # an input gradient with 128-wide column tiles (H = 384)
    ("ragged-h512", W("ragged512", R=4, E=12, B=3, K=3, S=500, H=512, Hp=512),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.2, seed=11), 0),
    ("ragged-h384", W("ragged384", R=4, E=12, B=3, K=3, S=400, H=384, Hp=512),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.2, seed=12), 0),
    # 128-wide weight-gradient column tiles (H' = 384) on the single-CTA kernel
    ("bn128-h384", W("bn128", R=4, E=8, B=2, K=2, S=300, H=256, Hp=384),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.5, seed=14), 0),
    # every group shorter than one 64-row block: each weight-gradient item's
    # only block runs past the group's end (CTA-pair kernel, H and H' of 256)
    ("groups-under-64-rows", W("short-groups", R=4, E=64, B=16, K=2, S=64, H=256, Hp=256),
     lambda w: syn.gumbel_topk_routing(w.R, w.S, w.K, w.E, alpha=1.0, seed=13), 0),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gh.ensure_library()


def _setup(w, mk, policy, gemm_rows=0):
    rt = mk(w)
    od = gh.odims(w, policy)
    fp = oplanner.full_plan(rt.idx, od)
    run = gh.Run(w, rt, policy=policy, gemm_rows=gemm_rows)
    run.plan()
    return rt, od, fp, run


@pytest.mark.parametrize("name,w,mk,policy", CASES, ids=[c[0] for c in CASES])
def test_combine_backward(name, w, mk, policy):
    rt, od, fp, run = _setup(w, mk, policy)
    y = syn.normal_bf16((w.N, w.Hp), 1.0, 81).cuda()
    dout = syn.normal_bf16((w.R, w.S, w.Hp), 1.0, 82).cuda()
    dy = torch.zeros(w.N * w.Hp, dtype=torch.bfloat16, device="cuda")
    dg = torch.zeros(w.N, dtype=torch.float32, device="cuda")
    mx.moonep_combine_backward(run.d, run.ws.buf, y.view(-1), run.gates, dout.view(-1), dy, dg)
    dst = fp["dst"].reshape(-1)
    ycopy = gh.host_bits(y)[dst]
    want_dy, want_dg = olayer.combine_backward(ycopy, gh.host_bits(dout), rt.gates, od)
    got_dy = gh.host_bits(dy).reshape(w.N, w.Hp)[dst]
    assert np.array_equal(got_dy, want_dy)  # one rounding of an exact fp32 product
    gh.assert_close(dg.cpu().numpy().reshape(w.R, w.S, w.K), want_dg, f"{name} d_gates")


@pytest.mark.parametrize("name,w,mk,policy", CASES, ids=[c[0] for c in CASES])
def test_grouped_gemm_dx(name, w, mk, policy):
    rt, od, fp, run = _setup(w, mk, policy)
    mx.moonep_prefetch_weights(run.d, run.ws.buf, run.w_home, run.w_slot)
    dy = syn.normal_bf16((w.N, w.Hp), 1.0, 83).cuda()
    drecv = torch.zeros(w.N * w.H, dtype=torch.bfloat16, device="cuda")
    mx.moonep_grouped_gemm_dx(run.d, run.ws.buf, dy.view(-1), run.w_home, run.w_slot, drecv)
    dst = fp["dst"].reshape(-1)
    per_e = olayer.expert_backward(gh.host_bits(run.x), gh.host_bits(run.w_home), rt.idx,
                                   gh.host_bits(dy)[dst], od)
    got = gh.bf16_to_np(drecv).reshape(w.N, w.H)
    for e, (cids, want, _) in per_e.items():
        if cids.size:
            gh.assert_close(got[dst[cids]], olayer.bf16_to_f64(want), f"{name} dRecv expert {e}")


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("name,w,mk,policy", [CASES[0], CASES[5], CASES[6]],
                         ids=[CASES[i][0] for i in (0, 5, 6)])
def test_grouped_gemm_dx_fixed_tile_rows(name, w, mk, policy, rows):
    """The input-gradient GEMM with the work-tile height fixed either way."""
    rt, od, fp, run = _setup(w, mk, policy, gemm_rows=rows)
    assert int(run.ws.tables()["counters"][7]) == rows
    mx.moonep_prefetch_weights(run.d, run.ws.buf, run.w_home, run.w_slot)
    dy = syn.normal_bf16((w.N, w.Hp), 1.0, 83).cuda()
    drecv = torch.zeros(w.N * w.H, dtype=torch.bfloat16, device="cuda")
    mx.moonep_grouped_gemm_dx(run.d, run.ws.buf, dy.view(-1), run.w_home, run.w_slot, drecv)
    dst = fp["dst"].reshape(-1)
    per_e = olayer.expert_backward(gh.host_bits(run.x), gh.host_bits(run.w_home), rt.idx,
                                   gh.host_bits(dy)[dst], od)
    got = gh.bf16_to_np(drecv).reshape(w.N, w.H)
    for e, (cids, want, _) in per_e.items():
        if cids.size:
            gh.assert_close(got[dst[cids]], olayer.bf16_to_f64(want), f"{name} dRecv expert {e}")


@pytest.mark.parametrize("name,w,mk,policy", CASES, ids=[c[0] for c in CASES])
def test_grouped_gemm_dw(name, w, mk, policy):
    rt, od, fp, run = _setup(w, mk, policy)
    recv = syn.normal_bf16((w.N, w.H), 1.0, 84).cuda()
    dy = syn.normal_bf16((w.N, w.Hp), 1.0, 85).cuda()
    g_home = syn.integer_f32((w.E, w.H, w.Hp), -4, 5, 86).cuda()
    g_slot = syn.integer_f32((w.R, w.B, w.H, w.Hp), -4, 5, 87).cuda()
    h0, s0 = g_home.cpu().numpy().astype(np.float64), g_slot.cpu().numpy().astype(np.float64)
    mx.moonep_grouped_gemm_dw(run.d, run.ws.buf, recv.view(-1), dy.view(-1), g_home.view(-1),
                              g_slot.view(-1))
    parts = olayer.grouped_gemm_dw_rows(gh.host_bits(recv), gh.host_bits(dy), fp["plan"])
    want_h, want_s = h0.copy(), s0.copy()
    for (u, g), dw in parts.items():
        if g < w.E:
            want_h[g] += dw
        else:
            want_s[u, g - w.E] += dw
    gh.assert_close(g_home.cpu().numpy(), want_h, f"{name} g_home")
    gh.assert_close(g_slot.cpu().numpy(), want_s, f"{name} g_slot")


@pytest.mark.parametrize("name,w,mk,policy", CASES, ids=[c[0] for c in CASES])
def test_dispatch_backward(name, w, mk, policy):
    rt, od, fp, run = _setup(w, mk, policy)
    drecv = syn.normal_bf16((w.N, w.H), 1.0, 88).cuda()
    dx = torch.zeros(w.R * w.S * w.H, dtype=torch.bfloat16, device="cuda")
    mx.moonep_dispatch_backward(run.d, run.ws.buf, drecv.view(-1), dx)
    want = olayer.dispatch_backward(gh.host_bits(drecv)[fp["dst"].reshape(-1)], od)
    gh.assert_close(gh.bf16_to_np(dx).reshape(w.R * w.S, w.H), olayer.bf16_to_f64(want),
                    f"{name} dx")


@pytest.mark.parametrize("name,w,mk,policy", CASES, ids=[c[0] for c in CASES])
def test_training_step_against_plan_free_gradients(name, w, mk, policy):
    """forward -> combine backward -> dX and dW GEMMs -> dispatch backward ->
    reduce_grad; compare with the dense per-expert definitions."""
    rt, od, fp, run = _setup(w, mk, policy)
    run.forward()
    d = run.d
    dout = syn.normal_bf16((w.R, w.S, w.Hp), 1.0, 89).cuda()
    dy = torch.zeros(w.N * w.Hp, dtype=torch.bfloat16, device="cuda")
    dg = torch.zeros(w.N, dtype=torch.float32, device="cuda")
    drecv = torch.zeros(w.N * w.H, dtype=torch.bfloat16, device="cuda")
    dx = torch.zeros(w.R * w.S * w.H, dtype=torch.bfloat16, device="cuda")
    g_home = syn.integer_f32((w.E, w.H, w.Hp), -4, 5, 90).cuda()
    g_slot = torch.zeros(w.R * w.B * w.H * w.Hp, dtype=torch.float32, device="cuda")
    h0 = g_home.cpu().numpy().astype(np.float64)
    mx.moonep_combine_backward(d, run.ws.buf, run.y, run.gates, dout.view(-1), dy, dg)
    mx.moonep_grouped_gemm_dx(d, run.ws.buf, dy, run.w_home, run.w_slot, drecv)
    mx.moonep_grouped_gemm_dw(d, run.ws.buf, run.recv, dy, g_home.view(-1), g_slot)
    mx.moonep_dispatch_backward(d, run.ws.buf, drecv, dx)
    mx.moonep_reduce_grad(d, run.ws.buf, g_home.view(-1), g_slot)
    torch.cuda.synchronize()
    assert mx.moonep_read_status(d, run.ws.buf) == 0

    xb, wb = gh.host_bits(run.x), gh.host_bits(run.w_home)
    per_e = olayer.expert_outputs(xb, wb, rt.idx, od)
    ycopy = np.zeros((w.N, w.Hp), dtype=np.uint16)
    for e, (cids, yb) in per_e.items():
        ycopy[cids] = yb
    dyc, _ = olayer.combine_backward(ycopy, gh.host_bits(dout), rt.gates, od)
    bwd = olayer.expert_backward(xb, wb, rt.idx, dyc, od)
    want_h = h0.copy()
    drc = np.zeros((w.N, w.H), dtype=np.uint16)
    for e, (cids, drb, dw) in bwd.items():
        want_h[e] += dw
        drc[cids] = drb
    gh.assert_close(g_home.cpu().numpy(), want_h, f"{name} folded weight gradient")
    assert bool((g_slot == 0).all())  # every slot was consumed by reduce_grad
    want_dx = olayer.dispatch_backward(drc, od)
    gh.assert_close(gh.bf16_to_np(dx).reshape(w.R * w.S, w.H), olayer.bf16_to_f64(want_dx),
                    f"{name} token gradient")
