"""Backward parity at the full benchmark sizes (pages and K3 shapes).

Each backward kernel runs once on the planned full-size layer with seeded
synthetic inputs (the same recipe the small cases use), and seeded samples of
its outputs are checked against the oracle's definitions computed one by one:

* combine backward: sampled tokens, every one of their K copies;
* input-gradient GEMM: sampled copies (migrated and kept) of every
  slot-holding expert (capped) plus random experts;
* weight-gradient GEMM followed by reduce_grad: sampled rows of the home
  gradient of sampled experts equal their initial value plus the plan-free sum
  over all copies of the expert of x_token[h] * dY[copy] (slot groups folded
  back by reduce_grad), and every slot is zero afterwards;
* dispatch backward: sampled tokens.

Expected values come from the synthetic inputs and the oracle's plan only.
Tolerance as everywhere: |got - want| <= 1e-2 + 2e-2 |want|.
"""
import gc

import numpy as np
import pytest
import torch

import perfectly_balanced_token_gb300 as mx
from oracle import layer as olayer
from oracle import planner as oplanner
from perfectly_balanced_token_gb300 import synthetic as syn
from tests import gpu_harness as gh

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gh.ensure_library()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _experts(fp, E, rng, n_slot, n_rand):
    held = sorted(set(int(e) for e in fp["slot_expert"].reshape(-1) if e >= 0))
    pick = [int(e) for e in rng.permutation(held)[:n_slot]] if held else []
    rest = [int(e) for e in rng.permutation(E) if e not in pick]
    return pick + rest[:n_rand]


def _rows(t, idx):
    return t[torch.from_numpy(np.asarray(idx, dtype=np.int64)).cuda()]


LARGE = [
    ("pages-maxvio1", syn.PAGES, 1.0),
    ("k3-maxvio10", syn.K3, 10.0),
]


@pytest.mark.parametrize("name,w,mv", LARGE, ids=[c[0] for c in LARGE])
def test_full_size_backward(name, w, mv):
    _free()
    rng = np.random.default_rng(3)
    rt = syn.routing_for(w, mv, seed=0)
    od = gh.odims(w)
    fp = oplanner.full_plan(rt.idx, od)
    run = gh.Run(w, rt, guard=1 << 16)
    run.forward()  # plan, slot weights and the dispatched rows the backward reads
    d, ws = run.d, run.ws.buf
    bf, f32 = torch.bfloat16, torch.float32
    flat = rt.idx.reshape(-1)
    dst = fp["dst"].reshape(-1)
    q, keep = fp["gidx"].reshape(-1), fp["keep"]

    # synthetic inputs of each kernel
    y_in = syn.normal_bf16((w.N, w.Hp), 1.0, 80, "cuda")
    dout = syn.normal_bf16((w.R * w.S, w.Hp), 1.0, 81, "cuda")
    dy_in = syn.normal_bf16((w.N, w.Hp), 1.0, 82, "cuda")
    drecv_in = syn.normal_bf16((w.N, w.H), 1.0, 83, "cuda")
    g_home = syn.normal_f32((w.E, w.H, w.Hp), 1.0, 84, "cuda")
    g_slot = torch.zeros(w.R * w.B * w.H * w.Hp, dtype=f32, device="cuda")
    dy_cb = torch.zeros(w.N * w.Hp, dtype=bf, device="cuda")
    dg = torch.zeros(w.N, dtype=f32, device="cuda")
    drecv = torch.zeros(w.N * w.H, dtype=bf, device="cuda")
    dx = torch.zeros(w.R * w.S * w.H, dtype=bf, device="cuda")

    dw_experts = _experts(fp, w.E, rng, n_slot=8, n_rand=8)
    h_rows = np.sort(rng.choice(w.H, size=16, replace=False))
    h_t = torch.from_numpy(h_rows).cuda()
    g0 = {e: g_home[e][h_t].cpu().numpy().astype(np.float64) for e in dw_experts}

    mx.moonep_combine_backward(d, ws, y_in.view(-1), run.gates, dout.view(-1), dy_cb, dg)
    mx.moonep_grouped_gemm_dx(d, ws, dy_in.view(-1), run.w_home, run.w_slot, drecv)
    mx.moonep_grouped_gemm_dw(d, ws, run.recv, dy_in.view(-1), g_home.view(-1), g_slot)
    mx.moonep_reduce_grad(d, ws, g_home.view(-1), g_slot)
    mx.moonep_dispatch_backward(d, ws, drecv_in.view(-1), dx)
    torch.cuda.synchronize()
    assert mx.moonep_read_status(d, ws) == 0

    # combine backward on sampled tokens (the oracle on the gathered copies)
    toks = np.sort(rng.choice(w.R * w.S, size=min(1024, w.R * w.S), replace=False))
    cids = (toks[:, None] * w.K + np.arange(w.K)).reshape(-1)
    sub = oplanner.Dims(R=1, E=od.E, B=od.B, K=w.K, S=toks.size, H=w.H, Hp=w.Hp)
    ysub = gh.host_bits(_rows(y_in, dst[cids]))
    want_dy, want_dg = olayer.combine_backward(
        ysub, gh.host_bits(_rows(dout, toks)), rt.gates.reshape(-1, w.K)[toks][None], sub)
    got_dy = gh.host_bits(_rows(dy_cb.view(w.N, w.Hp), dst[cids]))
    assert np.array_equal(got_dy, want_dy), f"{name} combine-backward dY"  # one rounding of an exact product
    gh.assert_close(dg.cpu().numpy()[cids], want_dg.reshape(-1), f"{name} combine-backward dgate")

    # input gradient on sampled copies: dRecv[row] = bf16(dY[row] . W_e^T)
    drv = drecv.view(w.N, w.H)
    for e in _experts(fp, w.E, rng, n_slot=16, n_rand=16):
        ce = np.nonzero(flat == e)[0]
        if ce.size == 0:
            continue
        moved, kept = ce[q[ce] >= keep[e]], ce[q[ce] < keep[e]]
        take = np.concatenate([rng.permutation(moved)[:16], rng.permutation(kept)[:16]])
        rows = dst[take]
        want = olayer.to_bf16(olayer.bf16_to_f64(gh.host_bits(_rows(dy_in, rows)))
                              @ olayer.bf16_to_f64(gh.host_bits(run.w_home[e])).T)
        gh.assert_close(gh.bf16_to_np(_rows(drv, rows)), olayer.bf16_to_f64(want),
                        f"{name} dRecv expert {e}")

    # weight gradient after reduce_grad: plan-free per-expert sums on sampled rows
    xs = run.x.view(w.R * w.S, w.H)
    for e in dw_experts:
        ce = np.nonzero(flat == e)[0]
        xe = olayer.bf16_to_f64(gh.host_bits(_rows(xs, ce // w.K)[:, h_t]))
        dye = olayer.bf16_to_f64(gh.host_bits(_rows(dy_in, dst[ce])))
        want = g0[e] + xe.T @ dye
        gh.assert_close(g_home[e][h_t].cpu().numpy(), want, f"{name} dW expert {e}")
    assert bool((g_slot == 0).all()), f"{name}: a slot gradient was not consumed"

    # dispatch backward on sampled tokens: dx[t] = bf16(sum_k dRecv[dst[t, k]])
    toks = np.sort(rng.choice(w.R * w.S, size=min(1024, w.R * w.S), replace=False))
    cids = (toks[:, None] * w.K + np.arange(w.K)).reshape(-1)
    sub = oplanner.Dims(R=1, E=od.E, B=od.B, K=w.K, S=toks.size, H=w.H, Hp=w.Hp)
    want = olayer.dispatch_backward(gh.host_bits(_rows(drecv_in, dst[cids])), sub)
    got = gh.bf16_to_np(_rows(dx.view(w.R * w.S, w.H), toks))
    gh.assert_close(got, olayer.bf16_to_f64(want), f"{name} dX")

    del run, y_in, dout, dy_in, drecv_in, g_home, g_slot, dy_cb, dg, drecv, dx
    _free()
