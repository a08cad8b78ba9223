"""Parity at the full benchmark sizes, in the launch configuration bench.py times.

Plans and indices are compared in full and bit-exact; the dispatch buffer and
the prefetched slots are compared in full on the device (byte-exact gathers
driven by the oracle's inverse permutation and slot table); GEMM, combine and
reduce_grad are compared on seeded samples the oracle computes one by one:
every slot-holding expert (capped) plus random experts, migrated and kept
copies of each, random tokens for combine, and whole expert rows for
reduce_grad.
"""
import gc

import numpy as np
import pytest
import torch

import perfectly_balanced_token_gb300 as mx
from oracle import layer as olayer
from oracle import planner as oplanner
from oracle import theory
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


def _sample_experts(fp, E, rng, n_slot=16, n_rand=16):
    held = sorted(set(int(e) for e in fp["slot_expert"].reshape(-1) if e >= 0))
    pick = list(rng.permutation(held)[:n_slot]) if held else []
    rest = [e for e in rng.permutation(E) if e not in pick]
    return [int(e) for e in pick + rest[:n_rand]]


def _check_gemm_sample(run, fp, rt, w, rng, per_expert=48):
    od = gh.odims(w)
    flat = rt.idx.reshape(-1)
    keep = fp["keep"]
    q = fp["gidx"].reshape(-1)
    dst = fp["dst"].reshape(-1)
    xs = run.x.view(w.R * w.S, w.H)
    y = run.y.view(w.N, w.Hp)
    for e in _sample_experts(fp, w.E, rng):
        cids = np.nonzero(flat == e)[0]
        if cids.size == 0:
            continue
        moved = cids[q[cids] >= keep[e]]
        kept = cids[q[cids] < keep[e]]
        take = np.concatenate([rng.permutation(moved)[:per_expert // 2],
                               rng.permutation(kept)[:per_expert // 2]])
        xb = syn.bf16_bits(xs[torch.from_numpy(take // w.K).cuda()].cpu())
        wb = syn.bf16_bits(run.w_home[e].cpu())
        want = olayer.to_bf16(olayer.bf16_to_f64(xb) @ olayer.bf16_to_f64(wb))
        got = gh.bf16_to_np(y[torch.from_numpy(dst[take]).cuda()])
        gh.assert_close(got, olayer.bf16_to_f64(want), f"{w.name} Y expert {e}")
    del od


def _check_full_dispatch_and_prefetch(run, fp, w):
    inv = torch.from_numpy(fp["inverse"]).cuda()
    want = run.x.view(w.R * w.S, w.H)[inv // w.K]
    assert torch.equal(run.recv.view(w.N, w.H), want)
    del want, inv
    if w.B:
        ws = run.w_slot.view(w.R * w.B, w.H, w.Hp)
        occ = fp["slot_expert"].reshape(-1)
        for s in np.nonzero(occ >= 0)[0]:
            assert torch.equal(ws[int(s)], run.w_home[int(occ[s])]), f"slot {s}"
        empty = np.nonzero(occ < 0)[0]
        for s in empty[:8]:
            assert bool((ws[int(s)].view(torch.int16) == 0x7F7F).all())


def _check_combine_isolated(run, fp, rt, w, rng, n_tok=2048):
    od = gh.odims(w)
    y = syn.normal_bf16((w.N, w.Hp), 1.0, 78, "cuda")
    mx.moonep_combine(run.d, run.ws.buf, y.view(-1), run.gates, run.out)
    toks = np.sort(rng.choice(w.R * w.S, size=n_tok, replace=False))
    rows = fp["dst"].reshape(w.R * w.S, w.K)[toks]
    ysub = syn.bf16_bits(y[torch.from_numpy(rows.reshape(-1)).cuda()].cpu())
    # combine over the gathered rows: rebase destinations onto the gathered copy
    sub = oplanner.Dims(R=1, E=od.E, B=od.B, K=w.K, S=n_tok, H=w.H, Hp=w.Hp)
    local_dst = np.arange(n_tok * w.K).reshape(1, n_tok, w.K)
    gsub = rt.gates.reshape(w.R * w.S, w.K)[toks].reshape(1, n_tok, w.K)
    want = olayer.combine(ysub, local_dst, gsub, sub)
    got = gh.bf16_to_np(run.out.view(w.R * w.S, w.Hp)[torch.from_numpy(toks).cuda()])
    gh.assert_close(got, olayer.bf16_to_f64(want), f"{w.name} combine")
    del y


def _check_reduce_sample(run, fp, w, rng, n_exp=6):
    plan = fp["plan"]
    hh = w.H * w.Hp
    g_home = syn.normal_f32((w.E, w.H, w.Hp), 1.0, 90, "cuda")
    g_slot = syn.normal_f32((w.R, w.B, w.H, w.Hp), 1.0, 91, "cuda")
    occ = fp["slot_expert"] >= 0
    occ_t = torch.from_numpy(occ).cuda()
    g_slot[~occ_t] = 7.0
    lists = oplanner.reduce_lists(plan)
    with_slots = [e for e in range(w.E) if lists[e]]
    pick = [int(e) for e in rng.permutation(with_slots)[:n_exp]]
    before_home = {e: g_home[e].cpu().numpy().copy() for e in pick}
    before_slot = {(u, j): g_slot[u, j].cpu().numpy().copy() for e in pick for (u, j) in lists[e]}
    mx.moonep_reduce_grad(run.d, run.ws.buf, g_home.view(-1), g_slot.view(-1))
    torch.cuda.synchronize()
    for e in pick:
        acc = before_home[e].astype(np.float32)
        for (u, j) in lists[e]:
            acc = acc + before_slot[(u, j)]
        assert np.array_equal(g_home[e].cpu().numpy(), acc), f"reduce expert {e}"
    assert bool((g_slot[occ_t] == 0).all())
    assert bool((g_slot[~occ_t] == 7.0).all())
    assert hh > 0
    del g_home, g_slot


# every routing the benchmark times, under the planner policy it times it with:
# the pages shape at maxvio 0.2, 1, 10 and 20 and the K3 shape at maxvio 1 and
# 10 with the plain policy; the largest-first policy at the most skewed routing
# of each shape
LARGE = [
    ("pages-maxvio0.2", syn.PAGES, 0.2, 0),
    ("pages-maxvio1", syn.PAGES, 1.0, 0),
    ("pages-maxvio10", syn.PAGES, 10.0, 0),
    ("pages-maxvio20", syn.PAGES, 20.0, 0),
    ("k3-maxvio1", syn.K3, 1.0, 0),
    ("k3-maxvio10", syn.K3, 10.0, 0),
    ("pages-maxvio20-largest-first", syn.PAGES, 20.0, 1),
    ("k3-maxvio10-largest-first", syn.K3, 10.0, 1),
]


@pytest.mark.parametrize("name,w,mv,policy", LARGE, ids=[c[0] for c in LARGE])
def test_full_size_parity(name, w, mv, policy):
    _free()
    rng = np.random.default_rng(0)
    rt = syn.routing_for(w, mv, seed=0)
    fp = oplanner.full_plan(rt.idx, gh.odims(w, policy))
    run = gh.Run(w, rt, guard=1 << 16, policy=policy)
    run.forward()
    assert mx.moonep_read_status(run.d, run.ws.buf) == 0
    gh.compare_plan(run.ws.tables(), fp, gh.odims(w, policy))
    _check_full_dispatch_and_prefetch(run, fp, w)
    _check_gemm_sample(run, fp, rt, w, rng)
    run.check_all_guards()
    _check_combine_isolated(run, fp, rt, w, rng)
    _check_reduce_sample(run, fp, w, rng)
    del run
    _free()


def test_theorem2_worst_case_on_gpu_train_then_infer():
    _free()
    rng = np.random.default_rng(1)
    for w in (syn.ADVERSARIAL_TRAIN, syn.ADVERSARIAL_INFER):
        rt = syn.routing_for(w)
        fp = oplanner.full_plan(rt.idx, gh.odims(w))
        run = gh.Run(w, rt, guard=1 << 16)
        run.forward()
        tabs = run.ws.tables()
        gh.compare_plan(tabs, fp, gh.odims(w))
        assert int(tabs["n_recv"][0]) == theory.theorem2_bound(w.R, w.E) == 42
        assert tabs["n_recv"].tolist() == [42, 36, 30, 24, 18, 12, 6, 0]
        if w.mode == 1:  # B=4: experts beyond the slots run from their home rows
            assert any(fp["plan"].overflow[u] for u in range(w.R))
        _check_full_dispatch_and_prefetch(run, fp, w)
        _check_gemm_sample(run, fp, rt, w, rng, per_expert=32)
        run.check_all_guards()
        del run
        _free()
