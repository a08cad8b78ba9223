"""moonep_plan_noalloc: the planner for callers that cannot allocate device
memory (fixed pools, allocators frozen after warm-up), checked against
moonep_plan.

It keeps the planner's internal scratch in a static device array inside the
library instead of the caller's workspace.  Its output tables must equal
moonep_plan's bit for bit (they are integer tables), on two calls in a row with
different routings, so scratch left by the first call cannot leak into the
second.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import perfectly_balanced_token_gb300 as mx
from perfectly_balanced_token_gb300 import _lib
from perfectly_balanced_token_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

OUTPUT_TABLES = ("status", "counters", "T", "load", "keep", "gidx", "fills", "slot_expert",
                 "n_recv", "src", "cu_seqlens", "dst", "inverse", "route", "occupied", "reduce")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from perfectly_balanced_token_gb300.build import build
    build()
    mx.library()


def _a256(n):
    return (max(n, 4) + 255) // 256 * 256


def _regions(ws: mx.PlanWorkspace, n_mtiles: int):
    """Byte ranges of every output table in the workspace.  The reduce lists
    are the slot table [E][R] and two [E] tables; the tile list is cut at the
    tiles the plan produced; the planner's internal scratch is excluded."""
    lay, d = ws.layout, ws.dims
    offs = sorted((getattr(lay, f), f) for f in _lib._LAYOUT_FIELDS[1:])
    ends = {f: (offs[i + 1][0] if i + 1 < len(offs) else lay.total_bytes)
            for i, (_, f) in enumerate(offs)}
    out = {f: (getattr(lay, f), ends[f]) for f in OUTPUT_TABLES}
    out["reduce"] = (lay.reduce, lay.reduce + _a256(4 * d.E * d.R) + 2 * _a256(4 * d.E))
    out["mtiles"] = (lay.mtiles, lay.mtiles + 16 * n_mtiles)
    n_groups = int(ws.view("counters", (8,))[6])
    out["groups"] = (lay.groups, lay.groups + 16 * n_groups)
    return out


def _plan_both(d, idx):
    ref = mx.PlanWorkspace(d)
    new = mx.PlanWorkspace(d)
    new.buf.fill_(0xA5)  # the variant must write every output it owns
    ref.buf.fill_(0xA5)
    lib = mx.library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.moonep_plan(ctypes.byref(d), ctypes.c_void_p(idx.data_ptr()),
                           ctypes.c_void_p(ref.buf.data_ptr()), stream) == 0
    assert lib.moonep_plan_noalloc(ctypes.byref(d), ctypes.c_void_p(idx.data_ptr()),
                                   ctypes.c_void_p(new.buf.data_ptr()), stream) == 0
    torch.cuda.synchronize()
    return ref, new


@pytest.mark.parametrize("w,maxvios", [(syn.SMALL, (5.0, 1.0)), (syn.PAGES, (20.0, 0.2))],
                         ids=["r8-e64", "pages-benchmark-shaped"])
def test_noalloc_plan_matches_plan_on_two_calls_in_a_row(w, maxvios):
    d = mx.dims(w.R, w.E, w.B, w.K, w.S, w.H, w.Hp, w.mode)
    for mv in maxvios:  # two calls in a row, different routings
        rt = syn.routing_for(w, mv, seed=3)
        idx = torch.from_numpy(rt.idx).cuda()
        ref, new = _plan_both(d, idx)
        assert mx.moonep_read_status(d, new.buf) == 0
        n_mt = int(ref.view("counters", (8,))[1])
        for name, (a, b) in _regions(ref, n_mt).items():
            assert torch.equal(ref.buf[a:b], new.buf[a:b]), f"{name} differs (maxvio {mv})"
        # the variant's plan drives the rest of the path like the original's
        tabs = new.tables()
        assert np.all(tabs["cu_seqlens"][:, -1] == w.C)


def test_noalloc_plan_drives_dispatch_identically():
    w = syn.TINY
    d = mx.dims(w.R, w.E, w.B, w.K, w.S, w.H, w.Hp, w.mode)
    rt = syn.routing_for(w)
    idx = torch.from_numpy(rt.idx).cuda()
    ref, new = _plan_both(d, idx)
    x = syn.normal_bf16((w.R, w.S, w.H), 1.0, 1).cuda()
    r1 = torch.zeros(w.N * w.H, dtype=torch.bfloat16, device="cuda")
    r2 = torch.zeros_like(r1)
    mx.moonep_dispatch(d, ref.buf, x, r1)
    mx.moonep_dispatch(d, new.buf, x, r2)
    torch.cuda.synchronize()
    assert torch.equal(r1, r2)
