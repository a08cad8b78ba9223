"""Failure detection on the GPU without faulting it: a bounded device wait
that runs out (on an mbarrier nothing arrives on) must record
MOONEP_ERR_TIMEOUT in the status word and return, and the context must stay
usable for the next plan.  Routing errors are covered in test_gpu_parity."""
import numpy as np
import pytest
import torch

import perfectly_balanced_token_gb300 as mx
from perfectly_balanced_token_gb300 import _lib
from perfectly_balanced_token_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from perfectly_balanced_token_gb300.build import build
    build()
    mx.library()


@pytest.mark.parametrize("limit_us", [2000, 50000])
def test_bounded_wait_gives_up_with_timeout_status(limit_us):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int32, device="cuda")
    mx.moonep_selftest_bounded_wait(status, limit_us, elapsed)
    torch.cuda.synchronize()
    assert int(status.item()) & _lib.ERR_TIMEOUT
    waited = int(elapsed.item())
    assert limit_us <= waited < limit_us + 1_000_000
    # the context still works: a plan right after is correct and clean
    w = syn.TINY
    d = mx.dims(w.R, w.E, w.B, w.K, w.S, w.H, w.Hp, w.mode)
    ws = mx.PlanWorkspace(d)
    rt = syn.routing_for(w)
    mx.moonep_plan(d, torch.from_numpy(rt.idx).cuda(), ws.buf)
    assert mx.moonep_read_status(d, ws.buf) == 0
    assert np.all(ws.tables()["cu_seqlens"][:, -1] == w.C)
