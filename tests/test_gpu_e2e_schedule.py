"""The end-to-end schedule that bench.py times: with the host copies on their
own streams and the device buffers double-buffered, every step must still
compute on its own inputs. Seven steps go through the pipelined schedule with
inputs that change from step to step; each step's read-back must equal, bit
for bit, the same step run alone on one stream."""
import types

import pytest
import torch

import bench
import perfectly_balanced_token_gb300 as mx
from perfectly_balanced_token_gb300 import synthetic as syn
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu


def test_pipelined_schedule_runs_every_step_on_its_own_inputs():
    gh.ensure_library()
    w = syn.SMALL
    dev = torch.device("cuda")
    d = mx.dims(w.R, w.E, w.B, w.K, w.S, w.H, w.Hp, w.mode, 0)
    ws = mx.PlanWorkspace(d, device=dev)
    routings = [syn.routing_for(w, mv, seed=0) for mv in (1.0, 5.0, 0.0)]
    w_home = syn.normal_bf16((w.E, w.H, w.Hp), 0.02, 2, dev)
    w_slot = torch.zeros(w.R * w.B * w.H * w.Hp, dtype=torch.bfloat16, device=dev)
    g_home = torch.zeros(w.E * w.H * w.Hp, dtype=torch.float32, device=dev)
    g_slot = torch.zeros(w.R * w.B * w.H * w.Hp, dtype=torch.float32, device=dev)
    res = bench.run_e2e(types.SimpleNamespace(steps=8), mx, syn, torch, d, w, routings, ws,
                        w_home, w_slot, g_home, g_slot, dev, torch.cuda.current_stream(), 1,
                        verify_steps=7)
    assert res == {"steps": 7, "mismatches": 0}
    assert mx.moonep_read_status(d, ws.buf) == 0
