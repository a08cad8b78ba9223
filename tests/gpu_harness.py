"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the CPU oracle.

Float tolerance (bf16 values with fp32 accumulation): |got - want| <= 1e-2 +
2e-2 * |want|, elementwise, with `want` the oracle's value.
"""
from __future__ import annotations

import numpy as np
import torch

import perfectly_balanced_token_gb300 as mx
from oracle import layer as olayer
from oracle import planner as oplanner
from perfectly_balanced_token_gb300 import synthetic as syn

ATOL, RTOL = 1e-2, 2e-2


def ensure_library():
    from perfectly_balanced_token_gb300.build import build
    build()
    mx.library()


def odims(w, policy=0) -> oplanner.Dims:
    return oplanner.Dims(R=w.R, E=w.E, B=w.B, K=w.K, S=w.S, H=w.H, Hp=w.Hp, mode=w.mode,
                         policy=policy)


def cdims(w, policy=0, gemm_rows=0):
    return mx.dims(w.R, w.E, w.B, w.K, w.S, w.H, w.Hp, w.mode, policy, gemm_rows)


def assert_close(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want)
    bad = err > ATOL + RTOL * np.abs(want)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at "
                             f"{tuple(i)}: got {got[tuple(i)]}, want {want[tuple(i)]}")


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bits_to_np(bits: np.ndarray) -> np.ndarray:
    return olayer.bf16_to_f64(bits)


def compare_plan(tabs: dict, fp: dict, d: oplanner.Dims):
    """Bit-exact comparison of every exported plan table with the oracle."""
    assert int(tabs["status"][0]) == 0, mx.status_string(int(tabs["status"][0]))
    assert np.array_equal(tabs["T"], fp["T"]), "T"
    assert np.array_equal(tabs["load"], fp["load"]), "load"
    assert int(tabs["counters"][0]) == fp["n_fills"], "n_fills"
    nf = fp["n_fills"]
    assert np.array_equal(tabs["fills"][:nf], fp["fills"][:nf]), "fills"
    assert np.array_equal(tabs["keep"], fp["keep"]), "keep"
    assert np.array_equal(tabs["slot_expert"], fp["slot_expert"]), "slot_expert"
    assert np.array_equal(tabs["n_recv"], fp["n_recv"]), "n_recv"
    assert np.array_equal(tabs["src"], fp["src"]), "src"
    assert np.array_equal(tabs["gidx"], fp["gidx"]), "gidx"
    assert np.array_equal(tabs["cu_seqlens"], fp["cu_seqlens"]), "cu_seqlens"
    assert np.array_equal(tabs["dst"], fp["dst"]), "dst"
    assert np.array_equal(tabs["inverse"], fp["inverse"]), "inverse"
    assert int(tabs["counters"][2]) == int((fp["slot_expert"] >= 0).sum()), "n_occupied"


class Run:
    """Device buffers and one pass of the CUDA path for a workload."""

    def __init__(self, w, routing, seed=0, guard=4096, policy=0, gemm_rows=0):
        self.w, self.d, self.od = w, cdims(w, policy, gemm_rows), odims(w, policy)
        self.routing = routing
        dev = "cuda"
        self.ws = mx.PlanWorkspace(self.d)
        self.idx = torch.from_numpy(np.ascontiguousarray(routing.idx)).to(dev)
        self.gates = torch.from_numpy(np.ascontiguousarray(routing.gates)).to(dev)
        self.guard = guard
        big = w.R * w.S * w.H > (1 << 26)
        gen_dev = dev if big else "cpu"
        self.x = syn.normal_bf16((w.R, w.S, w.H), 1.0, seed + 1, gen_dev).to(dev)
        self.w_home = syn.normal_bf16((w.E, w.H, w.Hp), 0.02, seed + 2,
                                      dev if w.E * w.H * w.Hp > (1 << 26) else "cpu").to(dev)
        self.w_slot_full = self._guarded(w.R * w.B * w.H * w.Hp, torch.bfloat16, 0x7F7F)
        self.recv_full = self._guarded(w.N * w.H, torch.bfloat16, 0x7F7F)
        self.y_full = self._guarded(w.N * w.Hp, torch.bfloat16, 0x7F7F)
        self.out_full = self._guarded(w.R * w.S * w.Hp, torch.bfloat16, 0x7F7F)

    def _guarded(self, n, dtype, pattern):
        """A buffer with `guard` canary elements on both sides of the payload."""
        t = torch.empty(n + 2 * self.guard, dtype=dtype, device="cuda")
        t.view(torch.int16).fill_(pattern)
        return t

    def payload(self, t, n):
        return t[self.guard:self.guard + n]

    def check_guards(self, t, n, pattern, what):
        g = self.guard
        raw = t.view(torch.int16)
        assert bool((raw[:g] == pattern).all()) and bool((raw[g + n:] == pattern).all()), \
            f"{what}: canary overwritten"

    @property
    def w_slot(self):
        n = self.w.R * self.w.B * self.w.H * self.w.Hp
        return self.payload(self.w_slot_full, n) if n else None

    @property
    def recv(self):
        return self.payload(self.recv_full, self.w.N * self.w.H)

    @property
    def y(self):
        return self.payload(self.y_full, self.w.N * self.w.Hp)

    @property
    def out(self):
        return self.payload(self.out_full, self.w.R * self.w.S * self.w.Hp)

    def plan(self):
        mx.moonep_plan(self.d, self.idx, self.ws.buf)
        return self.ws.tables()

    def forward(self):
        d = self.d
        mx.moonep_plan(d, self.idx, self.ws.buf)
        mx.moonep_prefetch_weights(d, self.ws.buf, self.w_home, self.w_slot)
        mx.moonep_dispatch(d, self.ws.buf, self.x, self.recv)
        mx.moonep_grouped_gemm(d, self.ws.buf, self.recv, self.w_home, self.w_slot, self.y)
        mx.moonep_combine(d, self.ws.buf, self.y, self.gates, self.out)
        torch.cuda.synchronize()

    def check_all_guards(self):
        w = self.w
        self.check_guards(self.w_slot_full, w.R * w.B * w.H * w.Hp, 0x7F7F, "w_slot")
        self.check_guards(self.recv_full, w.N * w.H, 0x7F7F, "recv")
        self.check_guards(self.y_full, w.N * w.Hp, 0x7F7F, "y")
        self.check_guards(self.out_full, w.R * w.S * w.Hp, 0x7F7F, "out")


def host_bits(t: torch.Tensor) -> np.ndarray:
    return syn.bf16_bits(t.cpu())
