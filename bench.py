"""Benchmark of the MoonEP layer path on GB300.

One step = one pass of the whole path over one batch of synthetic routing:
moonep_plan -> moonep_prefetch_weights -> moonep_dispatch -> moonep_grouped_gemm
-> moonep_combine -> moonep_reduce_grad, all on one CUDA stream with every
input already resident in HBM.  Timed steps rotate through the routing
imbalance sweep maxvio in {0.2, 1, 10, 20} (the pages' benchmark setting,
"Moonshot AI 开源 MoonEP", section 与 DeepEP v2 的基准测试), shape R=8 simulated
ranks, E=384, B=48, K=8, S=8192, H=7168, H'=2048.

Metric: routed token-copies per second, N = R*S*K copies per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the path has no data exchange on one GPU); rank 0 prints one
JSON line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

# BLAS threads for the oracle legs (CPU baseline, reference arm): every host
# core, set before NumPy loads its BLAS
HOST_THREADS = os.cpu_count() or 1
for _var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ[_var] = str(HOST_THREADS)

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "routed token-copies/sec (plan+permute+GEMM+combine) vs maxvio; % HBM & bf16 roofline"
UNIT = "token-copies/s"
SWEEP = (0.2, 1.0, 10.0, 20.0)
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _profile_workload():
    from perfectly_balanced_token_gb300 import synthetic as syn
    # the pages shape's H, H', K with fewer experts and tokens: a few GB on the
    # device; ~4k rows per group, so the plans pick 256-row work tiles
    return syn.Workload("profile-sized", R=8, E=16, B=2, K=8, S=1024, H=7168, Hp=2048)


def _profile128_workload():
    from perfectly_balanced_token_gb300 import synthetic as syn
    # as above with E=64: ~0.9k rows per group, so the plans pick 128-row work
    # tiles (the GEMM variant the pages shape uses)
    return syn.Workload("profile-sized-128", R=8, E=64, B=8, K=8, S=1024, H=7168, Hp=2048)


def _profile_k3_workload():
    from perfectly_balanced_token_gb300 import synthetic as syn
    # the K3 shape's per-rank structure (14 experts per rank, K=16, S=1024, H=4096,
    # H'=1024, ~1.2k rows per group) on 8 ranks instead of 64: about 2 GB on the device
    return syn.Workload("profile-sized-k3", R=8, E=112, B=14, K=16, S=1024, H=4096, Hp=1024)


def _pages():
    from perfectly_balanced_token_gb300 import synthetic as syn
    return syn.PAGES


def _k3():
    from perfectly_balanced_token_gb300 import synthetic as syn
    return syn.K3


WORKLOADS = {"pages": _pages, "k3": _k3, "profile": _profile_workload,
             "profile128": _profile128_workload, "profile_k3": _profile_k3_workload}
DEFAULT_SWEEP = {"pages": SWEEP, "k3": (1.0, 10.0), "profile": (1.0,), "profile128": (1.0,),
                 "profile_k3": (1.0,)}


def measured_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from an ncu capture recorded under
    profiles/, or None if there is none or the GEMM code changed since."""
    p = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    src = os.path.join(ROOT, "perfectly_balanced_token_gb300", "csrc", "gemm.cu")
    if not (os.path.exists(p) and os.path.exists(src)):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("gemm_cu_code_sha256") != source_digest(src):
        return None
    return rec


def source_digest(path: str) -> str:
    """SHA-256 of a CUDA source with its // comments and blank lines removed, so
    that a recorded capture stays valid across comment-only edits."""
    import hashlib
    import re
    lines = []
    with open(path, encoding="utf-8") as f:
        for line in f:
            code = re.sub(r"\s*//.*$", "", line.rstrip("\n")).rstrip()
            if code:
                lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, world: int, device) -> float:
    """Max over ranks (one all-reduce on a scalar); identity for one rank."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(w, maxvios):
    return {"workload": f"{w.name}: R={w.R} E={w.E} B={w.B} K={w.K} S={w.S} H={w.H} H'={w.Hp}",
            "R": w.R, "E": w.E, "B": w.B, "K": w.K, "S": w.S, "H": w.H, "Hp": w.Hp,
            "mode": "training" if w.mode == 0 else "inference",
            "maxvio_sweep": list(maxvios),
            "step": "plan+prefetch+dispatch+grouped_gemm+combine+reduce_grad",
            "l2": "256 MiB L2 flush write between timed steps; x, recv, W and grads exceed L2",
            "parallelism": "replicas (R ranks simulated on each GPU)"}


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampled every 50 ms.  Started before the warm-up (its own
    start-up must not overlap the timed region); summary() keeps only the
    samples taken inside the timed window (plus one sampling interval on each
    side, so that a short window still gets a sample)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, gpu_index: int):
        self.proc = None
        self.reader = None
        self.gpu = gpu_index
        self.lines = []

    def command(self):
        return ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)]

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(self.command(), stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # drain the pipe as lines arrive: a full pipe would stall the sampler
        # long before a multi-minute run ends
        self.reader = threading.Thread(target=self._drain, args=(self.proc.stdout,), daemon=True)
        self.reader.start()

    def _drain(self, pipe):
        for line in pipe:
            line = line.strip()
            if line:
                self.lines.append(line)

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.reader.join(timeout=5)
        self.proc = None

    def summary(self, t0: float, t1: float):
        import datetime
        sm, mx, reasons = [], [], set()
        for line in self.lines:
            parts = [q.strip() for q in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, cmax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            pad = self.INTERVAL_MS / 1000.0
            if not (t0 - pad <= ts <= t1 + pad):
                continue
            sm.append(clk)
            mx.append(cmax)
            for n, v in zip(self.REASONS, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def run_ours(args):
    import torch

    import perfectly_balanced_token_gb300 as mx
    from perfectly_balanced_token_gb300 import synthetic as syn

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mx.library()

    w = WORKLOADS[args.workload]()
    sweep = tuple(args.maxvio) if args.maxvio else DEFAULT_SWEEP.get(args.workload, SWEEP)
    N = w.N
    st = torch.cuda.current_stream()

    routings = [syn.routing_for(w, mv, seed=0) for mv in sweep]
    measured_mv = [syn.input_skew(r.idx, w.E) for r in routings]
    idx = [torch.from_numpy(r.idx).to(dev) for r in routings]
    gates = [torch.from_numpy(r.gates).to(dev) for r in routings]
    x = syn.normal_bf16((w.R, w.S, w.H), 1.0, 1, dev)
    w_home = syn.normal_bf16((w.E, w.H, w.Hp), 0.02, 2, dev)
    w_slot = torch.zeros(w.R * w.B * w.H * w.Hp, dtype=torch.bfloat16, device=dev)
    recv = torch.empty(N * w.H, dtype=torch.bfloat16, device=dev)
    y = torch.empty(N * w.Hp, dtype=torch.bfloat16, device=dev)
    out = torch.empty(w.R * w.S * w.Hp, dtype=torch.bfloat16, device=dev)
    g_home = syn.normal_f32((w.E, w.H, w.Hp), 1.0, 3, dev)
    g_slot = syn.normal_f32((w.R, w.B, w.H, w.Hp), 1.0, 4, dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    names = ("plan", "prefetch", "dispatch", "gemm", "combine", "reduce_grad")
    clocks = ClockSampler(local)
    clocks.start()  # before the warm-up, so nvidia-smi's start-up is over by the timed region

    bwd = {}  # backward buffers, allocated only when the training step is timed

    def time_policy(policy, warmup, steps, training=False):
        """Warm up eagerly, capture one CUDA graph per (routing, segment), then
        time `steps` steps of graph replays with events between segments.  The
        forward step is plan .. combine + reduce_grad; a training step inserts
        the backward (combine backward, the two GEMM gradients, dispatch
        backward) before reduce_grad."""
        d = mx.dims(w.R, w.E, w.B, w.K, w.S, w.H, w.Hp, w.mode, policy, args.gemm_rows)
        ws = mx.PlanWorkspace(d, device=dev)

        def calls(j):
            # stream=None: the current stream (the capture stream while capturing)
            fwd = (
                lambda: mx.moonep_plan(d, idx[j], ws.buf),
                lambda: mx.moonep_prefetch_weights(d, ws.buf, w_home, w_slot),
                lambda: mx.moonep_dispatch(d, ws.buf, x, recv),
                lambda: mx.moonep_grouped_gemm(d, ws.buf, recv, w_home, w_slot, y),
                lambda: mx.moonep_combine(d, ws.buf, y, gates[j], out),
            )
            back = ()
            if training:
                b = bwd
                back = (
                    lambda: mx.moonep_combine_backward(d, ws.buf, y, gates[j], b["dout"], b["dy"],
                                                       b["dgates"]),
                    lambda: mx.moonep_grouped_gemm_dx(d, ws.buf, b["dy"], w_home, w_slot,
                                                      b["drecv"]),
                    lambda: mx.moonep_grouped_gemm_dw(d, ws.buf, recv, b["dy"], g_home, g_slot),
                    lambda: mx.moonep_dispatch_backward(d, ws.buf, b["drecv"], b["dx"]),
                )
            return fwd + back + (lambda: mx.moonep_reduce_grad(d, ws.buf, g_home, g_slot),)
        nseg = len(calls(0))

        for i in range(warmup):
            for c in calls(i % len(sweep)):
                c()
        torch.cuda.synchronize()
        status = mx.moonep_read_status(d, ws.buf)
        if status:
            raise RuntimeError(f"device status {status:#x}: {mx.status_string(status)}")

        counters = []  # per-maxvio plan counters (outside the timed region)
        for j in range(len(sweep)):
            mx.moonep_plan(d, idx[j], ws.buf, st)
            c = ws.view("counters", (8,)).cpu().tolist()
            n_recv = ws.view("n_recv", (w.R,)).cpu()
            payload = 2 * w.H
            counters.append({"fills": c[0], "mtiles": c[1], "occupied_slots": c[2],
                             "reduced_experts": c[3], "max_redundant_per_rank": int(n_recv.max()),
                             "link_bytes_per_entry": c[4] * (payload + 4),
                             "link_bytes_send_once": c[5] * payload + c[4] * 4,
                             "gemm_tile_rows": c[7]})

        # the timed loop only replays graphs, so host-side enqueue cost never
        # shows up between the per-segment events
        graphs, graph_launches = [], []
        for j in range(len(sweep)):
            gj, lj = [], []
            for c in calls(j):
                g = torch.cuda.CUDAGraph()
                n0 = mx.moonep_launch_count()
                with torch.cuda.graph(g):
                    c()
                lj.append(mx.moonep_launch_count() - n0)
                gj.append(g)
            graphs.append(gj)
            graph_launches.append(lj)
        for j in range(len(sweep)):  # first replay uploads each graph
            for g in graphs[j]:
                g.replay()
        torch.cuda.synchronize()

        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nseg + 1)] for _ in range(steps)]
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        launches = 0
        t0 = time.time()
        for i in range(steps):
            j = i % len(sweep)
            flush.fill_(float(i))  # evict L2 between steps (not inside a step's events)
            for k in range(nseg):
                evs[i][k].record()
                graphs[j][k].replay()
            evs[i][nseg].record()
            launches += sum(graph_launches[j])
        torch.cuda.synchronize()
        t1 = time.time()
        if world > 1:
            dist.barrier()
        status = mx.moonep_read_status(d, ws.buf)
        if status:
            raise RuntimeError(f"device status after the timed steps {status:#x}: "
                               f"{mx.status_string(status)}")
        seg = np.array([[evs[i][k].elapsed_time(evs[i][k + 1]) for k in range(nseg)]
                        for i in range(steps)])  # ms
        return d, ws, seg, counters, launches, (t0, t1)

    headline_rows = [0, 2, 3, 4]

    def per_maxvio(seg_, counters_):
        out_ = []
        sm = seg_.sum(axis=1)
        for j, mv in enumerate(sweep):
            rows = [i for i in range(seg_.shape[0]) if i % len(sweep) == j]
            if not rows:
                continue
            ms = float(sm[rows].mean())
            hl = float(seg_[rows][:, headline_rows].sum(axis=1).mean())
            out_.append({"maxvio_target": mv, "maxvio": round(measured_mv[j], 4),
                         "value": N / (ms / 1e3), "ms_per_step": ms,
                         "value_plan_permute_gemm_combine": N / (hl / 1e3),
                         "breakdown_ms": {n: float(seg_[rows][:, k].mean())
                                          for k, n in enumerate(names)},
                         **counters_[j]})
        return out_

    d, ws, seg, counters, launches, window = time_policy(0, args.warmup, args.steps)
    step_ms = seg.sum(axis=1)
    total_ms = reduce_max(float(step_ms.sum()), world, dev)
    t_wall = window[1] - window[0]
    per_mv = per_maxvio(seg, counters)
    policy1 = None
    if not args.no_policy_sweep:
        _, _, seg1, counters1, _, _ = time_policy(1, 1, args.steps)
        ms1 = reduce_max(float(seg1.sum()), world, dev)
        policy1 = {"planner": "largest first (dims.policy = 1)",
                   "value": N * args.steps * world / (ms1 / 1e3),
                   "ms_per_step": ms1 / args.steps,
                   "sweep": per_maxvio(seg1, counters1)}

    training = None
    if not args.no_training:
        bwd.update(
            dout=syn.normal_bf16((w.R, w.S, w.Hp), 1.0, 5, dev).view(-1),
            dy=torch.empty(N * w.Hp, dtype=torch.bfloat16, device=dev),
            dgates=torch.empty(N, dtype=torch.float32, device=dev),
            drecv=torch.empty(N * w.H, dtype=torch.bfloat16, device=dev),
            dx=torch.empty(w.R * w.S * w.H, dtype=torch.bfloat16, device=dev))
        _, _, segt, _, _, _ = time_policy(0, 1, args.steps, training=True)
        tnames = names[:5] + ("combine_backward", "gemm_dx", "gemm_dw", "dispatch_backward",
                              "reduce_grad")
        mst = reduce_max(float(segt.sum()), world, dev)
        bd = {n: float(segt[:, k].mean()) for k, n in enumerate(tnames)}
        fl = 2.0 * N * w.H * w.Hp
        training = {"step": "forward (plan .. combine) + combine backward + input-gradient GEMM "
                            "+ weight-gradient GEMM + dispatch backward + reduce_grad",
                    "value": N * args.steps * world / (mst / 1e3), "ms_per_step": mst / args.steps,
                    "breakdown_ms": bd,
                    "gemm_dx_tflops": fl / (bd["gemm_dx"] / 1e3) / 1e12,
                    "gemm_dw_tflops": fl / (bd["gemm_dw"] / 1e3) / 1e12}
        for b_ in list(bwd):
            del bwd[b_]
        torch.cuda.empty_cache()

    send_once = None if args.no_send_once else time_send_once(
        mx, torch, d, ws, w, sweep, idx, x, gates, recv, flush, args.warmup, args.steps)

    # e2e: host buffers through the same C ABI, copies inside the timed region
    e2e = None if args.no_e2e else run_e2e(args, mx, syn, torch, d, w, routings, ws, w_home, w_slot,
                                            g_home, g_slot, dev, st, world)
    clocks.stop()
    clk = clocks.summary(*window)

    peaks, peak_src = load_peaks()
    bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gemm_ms = float(seg[:, 3].mean())
    flops = 2.0 * N * w.H * w.Hp
    achieved_tf = flops / (gemm_ms / 1e3) / 1e12
    # the variant the plans chose (the other one is launched and returns at once)
    rows_chosen = sorted({c["gemm_tile_rows"] for c in counters})
    wide = w.Hp % 256 == 0  # 256-wide column tiles: 256-row tiles run on CTA pairs
    gemm_kernel = "+".join(("k_ggemm_2sm" if wide else "k_ggemm_m256") if r == 256 else "k_ggemm_m128"
                           for r in rows_chosen)
    traffic = measured_traffic(gemm_kernel) if args.workload == "pages" else None
    occ = np.mean([c["occupied_slots"] for c in counters])
    red = np.mean([c["reduced_experts"] for c in counters])
    hh = w.H * w.Hp
    roofline = {"kernel": f"{gemm_kernel} (moonep_grouped_gemm)", "bound": "tensor",
                "achieved": achieved_tf, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": achieved_tf / bf16_peak, "peak_source": f"bf16_tflops ({peak_src}, burst)",
                "traffic": traffic["bytes_per_launch"] if traffic else None,
                "traffic_source": traffic["source"] if traffic else None,
                "traffic_method": traffic.get("method") if traffic else None,
                "algorithmic_flops_per_launch": flops, "ms_per_launch": gemm_ms,
                # recv read once, each used weight panel once, Y written once
                "algorithmic_bytes_per_launch": float(N * w.H * 2 + (w.E + occ) * hh * 2
                                                      + N * w.Hp * 2)}
    algo_bytes = {
        "dispatch": w.R * w.S * w.H * 2 + N * w.H * 2 + N * 4,
        "combine": N * w.Hp * 2 + N * 8 + w.R * w.S * w.Hp * 2,
        "prefetch": occ * hh * 2 * 2,
        "reduce_grad": (occ + red) * hh * 4 * 2,
    }
    col = {"dispatch": 2, "combine": 4, "prefetch": 1, "reduce_grad": 5}
    rooflines = {}
    for k, b in algo_bytes.items():
        ms = float(seg[:, col[k]].mean())
        gbs = b / (ms / 1e3) / 1e9 if ms > 0 else 0.0
        rooflines[k] = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                        "frac": gbs / hbm_peak, "bytes_per_launch": b, "ms_per_launch": ms}
    rooflines["plan"] = {"bound": "latency", "us_per_launch": float(seg[:, 0].mean()) * 1e3}
    if training is not None:
        # the backward's streaming kernels against the same HBM peak
        tb = {"combine_backward": (2 * N + w.R * w.S) * w.Hp * 2 + N * 12,
              "dispatch_backward": (N + w.R * w.S) * w.H * 2 + N * 4}
        training["rooflines"] = {}
        for k, b in tb.items():
            ms = training["breakdown_ms"][k]
            gbs = b / (ms / 1e3) / 1e9 if ms > 0 else 0.0
            training["rooflines"][k] = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                                        "unit": "GB/s", "frac": gbs / hbm_peak,
                                        "bytes_per_launch": b, "ms_per_launch": ms}

    result = {
        "metric": METRIC, "value": N * args.steps * world / (total_ms / 1e3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, sweep),
        "value_plan_permute_gemm_combine": N * args.steps * world /
        (reduce_max(float(seg[:, headline_rows].sum()), world, dev) / 1e3),
        "sweep": per_mv, "e2e": e2e, "gpu_launches": launches,
        "roofline": roofline, "rooflines": rooflines, "clocks": clk,
        "wall_s_timed_region": t_wall, "timing": "CUDA events between CUDA-graph replays of each "
        "segment on the launching stream; gpu_launches counted from the captured graphs",
        "step_ms": [float(v) for v in step_ms],
        "planner": "Theorem 1 construction, fixed tie-break (dims.policy = 0)",
        "planner_largest_first": policy1,
        "training_step": training,
        "send_once_dispatch": send_once,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "pages":
        result["cpu_baseline"] = cpu_baseline(args.cpu_budget_s)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def time_send_once(mx, torch, d, ws, w, sweep, idx, x, gates, recv, flush, warmup, steps):
    """The send-once dispatch (send pass + receive copy) per routing, outside the
    timed step: one CUDA graph per routing, an L2 flush before every replay,
    CUDA events around it.  HBM bytes of the two passes on one GPU: x read once,
    one row written per (token, destination rank) pair, each later entry for
    the same rank read back and written again on the receiver, plus the route,
    destination, gate reads and weight writes (16 B per entry); the bytes that
    would cross ranks are the per-entry and send-once link figures."""
    recv_w = torch.empty(w.N, dtype=torch.float32, device=recv.device)
    rows = []
    for j, mv in enumerate(sweep):
        mx.moonep_plan(d, idx[j], ws.buf)
        route = ws.view("route", (w.N,))
        dups = int((route < 0).sum().item())
        c = ws.view("counters", (8,)).cpu().tolist()
        for _ in range(warmup):
            mx.moonep_dispatch_send_once(d, ws.buf, x, gates[j], recv, recv_w)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            mx.moonep_dispatch_send_once(d, ws.buf, x, gates[j], recv, recv_w)
        g.replay()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            flush.fill_(float(i))
            evs[i][0].record()
            g.replay()
            evs[i][1].record()
        torch.cuda.synchronize()
        ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
        payload = 2 * w.H
        hbm = w.R * w.S * payload + w.N * payload + dups * payload + 16 * w.N
        rows.append({"maxvio_target": mv, "ms": ms, "hbm_bytes": hbm,
                     "achieved_gbs": hbm / (ms / 1e3) / 1e9,
                     "receiver_copies": dups,
                     "link_bytes_per_entry": c[4] * (payload + 4),
                     "link_bytes_send_once": c[5] * payload + c[4] * 4})
    status = mx.moonep_read_status(d, ws.buf)
    if status:
        raise RuntimeError(f"device status after the send-once dispatch {status:#x}: "
                           f"{mx.status_string(status)}")
    return {"call": "moonep_dispatch_send_once (k_send + k_receive_copy)", "sweep": rows}


def run_e2e(args, mx, syn, torch, d, w, routings, ws, w_home, w_slot, g_home, g_slot, dev, st,
            world, verify_steps=0):
    """Same step, but x / routing / gates start in pinned host memory and the
    combined output is read back to pinned host memory every step.

    Two schedules, both with every step's copies inside the timed region:
    `serial` issues copy-in, the step and copy-out on one stream; `pipelined`
    (the reported value) issues the copies on two more streams (inputs, and
    outputs) into double buffers, so step i+1's inputs travel and step i-1's
    output returns while step i computes, as a data loader feeding this layer
    would.

    With verify_steps > 0 nothing is timed: that many steps go through the
    pipelined schedule with inputs that change from step to step (three token
    matrices and the routings in turn, so no two steps that share a buffer
    have the same inputs), every step's read-back is kept, and the result
    counts the steps whose output differs from the same step run alone on one
    stream."""
    N = w.N
    nx = 3 if verify_steps else 1
    x_h = [syn.normal_bf16((w.R, w.S, w.H), 1.0, 1 + i, "cpu").pin_memory() for i in range(nx)]
    idx_h = [torch.from_numpy(r.idx).pin_memory() for r in routings]
    g_h = [torch.from_numpy(r.gates).pin_memory() for r in routings]
    out_h = [torch.empty(w.R * w.S * w.Hp, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x_h[0], device=dev) for _ in range(2)]
    kept = None  # per-step copies of the read-backs (verification only)
    idx_d = [torch.empty_like(idx_h[0], device=dev) for _ in range(2)]
    g_d = [torch.empty_like(g_h[0], device=dev) for _ in range(2)]
    out = [torch.empty(w.R * w.S * w.Hp, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    recv = torch.empty(N * w.H, dtype=torch.bfloat16, device=dev)
    y = torch.empty(N * w.Hp, dtype=torch.bfloat16, device=dev)
    # runs of at most eight steps (~0.1 s at the pages shape): a longer run is
    # more often caught by a transient slowdown of the shared host link
    steps = max(2, min(args.steps, 8))
    cs = torch.cuda.Stream(device=dev)   # copies in
    cos = torch.cuda.Stream(device=dev)  # copies out: the link carries both directions at once
    Ev = torch.cuda.Event

    def copy_in(i, stream):
        b, j = i % 2, i % len(routings)
        with torch.cuda.stream(stream):
            x_d[b].copy_(x_h[i % nx], non_blocking=True)
            idx_d[b].copy_(idx_h[j], non_blocking=True)
            g_d[b].copy_(g_h[j], non_blocking=True)

    def compute(i):
        b = i % 2
        mx.moonep_plan(d, idx_d[b], ws.buf, st)
        mx.moonep_prefetch_weights(d, ws.buf, w_home, w_slot, st)
        mx.moonep_dispatch(d, ws.buf, x_d[b], recv, st)
        mx.moonep_grouped_gemm(d, ws.buf, recv, w_home, w_slot, y, st)
        mx.moonep_combine(d, ws.buf, y, g_d[b], out[b], st)

    def copy_out(i, stream):
        with torch.cuda.stream(stream):
            out_h[i % 2].copy_(out[i % 2], non_blocking=True)
            if kept is not None:
                kept[i].copy_(out[i % 2], non_blocking=True)

    def serial(n):
        e0, e1 = Ev(enable_timing=True), Ev(enable_timing=True)
        e0.record(st)
        for i in range(n):
            copy_in(i, st)
            compute(i)
            mx.moonep_reduce_grad(d, ws.buf, g_home, g_slot, st)
            copy_out(i, st)
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def pipelined(n, detail=None):
        h2d = [Ev() for _ in range(2)]        # inputs of buffer b are on the device
        used = [Ev() for _ in range(2)]       # the step that read buffer b is past combine
        ready = [Ev() for _ in range(2)]      # out[b] holds a finished step
        d2h = [Ev() for _ in range(2)]        # out[b] has been read back
        e0, e1, end = Ev(enable_timing=True), Ev(enable_timing=True), Ev()
        # where each step's time went: compute and reduce_grad on the compute
        # stream, each copy on the copy stream
        t_c = [(Ev(enable_timing=True), Ev(enable_timing=True)) for _ in range(n)]
        t_in = [(Ev(enable_timing=True), Ev(enable_timing=True)) for _ in range(n)]
        t_out = [(Ev(enable_timing=True), Ev(enable_timing=True)) for _ in range(n)]
        e0.record(cs)
        t_in[0][0].record(cs)
        copy_in(0, cs)
        t_in[0][1].record(cs)
        h2d[0].record(cs)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                if i >= 1:
                    cs.wait_event(used[(i + 1) % 2])
                t_in[i + 1][0].record(cs)
                copy_in(i + 1, cs)
                t_in[i + 1][1].record(cs)
                h2d[(i + 1) % 2].record(cs)
            st.wait_event(h2d[b])
            if i >= 2:
                st.wait_event(d2h[b])
            t_c[i][0].record(st)
            compute(i)
            used[b].record(st)
            ready[b].record(st)
            mx.moonep_reduce_grad(d, ws.buf, g_home, g_slot, st)
            t_c[i][1].record(st)
            cos.wait_event(ready[b])
            t_out[i][0].record(cos)
            copy_out(i, cos)
            t_out[i][1].record(cos)
            d2h[b].record(cos)
        end.record(st)
        cs.wait_event(end)
        cs.wait_event(d2h[(n - 1) % 2])  # the last read-back (read-backs run in order)
        e1.record(cs)
        torch.cuda.synchronize()
        if detail is not None:
            span = lambda p: p[0].elapsed_time(p[1])
            med = lambda xs: float(np.median(xs))
            detail.update({
                "compute_ms_median": med([span(p) for p in t_c]),
                "copy_in_ms_median": med([span(p) for p in t_in]),
                "copy_out_ms_median": med([span(p) for p in t_out]),
                # compute-stream idle time between one step's end and the next's start
                "idle_between_steps_ms": [round(t_c[i - 1][1].elapsed_time(t_c[i][0]), 3)
                                          for i in range(1, n)],
                "first_step_start_ms": e0.elapsed_time(t_c[0][0]),
            })
        return e0.elapsed_time(e1)

    if verify_steps:
        kept = [torch.empty_like(out_h[0]).pin_memory() for _ in range(verify_steps)]
        pipelined(verify_steps)
        bad = 0
        for i in range(verify_steps):
            copy_in(i, st)
            compute(i)
            torch.cuda.synchronize()
            bad += int(not torch.equal(out[i % 2].cpu(), kept[i]))
        return {"steps": verify_steps, "mismatches": bad}

    serial(2)
    pipelined(2)
    # each schedule is timed seven times and the median run reported: the host
    # copies share the host's memory and link with other work on the machine,
    # and a run that catches a transient slowdown of its copies can take
    # tens of milliseconds longer
    reps = 7
    serial_ms = [reduce_max(serial(steps), world, dev) for _ in range(reps)]
    runs = []
    for _ in range(reps):
        det = {}
        runs.append((reduce_max(pipelined(steps, det), world, dev), det))
    ms_serial = sorted(serial_ms)[reps // 2]
    ms, detail = sorted(runs, key=lambda r: r[0])[reps // 2]
    h2d_bytes = x_h[0].numel() * 2 + idx_h[0].numel() * 4 + g_h[0].numel() * 4
    return {"value": N * steps * world / (ms / 1e3), "unit": UNIT, "steps": steps,
            "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(out_h[0].numel() * 2),
            "schedule": "copies in and out on two more streams, double-buffered, overlapping the "
                        "previous and next steps' compute; median of seven timed runs",
            "runs_ms": [round(r[0], 3) for r in runs],
            "serial_value": N * steps * world / (ms_serial / 1e3),
            "serial_schedule": "copy-in, step, copy-out on one stream; median of seven timed runs",
            "serial_runs_ms": [round(x, 3) for x in serial_ms],
            "pipelined_detail": detail}


# ----------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ----------------------------------------------------------------------------
class OracleSample:
    """Time the oracle (as it stands) on a bounded sample of the workload.

    Sample: the full plan (histogram, constructive plan, every destination)
    over all N copies of one maxvio=1 routing, then permute + expert GEMM +
    combine for the copies of a few experts, scaled to all N copies by copy
    count.  Inputs are drawn once; run() returns (copies_per_s, description,
    seconds spent)."""

    def __init__(self, seed: int = 0):
        from oracle import planner as oplanner
        from perfectly_balanced_token_gb300 import synthetic as syn

        self.w = w = syn.PAGES
        self.od = oplanner.Dims(R=w.R, E=w.E, B=w.B, K=w.K, S=w.S, H=w.H, Hp=w.Hp)
        self.rt = syn.routing_for(w, 1.0, seed=seed)
        self.x = syn.bf16_bits(syn.normal_bf16((w.R, w.S, w.H), 1.0, 1, "cpu")).reshape(-1, w.H)
        self.seed = seed

    def run(self, budget_s: float):
        from oracle import layer as olayer
        from oracle import planner as oplanner
        from perfectly_balanced_token_gb300 import synthetic as syn

        w = self.w
        t0 = time.perf_counter()
        oplanner.full_plan(self.rt.idx, self.od)
        t_plan = time.perf_counter() - t0
        rng = np.random.default_rng(self.seed)
        copies, t_rest, experts = 0, 0.0, []
        while t_plan + t_rest < budget_s and len(experts) < w.E:
            e = int(rng.integers(0, w.E))
            if e in experts:
                continue
            experts.append(e)
            wb = syn.bf16_bits(syn.normal_bf16((w.H, w.Hp), 0.02, 100 + e, "cpu"))
            t1 = time.perf_counter()
            # the oracle's own per-expert step: gather the copies' token rows
            # (permute) and multiply by the expert's weights
            cids, yb = olayer.expert_outputs(self.x, lambda _e: wb, self.rt.idx, self.od,
                                             experts=[e])[e]
            # combine's share for these copies: the oracle's fp64 gate-weighted
            # accumulation and bf16 rounding (combine itself needs every copy)
            g = self.rt.gates.reshape(-1)[cids].astype(np.float64)[:, None]
            olayer.to_bf16(g * olayer.bf16_to_f64(yb))
            t_rest += time.perf_counter() - t1
            copies += cids.size
        per_copy = t_plan / w.N + t_rest / max(copies, 1)
        desc = (f"oracle full plan over all {w.N} copies (maxvio 1) in {t_plan:.2f} s; "
                f"permute+GEMM+combine for {copies} copies of {len(experts)} experts in "
                f"{t_rest:.2f} s; scaled per copy")
        return 1.0 / per_copy, desc, t_plan + t_rest


def blas_threads() -> int:
    """Threads NumPy's BLAS uses (threadpoolctl where installed, else the
    environment variable set at start-up)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return int(os.environ.get("OPENBLAS_NUM_THREADS", HOST_THREADS))


class _SlotRows(dict):
    """The occupied slots' gradient rows keyed by (rank, slot); assigning a
    scalar fills the row in place, as it does for a slice of one array."""

    def __setitem__(self, key, value):
        dict.__getitem__(self, key)[...] = value


def oracle_reduce_sample(seed: int = 0):
    """The oracle's reduce_grad timed on its own on the occupied slots of the
    pages-shaped maxvio-1 plan: every expert holding a slot and every occupied
    slot, fp32 N(0,1) rows (the experts renumbered so only they are held)."""
    from types import SimpleNamespace

    from oracle import layer as olayer
    from oracle import planner as oplanner
    from perfectly_balanced_token_gb300 import synthetic as syn

    w = syn.PAGES
    od = oplanner.Dims(R=w.R, E=w.E, B=w.B, K=w.K, S=w.S, H=w.H, Hp=w.Hp)
    plan = oplanner.build_plan(syn.routing_for(w, 1.0, seed=seed).idx, od)
    occ = [(u, j, int(plan.slot_expert[u, j])) for u in range(w.R) for j in range(w.B)
           if plan.slot_expert[u, j] >= 0]
    experts = sorted({e for _, _, e in occ})
    local = {e: i for i, e in enumerate(experts)}
    rng = np.random.default_rng(seed)
    g_home = rng.standard_normal((len(experts), w.H, w.Hp), dtype=np.float32)
    slots = _SlotRows({(u, j): rng.standard_normal((w.H, w.Hp), dtype=np.float32)
                       for u, j, _ in occ})
    se = np.full((w.R, w.B), -1, dtype=np.int64)
    for u, j, e in occ:
        se[u, j] = local[e]
    view = SimpleNamespace(dims=SimpleNamespace(E=len(experts), R=w.R, B=w.B), slot_expert=se)
    t0 = time.perf_counter()
    olayer.reduce_grad(g_home, slots, view, experts=range(len(experts)))
    sec = time.perf_counter() - t0
    nbytes = (len(experts) + len(occ)) * w.H * w.Hp * 4 * 2
    return {"ms": sec * 1e3, "experts": len(experts), "occupied_slots": len(occ),
            "bytes": nbytes, "gbs": nbytes / sec / 1e9,
            "sample": "oracle reduce_grad of the maxvio-1 plan's occupied slots into their "
                      "home experts (home rows read and written, slots read and zeroed)"}


def cpu_baseline(budget_s: float):
    v, desc, _ = OracleSample().run(budget_s)
    return {"value": v, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": desc, "host_cores": os.cpu_count(),
            "threads_note": "OMP_NUM_THREADS / OPENBLAS_NUM_THREADS set to the host core count",
            "reduce_grad": oracle_reduce_sample()}


def run_reference(args):
    """The oracle timed as it stands on the host cores.  One step is one bounded
    sample of the pages-shaped workload (the full plan over all N copies, then
    permute + expert GEMM + combine for the copies of as many experts as fit
    the per-step budget); `ms_per_step` is the sample's measured wall time and
    `value` the copies per second that sample sustains, scaled per copy."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import perfectly_balanced_token_gb300.synthetic as syn
    w = syn.PAGES
    budget = max(2.0, args.cpu_budget_s / max(1, args.steps + args.warmup))
    sample = OracleSample()
    for _ in range(args.warmup):
        sample.run(budget)
    vals, secs = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, desc, s = sample.run(budget)
        vals.append(v)
        secs.append(s)
    wall = time.perf_counter() - t0
    v = float(np.mean(vals))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(secs)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, (1.0,)),
        "step": "one bounded sample of the workload per step (last: " + desc + ")",
        "wall_s_timed_region": wall,
        "cpu_baseline": {"kind": "oracle", "cores": blas_threads(), "host_cores": os.cpu_count(),
                         "sample": desc, "value": v},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--maxvio", type=float, nargs="*", default=None)
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-policy-sweep", action="store_true",
                    help="skip timing the largest-first planner policy")
    ap.add_argument("--no-training", action="store_true",
                    help="skip timing the training step (forward + backward)")
    ap.add_argument("--no-send-once", action="store_true",
                    help="skip timing the send-once dispatch")
    ap.add_argument("--gemm-rows", type=int, choices=(0, 128, 256), default=0,
                    help="GEMM work-tile height: 0 = chosen per plan by the cost model (the "
                         "default), 128 or 256 = fixed (to profile one GEMM variant)")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="pages",
                    help="pages = the headline configuration; the others are smaller cases "
                         "of the same kernels for profiling")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
