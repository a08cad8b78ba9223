"""Offline tuning of the grouped GEMM's cost model (csrc/gemm_cost.cuh).

  python -m perfectly_balanced_token_gb300.tuning.fit_gemm_cost measure   # on a GPU
  python -m perfectly_balanced_token_gb300.tuning.fit_gemm_cost fit       # anywhere

`measure` plans a set of synthetic workloads whose rows per (rank, weight row)
group range from a few hundred to several thousand, times the forward grouped
GEMM with the work-tile height fixed at 128 and at 256 rows (CUDA events,
L2 flushed and a 30 ms idle gap before every launch, the two heights launched
alternately, median of several launches), and stores the
times with the tile and group counts of each plan in gemm_cost_measurements.json.

`fit` fits, per tile height, non-negative coefficients of the model documented
in gemm_cost.cuh (time / ((K/64)(N/256)) against tile, group and length
terms), weighting each workload by the inverse of its time, prints each
workload's measured and predicted times and the choice, and rewrites
gemm_cost.cuh with the coefficients.
"""
from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
DATA = os.path.join(HERE, "gemm_cost_measurements.json")
HEADER = os.path.join(os.path.dirname(HERE), "csrc", "gemm_cost.cuh")

# (name, R, E, B, K, S, H, Hp, maxvio)
WORKLOADS = [
    ("pages-mv1", 8, 384, 48, 8, 8192, 7168, 2048, 1.0),
    ("pages-mv20", 8, 384, 48, 8, 8192, 7168, 2048, 20.0),
    ("e384-s512", 8, 384, 48, 8, 512, 7168, 2048, 1.0),
    ("e384-s1024", 8, 384, 48, 8, 1024, 7168, 2048, 1.0),
    ("e256", 8, 256, 32, 8, 1024, 7168, 2048, 1.0),
    ("e128", 8, 128, 16, 8, 1024, 7168, 2048, 1.0),
    ("e64", 8, 64, 8, 8, 1024, 7168, 2048, 1.0),
    ("e48", 8, 48, 6, 8, 1024, 7168, 2048, 1.0),
    ("e24", 8, 24, 3, 8, 1024, 7168, 2048, 1.0),
    ("e16", 8, 16, 2, 8, 1024, 7168, 2048, 1.0),
    ("e16-mv10", 8, 16, 2, 8, 1024, 7168, 2048, 10.0),
    ("e8-k4", 8, 8, 1, 4, 2048, 7168, 2048, 1.0),
    ("e8-k4-s4096", 8, 8, 1, 4, 4096, 7168, 2048, 1.0),
    ("k3-mv1", 64, 896, 14, 16, 1024, 4096, 1024, 1.0),
    ("k3-mv10", 64, 896, 14, 16, 1024, 4096, 1024, 10.0),
    ("h4096-e256", 8, 256, 32, 8, 1024, 4096, 1024, 1.0),
    ("h4096-e64", 8, 64, 8, 8, 2048, 4096, 1024, 1.0),
    ("h4096-e32", 8, 32, 4, 8, 2048, 4096, 1024, 1.0),
    ("h4096-e16", 8, 16, 2, 8, 2048, 4096, 1024, 1.0),
]


def tile_counts(cu: np.ndarray):
    """Work tiles at both heights and non-empty groups, from cu_seqlens [R][E+B+1]."""
    rows = np.diff(cu.astype(np.int64), axis=1).reshape(-1)
    rows = rows[rows > 0]
    n128 = int(np.sum((rows + 127) // 128))
    rem = rows % 256
    n256f = int(np.sum(rows // 256 + (rem > 128)))
    n256h = int(np.sum((rem > 0) & (rem <= 128)))
    return n128, n256f, n256h, int(rows.size)


def measure(reps: int = 10):
    import torch

    sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
    import perfectly_balanced_token_gb300 as mx
    from perfectly_balanced_token_gb300 import synthetic as syn

    out = []
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    for name, R, E, B, K, S, H, Hp, mv in WORKLOADS:
        w = syn.Workload(name, R=R, E=E, B=B, K=K, S=S, H=H, Hp=Hp)
        rt = syn.tune_alpha(R, S, K, E, mv, seed=0)
        idx = torch.from_numpy(rt.idx).cuda()
        x = syn.normal_bf16((R, S, H), 1.0, 1, "cuda")
        wh = syn.normal_bf16((E, H, Hp), 0.02, 2, "cuda")
        wsl = torch.zeros(R * B * H * Hp, dtype=torch.bfloat16, device="cuda")
        recv = torch.empty(w.N * H, dtype=torch.bfloat16, device="cuda")
        y = torch.empty(w.N * Hp, dtype=torch.bfloat16, device="cuda")
        rec = {"name": name, "R": R, "E": E, "B": B, "K": K, "S": S, "H": H, "Hp": Hp,
               "maxvio": float(syn.input_skew(rt.idx, E))}
        # both heights planned up front, then launched alternately (ABBA...),
        # so that neither sees a warmer or more power-capped GPU than the other
        runs = {}
        for rows in (128, 256):
            d = mx.dims(R, E, B, K, S, H, Hp, 0, 0, rows)
            ws = mx.PlanWorkspace(d)
            mx.moonep_plan(d, idx, ws.buf)
            mx.moonep_prefetch_weights(d, ws.buf, wh, wsl)
            mx.moonep_dispatch(d, ws.buf, x, recv)
            runs[rows] = (d, ws)
        ts = {128: [], 256: []}
        for i in range(reps + 2):
            for rows in ((128, 256) if i % 2 == 0 else (256, 128)):
                d, ws = runs[rows]
                flush.fill_(i)
                # a short idle gap: every timed launch starts from the same
                # settled clock and power state instead of inheriting the
                # previous launch's
                torch.cuda.synchronize()
                time.sleep(0.03)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                mx.moonep_grouped_gemm(d, ws.buf, recv, wh, wsl, y)
                b.record()
                torch.cuda.synchronize()
                if i >= 2:
                    ts[rows].append(a.elapsed_time(b))
        for rows in (128, 256):
            d, ws = runs[rows]
            if mx.moonep_read_status(d, ws.buf) != 0:
                raise RuntimeError(f"{name}: status {mx.moonep_read_status(d, ws.buf)}")
            rec[f"ms{rows}"] = float(np.median(ts[rows]))
        cu = runs[128][1].tables()["cu_seqlens"]
        rec["n128"], rec["n256f"], rec["n256h"], rec["groups"] = tile_counts(cu)
        del runs
        print(json.dumps(rec), flush=True)
        out.append(rec)
        del x, wh, wsl, recv, y, idx
        torch.cuda.empty_cache()
    with open(DATA, "w") as f:
        json.dump(out, f, indent=1)


def _features(recs):
    n128 = np.array([r["n128"] for r in recs], np.float64)
    nf = np.array([r["n256f"] for r in recs], np.float64)
    nh = np.array([r["n256h"] for r in recs], np.float64)
    g = np.array([r["groups"] for r in recs], np.float64)
    waves = n128 * np.array([r["Hp"] / 256.0 for r in recs]) / 152.0
    return np.c_[n128, g, n128 * waves], np.c_[nf, nh, g, nf * waves]


COEFF_NAMES = ("kCostA128", "kCostG128", "kCostW128", "kCostA256Full", "kCostA256Half",
               "kCostG256", "kCostW256")


def fit_coefficients(recs):
    """Non-negative least squares per tile height, relative errors (each
    workload weighted by 1 / its time).  Returns (coefficients by name, table
    rows (name, rows per group, ms128, predicted, ms256, predicted, best, pick))."""
    from scipy.optimize import nnls

    unit = np.array([(r["H"] / 64) * (r["Hp"] / 256) for r in recs])
    y128 = np.array([r["ms128"] * 1e3 for r in recs]) / unit
    y256 = np.array([r["ms256"] * 1e3 for r in recs]) / unit
    X128, X256 = _features(recs)
    c128, _ = nnls(X128 / y128[:, None], np.ones_like(y128))
    c256, _ = nnls(X256 / y256[:, None], np.ones_like(y256))
    p128, p256 = X128 @ c128, X256 @ c256
    rows = []
    for r, pa, pb, u in zip(recs, p128, p256, unit):
        rows.append((r["name"], r["R"] * r["S"] * r["K"] / r["groups"], r["ms128"], pa * u / 1e3,
                     r["ms256"], pb * u / 1e3, 128 if r["ms128"] <= r["ms256"] else 256,
                     256 if pb < pa else 128))
    return dict(zip(COEFF_NAMES, list(c128) + list(c256))), rows


def fit():
    recs = json.load(open(DATA))
    coeffs, rows = fit_coefficients(recs)
    print(f"{'workload':16s} {'rows/grp':>8s} {'ms128':>8s} {'pred':>8s} {'ms256':>8s} {'pred':>8s}  best model")
    for name, rpg, a, pa, b, pb, best, pick in rows:
        print(f"{name:16s} {rpg:8.0f} {a:8.3f} {pa:8.3f} {b:8.3f} {pb:8.3f}  {best} {pick}")
    right = sum(best == pick for *_, best, pick in rows)
    picked = sum(a if pick == 128 else b for _, _, a, _, b, _, _, pick in rows)
    fastest = sum(min(a, b) for _, _, a, _, b, _, _, _ in rows)
    err = max(max(abs(pa / a - 1), abs(pb / b - 1)) for _, _, a, pa, b, pb, _, _ in rows)
    print(f"choice matches the faster kernel on {right} of {len(rows)} workloads; "
          f"largest relative error of a predicted time {err:.3f}; picked kernels' total time "
          f"{picked / fastest - 1:+.2%} over the faster ones")
    src = open(HEADER).read()
    import re
    for name, val in coeffs.items():
        src = re.sub(rf"constexpr float {name} = [^;]*;", f"constexpr float {name} = {val:.6e}f;", src)
    open(HEADER, "w").write(src)


if __name__ == "__main__":
    cmd = sys.argv[1] if len(sys.argv) > 1 else "fit"
    measure() if cmd == "measure" else fit()
