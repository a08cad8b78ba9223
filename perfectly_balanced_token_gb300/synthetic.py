"""Seeded synthetic inputs for the MoonEP layer path.

This module only *draws* inputs: router top-K matrices, gates, token
activations, expert weights and gradient buffers.  It holds none of the
method's arithmetic (no histogram-based planning, no permutation, no GEMM, no
combine, no reduction); both the CUDA path and the CPU oracle receive what it
returns.

Routing recipes (all seeded):

* ``zipf_bias_routing`` -- router logits ~ N(0,1) plus a per-expert bias
  -1.2*log(pi(e)+1), a Zipf popularity law over a seeded permutation pi;
  top-K distinct experts by logit; gates = softmax of the chosen K logits.
  This is the small smoke-sized workload; ``zipf_sample_bias_routing`` keeps
  the literal form with raw Zipf(1.2) samples as the bias.
* ``gumbel_topk_routing`` -- weighted sampling without replacement by the
  Gumbel-max trick: score_e = log w_e + Gumbel noise, w_e = (pi(e)+1)^-alpha
  with pi a seeded permutation so hot experts land on different home ranks.
  ``tune_alpha`` bisects alpha until the routing's measured imbalance
  max_e(T_e / mean) - 1 hits a target; the pages' benchmark sweeps this
  imbalance ("maxvio") over synthetic shared-seed routing matrices
  (Moonshot AI 开源 MoonEP, section 与 DeepEP v2 的基准测试).
* ``round_robin_routing`` -- copy c = (r*S + s)*K + k goes to expert
  ``first + c mod (E - first)``.  ``first = 0`` is exactly balanced;
  ``first = E/R`` is the worst case of Theorem 2 (rank 0's own experts get no
  copies and the other experts split all copies equally), Kimi K3 模型结构（8）,
  section 定理 2.

The imbalance statistic computed here is a property of the *input* only and is
used to steer the generator toward a requested skew.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass
class Routing:
    idx: np.ndarray     # [R, S, K] int32 expert ids, distinct within a token
    gates: np.ndarray   # [R, S, K] float32 router weights of the chosen experts
    alpha: float | None = None


def _softmax_last(v: np.ndarray) -> np.ndarray:
    v = v - v.max(axis=-1, keepdims=True)
    ev = np.exp(v)
    return ev / ev.sum(axis=-1, keepdims=True)


def _topk_desc(scores: np.ndarray, K: int) -> np.ndarray:
    """Indices of the K largest entries of the last axis, largest first."""
    part = np.argpartition(-scores, K - 1, axis=-1)[..., :K]
    chosen = np.take_along_axis(scores, part, axis=-1)
    order = np.argsort(-chosen, axis=-1, kind="stable")
    return np.take_along_axis(part, order, axis=-1)


def input_skew(idx: np.ndarray, E: int) -> float:
    """max_e(T_e / mean T) - 1 of a routing matrix (an input statistic)."""
    t = np.bincount(idx.reshape(-1).astype(np.int64), minlength=E)
    return float(t.max() / (idx.size / E) - 1.0)


def zipf_bias_routing(R: int, S: int, K: int, E: int, seed: int = 0,
                      zipf_a: float = 1.2) -> Routing:
    rng = np.random.default_rng(seed)
    # Zipf popularity in logit space: expert of popularity rank p gets
    # -a*log(p+1), so popular experts win often but every token still draws
    # its own noise (raw Zipf samples as the bias would dwarf the noise and
    # send every token to the same K experts)
    bias = -zipf_a * np.log(rng.permutation(E) + 1.0)
    logits = rng.standard_normal((R, S, E)) + bias
    idx = _topk_desc(logits, K)
    gates = _softmax_last(np.take_along_axis(logits, idx, axis=-1))
    return Routing(idx.astype(np.int32), gates.astype(np.float32))


def zipf_sample_bias_routing(R: int, S: int, K: int, E: int, seed: int = 0,
                             zipf_a: float = 1.2) -> Routing:
    """The literal form of the small recipe: raw Zipf(zipf_a) samples as the
    per-expert bias.  Their heavy tail usually dwarfs the N(0,1) noise, so every
    token picks the same K experts: a degenerate but valid routing (kept as a
    parity case of its own)."""
    rng = np.random.default_rng(seed)
    bias = rng.zipf(zipf_a, size=E).astype(np.float64)
    logits = rng.standard_normal((R, S, E)) + bias
    idx = _topk_desc(logits, K)
    gates = _softmax_last(np.take_along_axis(logits, idx, axis=-1))
    return Routing(idx.astype(np.int32), gates.astype(np.float32))


class _GumbelSource:
    """Fixed noise for one (shape, seed) so every alpha sees the same draw."""

    def __init__(self, R, S, K, E, seed):
        rng = np.random.default_rng(seed)
        self.perm = rng.permutation(E)
        self.noise = rng.gumbel(size=(R, S, E)).astype(np.float32)
        self.K, self.E = K, E

    def draw(self, alpha: float) -> Routing:
        logw = (-alpha * np.log(self.perm + 1.0)).astype(np.float32)
        scores = self.noise + logw
        idx = _topk_desc(scores, self.K)
        chosen = np.take_along_axis(scores, idx, axis=-1).astype(np.float64)
        gates = _softmax_last(chosen)
        return Routing(idx.astype(np.int32), gates.astype(np.float32), alpha)


def gumbel_topk_routing(R, S, K, E, alpha: float, seed: int = 0) -> Routing:
    return _GumbelSource(R, S, K, E, seed).draw(alpha)


def tune_alpha(R, S, K, E, target: float, seed: int = 0, rel_tol: float = 0.05,
               abs_tol: float = 0.02, max_iter: int = 40) -> Routing:
    """Bisect the Zipf exponent until the routing skew is within tolerance."""
    src = _GumbelSource(R, S, K, E, seed)
    tol = max(abs_tol if target < 0.4 else 0.0, rel_tol * target)
    lo, hi = 0.0, 1.0
    best = src.draw(0.0)
    if input_skew(best.idx, E) >= target - tol:
        return best
    while True:  # grow the bracket
        r = src.draw(hi)
        v = input_skew(r.idx, E)
        if abs(v - target) <= tol:
            return r
        if v > target or hi > 64:
            break
        lo, hi = hi, hi * 2
    best, best_err = r, abs(v - target)
    for _ in range(max_iter):
        mid = 0.5 * (lo + hi)
        r = src.draw(mid)
        v = input_skew(r.idx, E)
        if abs(v - target) < best_err:
            best, best_err = r, abs(v - target)
        if best_err <= tol:
            break
        if v < target:
            lo = mid
        else:
            hi = mid
    return best


def round_robin_routing(R, S, K, E, first: int = 0, seed: int = 0) -> Routing:
    """Copy c goes to expert first + (c mod (E - first)); gates ~ softmax N(0,1)."""
    span = E - first
    if K > span:
        raise ValueError("round-robin routing needs K <= E - first")
    c = np.arange(R * S * K, dtype=np.int64).reshape(R, S, K)
    idx = (first + c % span).astype(np.int32)
    rng = np.random.default_rng(seed)
    gates = _softmax_last(rng.standard_normal((R, S, K))).astype(np.float32)
    return Routing(idx, gates)


def bad_routing_out_of_range(R, S, K, E) -> np.ndarray:
    idx = round_robin_routing(R, S, K, E).idx.copy()
    idx[R - 1, S - 1, K - 1] = E  # one id past the last expert
    return idx


def bad_routing_duplicate(R, S, K, E) -> np.ndarray:
    idx = round_robin_routing(R, S, K, E).idx.copy()
    idx[0, S // 2, K - 1] = idx[0, S // 2, 0]  # same expert twice in a token
    return idx


# ----------------------------------------------------------------------------
# Dense tensors.  Small shapes are drawn on the CPU (torch CPU generator) and
# can be moved to the device; large shapes are drawn directly on the device.
# ----------------------------------------------------------------------------

def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """bf16 tensor with N(0, std^2) entries, drawn in fp32 then rounded."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    step = 1 << 28
    for i in range(0, n, step):
        j = min(n, i + step)
        flat[i:j] = (torch.randn(j - i, generator=g, device=device,
                                 dtype=torch.float32) * std).to(torch.bfloat16)
    return out


def normal_f32(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=torch.float32, device=device)
    flat = out.view(-1)
    n = flat.numel()
    step = 1 << 28
    for i in range(0, n, step):
        j = min(n, i + step)
        flat[i:j] = torch.randn(j - i, generator=g, device=device,
                                dtype=torch.float32) * std
    return out


def integer_f32(shape, lo: int, hi: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 tensor of small integers in [lo, hi): sums of these are exact."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(lo, hi, shape, generator=g, device=device,
                         dtype=torch.int32).to(torch.float32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU tensor as uint16 numpy."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass(frozen=True)
class Workload:
    name: str
    R: int
    E: int
    B: int
    K: int
    S: int
    H: int
    Hp: int
    mode: int = 0  # 0 = training (B >= E/R), 1 = inference

    @property
    def L(self):
        return self.E // self.R

    @property
    def C(self):
        return self.S * self.K

    @property
    def N(self):
        return self.R * self.S * self.K


TINY = Workload("tiny", R=4, E=8, B=2, K=2, S=16, H=64, Hp=128)
SMALL = Workload("r8-e64", R=8, E=64, B=8, K=4, S=1024, H=1024, Hp=512)
PAGES = Workload("pages-benchmark-shaped", R=8, E=384, B=48, K=8, S=8192,
                 H=7168, Hp=2048)
K3 = Workload("k3-shaped", R=64, E=896, B=14, K=16, S=1024, H=4096, Hp=1024)
ADVERSARIAL_TRAIN = Workload("adversarial-train", R=8, E=384, B=48, K=8, S=8192,
                             H=7168, Hp=2048, mode=0)
ADVERSARIAL_INFER = Workload("adversarial-infer", R=8, E=384, B=4, K=8, S=8192,
                             H=7168, Hp=2048, mode=1)

MAXVIO_SWEEP = {
    "r8-e64": (0.0, 1.0, 5.0),
    "pages-benchmark-shaped": (0.2, 1.0, 10.0, 20.0),
    "k3-shaped": (1.0, 10.0),
}


def routing_for(w: Workload, maxvio: float | None = None, seed: int = 0) -> Routing:
    """The routing recipe used for each named workload."""
    if w.name == "tiny":
        return zipf_bias_routing(w.R, w.S, w.K, w.E, seed)
    if w.name.startswith("adversarial"):
        return round_robin_routing(w.R, w.S, w.K, w.E, first=w.E // w.R, seed=seed)
    if maxvio is not None and maxvio == 0.0:
        return round_robin_routing(w.R, w.S, w.K, w.E, first=0, seed=seed)
    assert maxvio is not None
    return tune_alpha(w.R, w.S, w.K, w.E, maxvio, seed)
