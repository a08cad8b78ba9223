"""Oracle: bf16 rounding, the expert GEMM, the gate-weighted combine, reduce_grad.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Sources (pages, by title and section):

* Moonshot AI 开源 MoonEP -- the framework contract paragraph: the grouped GEMM
  runs over one [E+B, H, H'] weight tensor, rows [0,E) the home experts and
  rows [E,E+B) this rank's prefetch slots (exact copies of home rows), with
  cu_seqlens choosing the active rows; training keeps fp32 gradients
  [E+B, H, H'] whose rows [E,E+B) are separate reduce buffers seen by every
  rank as one [R, B, H, H'] view; reduce_grad reads the slots holding a rank's
  own experts, adds them into the parameter gradients and zeroes the consumed
  slots.
* Kimi K3 模型结构（8） -- "在线规划、零拷贝、静态 shape": each (token, expert) pair
  carries one fp32 router weight; combine multiplies every expert output by its
  own weight.

Numerics (readings; the pages fix no precision for these steps): inputs are
bf16; the GEMM and the combine accumulate here in fp64 and round once to bf16
(round to nearest, ties to even); reduce_grad adds fp32 values in fp32, the
home row first and then the slots in ascending (rank, slot) order.
"""
from __future__ import annotations

import numpy as np

from .planner import Dims, Plan


# -- bf16 ---------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """A bf16 bit pattern is the top half of an fp32 bit pattern."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f32_bits_to_bf16_rne(u32: np.ndarray) -> np.ndarray:
    """Round fp32 bit patterns to bf16, nearest-even; NaN stays a (quiet) NaN."""
    u = np.asarray(u32, dtype=np.uint32)
    is_nan = (u & np.uint32(0x7F800000)) == np.uint32(0x7F800000)
    is_nan &= (u & np.uint32(0x007FFFFF)) != 0
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    rounded = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    nan_bits = (u >> np.uint32(16)) | np.uint32(0x0040)
    return np.where(is_nan, nan_bits, rounded).astype(np.uint16)


def to_bf16(x: np.ndarray) -> np.ndarray:
    """Round real values to bf16 bits: to fp32 first (nearest), then to bf16."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return f32_bits_to_bf16_rne(f.view(np.uint32))


# -- expert GEMM ----------------------------------------------------------------

def expert_outputs(x_bits: np.ndarray, w_bits, idx: np.ndarray, d: Dims,
                   experts=None) -> dict:
    """Y for every copy: bf16( x[r,s,:] @ W[e] ), grouped by expert.

    ``w_bits`` is either the [E, H, H'] array or a callable e -> [H, H'].
    Returns {e: (copy_ids, Y_bits [n_e, H'])} with copy_ids = (r*S+s)*K+k in
    ascending order.  The result does not depend on any plan: a slot row is
    an exact copy of its home row.
    """
    flat = idx.reshape(-1)
    xs = x_bits.reshape(d.R * d.S, d.H)
    out = {}
    todo = range(d.E) if experts is None else experts
    for e in todo:
        cids = np.nonzero(flat == e)[0]
        if cids.size == 0:
            out[e] = (cids, np.zeros((0, d.Hp), np.uint16))
            continue
        w = w_bits(e) if callable(w_bits) else w_bits[e]
        a = bf16_to_f64(xs[cids // d.K])
        y = a @ bf16_to_f64(w)
        out[e] = (cids, to_bf16(y))
    return out


def grouped_gemm_rows(recv_bits: np.ndarray, plan: Plan, w_home_bits,
                      w_slot_bits=None) -> np.ndarray:
    """Y rows of every rank's buffer from its cu_seqlens, row by row of weights.

    For rank u and weight row g: rows cu[u][g]..cu[u][g+1] of u's buffer are
    multiplied by W_home[g] if g < E, else by slot (u, g-E), which holds
    W_home[slot_expert[u][g-E]] after the prefetch.
    """
    d = plan.dims
    y = np.zeros((d.R * d.C, d.Hp), dtype=np.uint16)
    for u in range(d.R):
        for g in range(d.E + d.B):
            a0, a1 = plan.cu_seqlens[u, g], plan.cu_seqlens[u, g + 1]
            if a1 == a0:
                continue
            if g < d.E:
                w = w_home_bits[g]
            else:
                w = w_home_bits[plan.slot_expert[u, g - d.E]]
            a = bf16_to_f64(recv_bits[u * d.C + a0:u * d.C + a1])
            y[u * d.C + a0:u * d.C + a1] = to_bf16(a @ bf16_to_f64(w))
    return y


# -- combine ----------------------------------------------------------------------

def combine(y_rows_bits: np.ndarray, dst: np.ndarray, gates: np.ndarray, d: Dims,
            tokens=None) -> np.ndarray:
    """out[r,s,:] = bf16( sum over k ascending of gate[r,s,k] * Y[dst[r,s,k]] ).

    ``y_rows_bits`` is indexed by destination row (u*C + row).  ``tokens``
    optionally restricts the output to some flat token ids r*S+s.
    """
    dst2 = dst.reshape(d.R * d.S, d.K)
    g2 = gates.reshape(d.R * d.S, d.K).astype(np.float64)
    tok = np.arange(d.R * d.S) if tokens is None else np.asarray(tokens)
    acc = np.zeros((tok.size, d.Hp), dtype=np.float64)
    for k in range(d.K):
        acc += g2[tok, k][:, None] * bf16_to_f64(y_rows_bits[dst2[tok, k]])
    return to_bf16(acc)


def combine_from_copies(ycopies: dict, gates: np.ndarray, d: Dims) -> np.ndarray:
    """Combine from per-expert outputs (no plan involved at all)."""
    yc = np.zeros((d.N, d.Hp), dtype=np.float64)
    for e, (cids, yb) in ycopies.items():
        yc[cids] = bf16_to_f64(yb)
    yc = yc.reshape(d.R * d.S, d.K, d.Hp)
    g = gates.reshape(d.R * d.S, d.K).astype(np.float64)
    acc = np.zeros((d.R * d.S, d.Hp), dtype=np.float64)
    for k in range(d.K):
        acc += g[:, k][:, None] * yc[:, k]
    return to_bf16(acc)


# -- permute ----------------------------------------------------------------------

def permute(x_bits: np.ndarray, dst: np.ndarray, d: Dims) -> np.ndarray:
    """recv[dst[r,s,k]] = x[r,s] for every copy: the fixed [R*C, H] buffer."""
    recv = np.zeros((d.R * d.C, d.H), dtype=np.uint16)
    xs = x_bits.reshape(d.R * d.S, d.H)
    tok = np.arange(d.N) // d.K
    recv[dst.reshape(-1)] = xs[tok]
    return recv


def prefetch(w_home_bits: np.ndarray, plan: Plan) -> np.ndarray:
    """Slot (u, j) receives a copy of W_home[slot_expert[u][j]]."""
    d = plan.dims
    out = np.zeros((d.R, d.B) + w_home_bits.shape[1:], dtype=w_home_bits.dtype)
    for u in range(d.R):
        for j in range(d.B):
            e = plan.slot_expert[u, j]
            if e >= 0:
                out[u, j] = w_home_bits[e]
    return out


# -- reduce_grad ------------------------------------------------------------------

def reduce_grad(g_home: np.ndarray, g_slot: np.ndarray, plan: Plan,
                experts=None) -> None:
    """In place: G_home[e] += each slot holding e (ascending (u, j)); zero them.

    fp32 arithmetic, one add per slot, home row first.
    """
    d = plan.dims
    todo = range(d.E) if experts is None else experts
    for e in todo:
        acc = g_home[e].astype(np.float32, copy=True)
        for u in range(d.R):
            for j in range(d.B):
                if plan.slot_expert[u, j] == e:
                    acc = acc + g_slot[u, j].astype(np.float32)
                    g_slot[u, j] = 0.0
        g_home[e] = acc


# -- backward ---------------------------------------------------------------------
# The routed-expert backward that produces the slot gradients reduce_grad folds
# ("Moonshot AI 开源 MoonEP", contract paragraph: training keeps fp32 [E+B, H, H']
# gradients whose rows [E, E+B) are the reduce buffers; MoonEP : l'équilibrage
# parfait, "L'idée": in the backward pass the redundant experts' gradients are
# staged in a local reduce buffer and reduced to their home ranks afterwards).
# Written per copy, independent of any plan; with fp64 accumulation and one
# rounding to bf16 for bf16 outputs (readings: the pages fix no precision).

def combine_backward(y_copy_bits: np.ndarray, dout_bits: np.ndarray, gates: np.ndarray,
                     d: Dims):
    """For out[t] = sum_k g[t,k] * Y[t,k]:  dY[t,k] = bf16(g[t,k] * dout[t]) and
    dg[t,k] = <Y[t,k], dout[t]>.  y_copy_bits is [N, H'] in copy order."""
    g = gates.reshape(d.N).astype(np.float64)
    dout = bf16_to_f64(dout_bits.reshape(d.R * d.S, d.Hp))
    tok = np.arange(d.N) // d.K
    dy = to_bf16(g[:, None] * dout[tok])
    dg = np.einsum("ch,ch->c", bf16_to_f64(y_copy_bits.reshape(d.N, d.Hp)), dout[tok])
    return dy, dg.reshape(d.R, d.S, d.K)


def expert_backward(x_bits: np.ndarray, w_bits, idx: np.ndarray, dy_copy_bits: np.ndarray,
                    d: Dims, experts=None) -> dict:
    """Per expert e: dRecv rows = bf16(dY @ W_e^T) for its copies, and
    dW_e = sum over its copies of x_token^T dY (fp64, [H, H'])."""
    flat = idx.reshape(-1)
    xs = bf16_to_f64(x_bits.reshape(d.R * d.S, d.H))
    dyc = bf16_to_f64(dy_copy_bits.reshape(d.N, d.Hp))
    out = {}
    for e in (range(d.E) if experts is None else experts):
        cids = np.nonzero(flat == e)[0]
        w = bf16_to_f64(w_bits(e) if callable(w_bits) else w_bits[e])
        drecv = to_bf16(dyc[cids] @ w.T)
        dw = xs[cids // d.K].T @ dyc[cids]
        out[e] = (cids, drecv, dw)
    return out


def dispatch_backward(drecv_copy_bits: np.ndarray, d: Dims) -> np.ndarray:
    """dx[t] = bf16( sum over k ascending of dRecv[t,k] ), [N, H] in copy order in."""
    r = bf16_to_f64(drecv_copy_bits.reshape(d.R * d.S, d.K, d.H))
    return to_bf16(r.sum(axis=1))


def dw_by_group(x_bits: np.ndarray, idx: np.ndarray, dy_copy_bits: np.ndarray, plan: Plan,
                dst: np.ndarray) -> dict:
    """The same weight gradient split the way the grouped GEMM produces it before
    reduce_grad: each (rank u, weight row g) group sums its own rows only.
    Returns {(u, g): [H, H'] fp64} for non-empty groups."""
    d = plan.dims
    xs = bf16_to_f64(x_bits.reshape(d.R * d.S, d.H))
    dyc = bf16_to_f64(dy_copy_bits.reshape(d.N, d.Hp))
    dflat = dst.reshape(-1)
    out = {}
    for u in range(d.R):
        for g in range(d.E + d.B):
            a0, a1 = plan.cu_seqlens[u, g], plan.cu_seqlens[u, g + 1]
            if a1 == a0:
                continue
            rows = set(range(u * d.C + a0, u * d.C + a1))
            cids = np.array([c for c in range(d.N) if dflat[c] in rows])
            out[(u, g)] = xs[cids // d.K].T @ dyc[cids]
    return out


def grouped_gemm_dw_rows(recv_bits: np.ndarray, dy_rows_bits: np.ndarray, plan: Plan) -> dict:
    """{(u, g): recv[rows of g]^T . dY[rows of g]} (fp64) over every rank's
    buffer, from its cu_seqlens, for non-empty groups."""
    d = plan.dims
    out = {}
    for u in range(d.R):
        for g in range(d.E + d.B):
            a0, a1 = plan.cu_seqlens[u, g], plan.cu_seqlens[u, g + 1]
            if a1 == a0:
                continue
            rows = slice(u * d.C + a0, u * d.C + a1)
            out[(u, g)] = bf16_to_f64(recv_bits[rows]).T @ bf16_to_f64(dy_rows_bits[rows])
    return out
