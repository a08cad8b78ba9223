"""Oracle: the MoonEP balancing planner and the per-copy destinations.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Sources (pages, by title and section):

* Kimi K3 模型结构（8）：训练并行，MoonEP 与四类等待 -- "MoonEP：从「完全平衡」这个目标出发"
  (every rank must compute exactly S x K token copies), "定理 1" (the
  constructive proof: classify ranks as under-/over-loaded, repeatedly fill one
  underloaded rank u exactly to S x K from one overloaded rank o, put o back in
  the matching set; at most R-1 fills; u's remote copies all come from one rank
  and belong to at most E/R of that rank's local experts), "在线规划、零拷贝、静态
  shape" (each copy's destination is computed by the planner; permute writes
  it straight to its expert-grouped position in a fixed S x K buffer).
* MoonEP : l'équilibrage parfait -- "Le théorème" (the same construction;
  an overloaded rank never received anything, so what it moves belongs to its
  own local experts).
* Moonshot AI 开源 MoonEP -- the framework contract paragraph: one
  [E+B, H, H'] weight tensor per projection; rows [0,E) hold every rank's local
  experts, E/R rows per rank; rows [E, E+B) are this rank's prefetch slots;
  dispatch returns cu_seqlens over the E+B rows; training uses B = E/R, and in
  inference (B < E/R) experts beyond the slots are read from their home rows.

Readings where the pages are silent (each is a fixed, documented choice):

* home(e) = e // (E/R): contiguous blocks of E/R experts per rank.
* Which pair: the smallest-id underloaded rank u and the smallest-id
  overloaded rank o.  o gives exactly C - load(u) copies, even if it drops
  below C.
* Which copies: o's local experts in descending expert id; within one expert
  the copies with the highest global ordinal first, i.e. descending
  (token's owner rank, token, k).
* Slots: u's received experts in acquisition order (descending expert id);
  slot j holds the j-th.  In inference mode only the first B get a slot; the
  others are "overflow" and use the home row g = e.
* cu_seqlens is int32 [R][E+B+1] with a leading 0; groups are the weight rows
  in ascending order; inside a group copies are in ascending global ordinal.
* The global ordinal of a copy is its position among all copies of the same
  expert in ascending (rank, token, k) order.
"""
from __future__ import annotations

from bisect import insort
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Dims:
    R: int
    E: int
    B: int
    K: int
    S: int
    H: int = 0
    Hp: int = 0
    mode: int = 0    # 0 training, 1 inference
    policy: int = 0  # 0 constructive tie-break, 1 largest first

    @property
    def L(self) -> int:
        return self.E // self.R

    @property
    def C(self) -> int:
        return self.S * self.K

    @property
    def N(self) -> int:
        return self.R * self.S * self.K

    def home(self, e: int) -> int:
        return e // self.L


class RoutingError(ValueError):
    pass


def check_routing(idx: np.ndarray, d: Dims) -> None:
    """Every token's K expert ids must lie in [0, E) and be distinct."""
    if idx.shape != (d.R, d.S, d.K):
        raise RoutingError("routing shape mismatch")
    if idx.size and (idx.min() < 0 or idx.max() >= d.E):
        raise RoutingError("expert id out of range")
    flat = idx.reshape(-1, d.K)
    srt = np.sort(flat, axis=1)
    if d.K > 1 and np.any(srt[:, 1:] == srt[:, :-1]):
        raise RoutingError("duplicate expert within a token")


def histogram(idx: np.ndarray, d: Dims):
    """counts[r][e], T[e] = sum_r counts[r][e], load[h] = sum over h's experts."""
    counts = np.zeros((d.R, d.E), dtype=np.int64)
    for r in range(d.R):
        counts[r] = np.bincount(idx[r].reshape(-1), minlength=d.E)
    T = counts.sum(axis=0)
    load = T.reshape(d.R, d.L).sum(axis=1)
    return counts, T, load


def global_ordinals(idx: np.ndarray, d: Dims) -> np.ndarray:
    """Position of each copy among all copies of its expert, ascending (r,s,k)."""
    seen = [0] * d.E
    out = []
    for e in idx.reshape(-1).tolist():
        out.append(seen[e])
        seen[e] += 1
    return np.asarray(out, dtype=np.int64).reshape(idx.shape)


@dataclass
class Fill:
    u: int                    # the underloaded rank being filled
    o: int                    # the overloaded rank it is filled from
    d: int                    # copies moved = C - load(u) at that moment
    pieces: list = field(default_factory=list)  # (e, lo, hi): ordinals [lo,hi) of e


@dataclass
class Plan:
    dims: Dims
    counts: np.ndarray        # [R, E]
    T: np.ndarray             # [E]
    load0: np.ndarray         # [R] initial per-home-rank loads
    fills: list               # [Fill] in the order performed
    keep: np.ndarray          # [E] copies of e computed on its home rank
    slot_expert: np.ndarray   # [R, B] expert id held by slot (u, j), -1 if empty
    n_recv: np.ndarray        # [R] distinct remote experts rank u computes
    src: np.ndarray           # [R] the one rank u receives from, -1 if none
    overflow: list            # per rank: experts computed from their home rows
    rows: np.ndarray          # [R, E+B] copies per (rank, weight row)
    cu_seqlens: np.ndarray    # [R, E+B+1]
    pieces_of: list           # per expert: [(lo, hi, u, g)] migrated ranges


def constructive_plan(T: np.ndarray, d: Dims) -> tuple[list, np.ndarray]:
    """Theorem 1's construction with a fixed tie-break.

    policy 0 (the proof's plain order): the smallest-id underloaded rank u is
    filled from the smallest-id overloaded rank o, taking o's experts in
    descending expert id.
    policy 1 (largest first): u is the underloaded rank with the largest
    deficit C - load, o the overloaded rank with the largest surplus
    load - C (ties: smallest id), and o's experts are taken in descending
    order of their remaining copies (ties: descending id).  Taking the largest
    remaining experts first covers a fill with the fewest distinct experts.
    Both: inside an expert the copies with the highest global ordinals move.
    The proof's bounds (at most R-1 fills, at most E/R experts per receiving
    rank) hold for any choice of u, o and copies.

    Returns the fills (each with the expert ranges it moved) and, per expert,
    how many of its copies were migrated away from the home rank.
    """
    C, L = d.C, d.L
    load = [int(x) for x in np.asarray(T).reshape(d.R, L).sum(axis=1)]
    under = sorted(h for h in range(d.R) if load[h] < C)
    over = sorted(h for h in range(d.R) if load[h] > C)
    cursor = {h: (h + 1) * L - 1 for h in over}   # next expert to draw from (policy 0)
    migrated = [0] * d.E
    fills = []
    while under:
        if d.policy == 1:
            u = min(under, key=lambda h: (load[h] - C, h))   # largest deficit
            o = max(over, key=lambda h: (load[h] - C, -h))   # largest surplus
        else:
            u, o = under[0], over[0]
        f = Fill(u=u, o=o, d=C - load[u])
        need = f.d
        while need > 0:
            if d.policy == 1:
                cand = [(int(T[e]) - migrated[e], e) for e in range(o * L, (o + 1) * L)]
                left, e = max(cand)  # most remaining copies, then highest id
                assert left > 0, "overloaded rank ran out of copies"
            else:
                e = cursor[o]
                left = int(T[e]) - migrated[e]
                if left == 0:
                    cursor[o] = e - 1
                    # o is overloaded, so its own unmigrated copies exceed `need`
                    assert cursor[o] >= o * L, "overloaded rank ran out of copies"
                    continue
            t = min(left, need)
            f.pieces.append((e, left - t, left))  # the highest remaining ordinals
            migrated[e] += t
            need -= t
        fills.append(f)
        load[u] = C
        load[o] -= f.d
        under.remove(u)
        if load[o] < C:
            over.remove(o)
            insort(under, o)
        elif load[o] == C:
            over.remove(o)
    assert not over, "loads do not sum to R*S*K"
    return fills, np.asarray(migrated, dtype=np.int64)


def build_plan(idx: np.ndarray, d: Dims) -> Plan:
    check_routing(idx, d)
    if d.E % d.R:
        raise ValueError("E must be a multiple of R")
    if d.mode == 0 and d.B < d.L:
        raise ValueError("training needs B >= E/R slots")
    counts, T, load0 = histogram(idx, d)
    fills, migrated = constructive_plan(T, d)
    keep = T - migrated

    slot_expert = np.full((d.R, d.B), -1, dtype=np.int64)
    n_recv = np.zeros(d.R, dtype=np.int64)
    src = np.full(d.R, -1, dtype=np.int64)
    overflow = [[] for _ in range(d.R)]
    rows = np.zeros((d.R, d.E + d.B), dtype=np.int64)
    pieces_of = [[] for _ in range(d.E)]

    for e in range(d.E):
        rows[d.home(e), e] += keep[e]
    for f in fills:
        assert src[f.u] == -1, "a rank is filled at most once"
        src[f.u] = f.o
        n_recv[f.u] = len(f.pieces)
        if d.mode == 0:
            assert len(f.pieces) <= d.L <= d.B
        for j, (e, lo, hi) in enumerate(f.pieces):
            if j < d.B:
                slot_expert[f.u, j] = e
                g = d.E + j
            else:
                overflow[f.u].append(e)
                g = e
            rows[f.u, g] += hi - lo
            pieces_of[e].append((lo, hi, f.u, g))

    cu = np.zeros((d.R, d.E + d.B + 1), dtype=np.int64)
    cu[:, 1:] = np.cumsum(rows, axis=1)
    assert np.all(cu[:, -1] == d.C)
    return Plan(d, counts, T, load0, fills, keep, slot_expert, n_recv, src,
                overflow, rows, cu, pieces_of)


def destinations(idx: np.ndarray, plan: Plan):
    """dst[r,s,k] = u*C + row of the copy in rank u's buffer; inverse of it.

    A copy with global ordinal q < keep[e] stays on home(e) in group e at row
    cu[home][e] + q; otherwise it lies in exactly one migrated range
    [lo, hi) -> (u, g) and lands at cu[u][g] + (q - lo).
    """
    d = plan.dims
    gidx = global_ordinals(idx, d)
    flat_e = idx.reshape(-1).tolist()
    flat_q = gidx.reshape(-1).tolist()
    cu = plan.cu_seqlens.tolist()
    keep = plan.keep.tolist()
    dst = np.empty(d.N, dtype=np.int64)
    for c, (e, q) in enumerate(zip(flat_e, flat_q)):
        if q < keep[e]:
            u, g, lo = e // d.L, e, 0
        else:
            hits = [(pu, pg, plo) for (plo, phi, pu, pg) in plan.pieces_of[e]
                    if plo <= q < phi]
            assert len(hits) == 1
            u, g, lo = hits[0]
        dst[c] = u * d.C + cu[u][g] + (q - lo)
    inverse = np.full(d.N, -1, dtype=np.int64)
    inverse[dst] = np.arange(d.N, dtype=np.int64)
    return gidx, dst.reshape(idx.shape), inverse


def reduce_lists(plan: Plan) -> list:
    """Per home expert e: the slots (u, j) holding a copy of e, ascending (u, j)."""
    d = plan.dims
    out = [[] for _ in range(d.E)]
    for u in range(d.R):
        for j in range(d.B):
            e = int(plan.slot_expert[u, j])
            if e >= 0:
                out[e].append((u, j))
    return out


def full_plan(idx: np.ndarray, d: Dims) -> dict:
    """Everything the GPU planner exports, as plain arrays."""
    p = build_plan(idx, d)
    gidx, dst, inverse = destinations(idx, p)
    nf = len(p.fills)
    fills = np.full((max(d.R - 1, 0), 3), -1, dtype=np.int64)
    for i, f in enumerate(p.fills):
        fills[i] = (f.u, f.o, f.d)
    return dict(plan=p, counts=p.counts, T=p.T, load=p.load0, gidx=gidx,
                n_fills=nf, fills=fills, keep=p.keep, slot_expert=p.slot_expert,
                n_recv=p.n_recv, src=p.src, cu_seqlens=p.cu_seqlens, dst=dst,
                inverse=inverse)


# ----------------------------------------------------------------------------
# Send-once route encoding (Kimi K3 模型结构（8）, section 在线规划、零拷贝、静态 shape:
# each route entry stores its write offset on the destination rank; an entry
# whose destination rank already appeared earlier in the same token stores
# -(offset) - 1, so the payload is sent once per (token, destination rank) and
# copied locally on the receiver, while the fp32 weight is always sent).
# Reading: "earlier" means a smaller k within the token.
# ----------------------------------------------------------------------------

def route_encoding(dst: np.ndarray, d: Dims) -> np.ndarray:
    """route[r,s,k] = offset, or -offset-1 if the token already used that rank."""
    flat = dst.reshape(d.R * d.S, d.K)
    out = np.empty_like(flat)
    for t in range(flat.shape[0]):
        seen = set()
        for k in range(d.K):
            u, off = int(flat[t, k]) // d.C, int(flat[t, k]) % d.C
            out[t, k] = -off - 1 if u in seen else off
            seen.add(u)
    return out.reshape(d.R, d.S, d.K)


def link_traffic(dst: np.ndarray, d: Dims, payload_bytes: int, weight_bytes: int = 4) -> dict:
    """Bytes that leave a token's own rank: once per entry (every entry carries
    its payload) versus send-once (payload once per destination rank, weight
    for every entry).  Entries whose destination is the token's own rank move
    nothing across ranks."""
    flat = dst.reshape(d.R, d.S, d.K)
    remote_entries = 0
    remote_pairs = 0
    for r in range(d.R):
        for s in range(d.S):
            ranks = [int(v) // d.C for v in flat[r, s]]
            remote = [u for u in ranks if u != r]
            remote_entries += len(remote)
            remote_pairs += len(set(remote))
    return {
        "remote_entries": remote_entries,
        "remote_pairs": remote_pairs,
        "per_entry_bytes": remote_entries * (payload_bytes + weight_bytes),
        "send_once_bytes": remote_pairs * payload_bytes + remote_entries * weight_bytes,
    }
