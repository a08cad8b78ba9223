"""Oracle: imbalance metric, Theorem 2's bound, brute-force minimum redundancy.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Sources (pages, by title and section):

* Moonshot AI 开源 MoonEP -- "MoonEP 针对的问题": maxvio = max_e(T_e / T_bar) - 1,
  T_e the copies routed to expert e, T_bar the count under perfect balance.
* Kimi K3 模型结构（8） -- "定理 2": if rank 0's experts get nothing and the other
  E(R-1)/R experts split all R*S*K copies equally, rank 0 must take S*K remote
  copies, each expert offers at most S*K*R^2/(E(R-1)), so rank 0 needs at
  least ceil(E(R-1)/R^2) redundant experts.
* MoonEP : l'équilibrage parfait -- "La planification en ligne": exact optima
  are computed offline as the reference a fast planner is measured against.
  Here the exact optimum of the minimax redundant count is found by brute force
  with a max-flow feasibility test, for tiny inputs only.
"""
from __future__ import annotations

from collections import deque
from itertools import combinations

import numpy as np


def maxvio(T: np.ndarray, N: int, E: int) -> float:
    """max_e(T_e / T_bar) - 1 with T_bar = N / E."""
    return float(np.max(T) / (N / E) - 1.0)


def theorem2_bound(R: int, E: int) -> int:
    """ceil(E (R-1) / R^2)."""
    return -(-E * (R - 1) // (R * R))


def rank_lower_bound(C: int, local_load: int, T_max: int) -> int:
    """A rank with `local_load` home copies must import C - local_load copies;
    every expert offers at most T_max, so it needs that many distinct remote
    experts at least (ceil)."""
    need = max(0, C - local_load)
    return -(-need // T_max) if need else 0


def _max_flow(cap: list, s: int, t: int) -> int:
    """Edmonds-Karp (shortest augmenting paths) on a dense capacity matrix."""
    n = len(cap)
    flow = 0
    residual = [row[:] for row in cap]
    while True:
        parent = [-1] * n
        parent[s] = s
        q = deque([s])
        while q and parent[t] == -1:
            a = q.popleft()
            for b in range(n):
                if parent[b] == -1 and residual[a][b] > 0:
                    parent[b] = a
                    q.append(b)
        if parent[t] == -1:
            return flow
        push = None
        b = t
        while b != s:
            a = parent[b]
            push = residual[a][b] if push is None else min(push, residual[a][b])
            b = a
        b = t
        while b != s:
            a = parent[b]
            residual[a][b] -= push
            residual[b][a] += push
            b = a
        flow += push


def feasible(T: np.ndarray, R: int, C: int, allowed: list) -> bool:
    """Can every rank compute exactly C copies if rank r may compute its home
    experts plus the experts in allowed[r]?  Source -> expert (cap T_e) ->
    permitted rank (cap inf) -> sink (cap C); feasible iff the flow is R*C."""
    E = len(T)
    L = E // R
    n = 2 + E + R
    s, t = 0, n - 1
    big = int(np.sum(T)) + 1
    cap = [[0] * n for _ in range(n)]
    for e in range(E):
        cap[s][1 + e] = int(T[e])
        cap[1 + e][1 + E + e // L] = big
    for r in range(R):
        for e in allowed[r]:
            cap[1 + e][1 + E + r] = big
        cap[1 + E + r][t] = C
    return _max_flow(cap, s, t) == R * C


def min_max_redundant(T: np.ndarray, R: int, C: int, m_max: int):
    """Smallest m such that some choice of <= m remote experts per rank is
    feasible; returns (m, witness allowed-sets) or (None, None) above m_max."""
    E = len(T)
    L = E // R
    cand = [[e for e in range(E) if e // L != r and T[e] > 0] for r in range(R)]
    for m in range(m_max + 1):
        subsets = [[c for i in range(m + 1) for c in combinations(cand[r], i)]
                   for r in range(R)]
        found = _search(T, R, C, subsets, 0, [])
        if found is not None:
            return m, found
    return None, None


def _search(T, R, C, subsets, r, chosen):
    if r == R:
        return list(chosen) if feasible(T, R, C, chosen) else None
    for sub in subsets[r]:
        chosen.append(sub)
        got = _search(T, R, C, subsets, r + 1, chosen)
        chosen.pop()
        if got is not None:
            return got
    return None
