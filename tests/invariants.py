"""Checks of what Theorem 1 and the buffer contract fix about any valid plan.

Theorem 1 (Kimi K3 模型结构（8）, section 定理 1; MoonEP : l'équilibrage parfait,
section Le théorème): every rank computes exactly S*K copies; a rank's remote
copies all come from one other rank, so they touch at most E/R experts; there
are at most R-1 fills.  The [E+B,H,H'] contract (Moonshot AI 开源 MoonEP,
contract paragraph): a rank computes an expert either as its home rank, from a
prefetch slot holding it, or (inference overflow) from the home row.

These checks work on plain arrays so they apply both to the oracle's plan and
to a plan exported from the GPU.
"""
import numpy as np


def check_plan_arrays(idx, R, E, B, K, S, mode, *, T, n_fills, fills, keep,
                      slot_expert, n_recv, src, cu_seqlens, dst, inverse, gidx=None):
    L, C, N = E // R, S * K, R * S * K
    flat = np.asarray(idx).reshape(-1).astype(np.int64)
    T = np.asarray(T)
    cu = np.asarray(cu_seqlens)
    dst = np.asarray(dst).reshape(-1)
    inverse = np.asarray(inverse).reshape(-1)
    slot_expert = np.asarray(slot_expert)

    assert np.array_equal(np.bincount(flat, minlength=E), T)
    # exactly S*K copies per rank
    assert cu.shape == (R, E + B + 1)
    assert np.all(cu[:, 0] == 0) and np.all(cu[:, -1] == C)
    assert np.all(np.diff(cu, axis=1) >= 0)
    # at most R-1 fills, each rank filled at most once, from one source
    assert 0 <= n_fills <= max(R - 1, 0)
    us = [int(f[0]) for f in np.asarray(fills)[:n_fills]]
    assert len(set(us)) == len(us)
    for u in range(R):
        if src[u] < 0:
            assert n_recv[u] == 0 and np.all(slot_expert[u] < 0)
            continue
        assert src[u] != u
        assert n_recv[u] <= L
        held = slot_expert[u][slot_expert[u] >= 0]
        assert len(held) == min(n_recv[u], B)
        assert np.all(held // L == src[u]), "slots hold experts of one source"
        assert len(set(held.tolist())) == len(held)
        if mode == 0:
            assert n_recv[u] <= B
    # dst is a bijection onto [0, R*C)
    assert dst.min() >= 0 and dst.max() < R * C
    assert np.array_equal(np.sort(dst), np.arange(N))
    assert np.array_equal(inverse[dst], np.arange(N))
    # every copy lands in a group whose weight row is its expert
    u_of = dst // C
    row = dst % C
    g_of = np.empty(N, dtype=np.int64)
    for u in range(R):
        m = u_of == u
        g_of[m] = np.searchsorted(cu[u], row[m], side="right") - 1
    for c in range(N):
        e, u, g = flat[c], u_of[c], g_of[c]
        if g < E:
            assert g == e, "home/overflow group must be the expert's own row"
            if e // L != u:
                assert mode == 1 and src[u] == e // L
        else:
            assert slot_expert[u, g - E] == e
    # keep + migrated == T: copies computed away from home
    away = np.bincount(flat[u_of != flat // L], minlength=E)
    assert np.array_equal(np.asarray(keep) + away, T)
    # inside a group copies follow ascending global ordinal
    if gidx is not None:
        q = np.asarray(gidx).reshape(-1)
        key = u_of * (E + B) + g_of
        order = np.lexsort((row, key))
        k2, q2 = key[order], q[order]
        same = k2[1:] == k2[:-1]
        assert np.all(q2[1:][same] > q2[:-1][same])
