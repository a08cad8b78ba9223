"""The range form of the plain policy's fills, which the GPU planner uses to
compute every piece independently, agrees with the oracle's one-copy-at-a-time
construction (host only).

Range form: a giver o's copies form one sequence -- its experts in descending
id, inside an expert the highest ordinals first -- and the f-th fill of the
run takes positions [b_f, b_f + d_f) of its giver's sequence, b_f being what o
gave before.  Expert e occupies positions [off_e, off_e + T_e) with off_e the
copies of o's higher-id experts, so fill f takes t = |[b_f, b_f + d_f) ∩
[off_e, off_e + T_e)| copies of e, the ordinals [left - t, left) with
left = T_e - max(0, b_f - off_e).  Its place in the fill's acquisition order is
the number of o's non-empty experts above it minus those used up before the
fill, and its index among e's pieces the number of o's earlier fills that end
after off_e."""
import numpy as np
import pytest

from oracle import planner as oplanner

try:
    import hypothesis as hyp
    import hypothesis.strategies as st
except ImportError:  # the property test needs hypothesis; everything else runs without
    hyp = st = None


def range_fills(T, R, L, C):
    load = [int(x) for x in np.asarray(T).reshape(R, L).sum(axis=1)]
    state = ["under" if x < C else "over" if x > C else "ok" for x in load]
    given = [0] * R
    seq = []
    while "under" in state:
        u = state.index("under")
        o = state.index("over")
        dd = C - load[u]
        seq.append((u, o, dd, given[o]))
        given[o] += dd
        load[u], state[u] = C, "ok"
        load[o] -= dd
        state[o] = "under" if load[o] < C else "over" if load[o] > C else "ok"
    # per expert: copies (off) and non-empty experts (nz) of the higher-id
    # experts of its rank
    off, nz = np.zeros(R * L, np.int64), np.zeros(R * L, np.int64)
    for h in range(R):
        run = runz = 0
        for e in range((h + 1) * L - 1, h * L - 1, -1):
            off[e], nz[e] = run, runz
            run += int(T[e])
            runz += int(T[e] > 0)
    fills = []
    for f, (u, o, dd, b) in enumerate(seq):
        # non-empty experts of o used up before this fill
        z = sum(1 for e in range(o * L, (o + 1) * L) if T[e] > 0 and off[e] + T[e] <= b)
        pieces = {}
        for e in range(o * L, (o + 1) * L):
            te = int(T[e])
            t = min(b + dd, off[e] + te) - max(b, off[e])
            if t <= 0:
                continue
            left = te - max(0, b - off[e])
            j = int(nz[e] - z)  # place in the fill's acquisition order
            pi = sum(1 for (_, o2, d2, b2) in seq[:f] if o2 == o and b2 + d2 > off[e])
            pieces[j] = (e, int(left - t), int(left), pi)
        fills.append((u, o, dd, [pieces[j] for j in range(len(pieces))]))
    return fills


def _loads(draw):
    R = draw(st.integers(1, 6))
    L = draw(st.integers(1, 5))
    C = draw(st.integers(1, 30))
    total = R * C
    # a random composition of R*C copies over the R*L experts, zeros allowed
    cuts = sorted(draw(st.lists(st.integers(0, total), min_size=R * L - 1, max_size=R * L - 1)))
    T = np.diff(np.array([0] + cuts + [total]))
    return R, L, C, T


def _check(case):
    R, L, C, T = case
    d = oplanner.Dims(R=R, E=R * L, B=L, K=1, S=C)
    fills, migrated = oplanner.constructive_plan(T, d)
    got = range_fills(T, R, L, C)
    assert len(got) == len(fills)
    seen = np.zeros(R * L, dtype=np.int64)  # pieces of each expert so far, in fill order
    for (u, o, dd, pieces), f in zip(got, fills):
        assert (u, o, dd) == (f.u, f.o, f.d)
        assert [pc[:3] for pc in pieces] == [tuple(int(v) for v in pc) for pc in f.pieces]
        for e, _, _, pi in pieces:
            assert pi == seen[e]
            seen[e] += 1
    moved = np.zeros(R * L, dtype=np.int64)
    for *_, pieces in got:
        for e, lo, hi, _ in pieces:
            moved[e] += hi - lo
    assert np.array_equal(moved, migrated)


if hyp is not None:
    @hyp.settings(max_examples=300, deadline=None)
    @hyp.given(st.composite(_loads)())
    def test_range_form_matches_the_construction(case):
        _check(case)
else:
    def test_range_form_matches_the_construction():
        pytest.skip("hypothesis is not installed")
