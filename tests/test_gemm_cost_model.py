"""The GEMM tile-height cost model: the committed coefficients are the fit of
the committed measurements, and with them the model picks the faster kernel
on every measured workload where the two kernels differ by more than 3 %
(host only)."""
import json
import os
import re

import pytest

from perfectly_balanced_token_gb300.tuning import fit_gemm_cost as fgc


def _header_coefficients():
    src = open(fgc.HEADER).read()
    return {k: float(v) for k, v in re.findall(r"constexpr float (kCost\w+) = ([-0-9.e+]+)f;", src)}


def test_header_holds_the_fit_of_the_measurements():
    pytest.importorskip("scipy")
    recs = json.load(open(fgc.DATA))
    coeffs, rows = fgc.fit_coefficients(recs)
    hdr = _header_coefficients()
    assert set(hdr) == set(coeffs)
    for k, v in coeffs.items():
        assert hdr[k] == pytest.approx(v, rel=1e-5, abs=1e-12), k
    # the faster kernel is picked wherever the two differ by more than 3 %
    # (the model's fit error), and the picks cost under 1 % over always taking
    # the faster one
    for name, _, a, _, b, _, best, pick in rows:
        assert best == pick or abs(a - b) <= 0.03 * min(a, b), name
    picked = sum(a if pick == 128 else b for _, _, a, _, b, _, _, pick in rows)
    fastest = sum(min(a, b) for _, _, a, _, b, _, _, _ in rows)
    assert picked <= 1.01 * fastest


def test_tile_counts_from_cu_seqlens():
    import numpy as np
    # groups of 100, 256, 0 and 344 rows on one rank
    cu = np.array([[0, 100, 356, 356, 700]])
    assert fgc.tile_counts(cu) == (1 + 2 + 3, 2, 2, 3)


def test_measurements_cover_both_outcomes():
    recs = json.load(open(fgc.DATA))
    wins = {128 if r["ms128"] <= r["ms256"] else 256 for r in recs}
    assert wins == {128, 256}
    assert os.path.basename(fgc.HEADER) == "gemm_cost.cuh"
