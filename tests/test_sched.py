"""The chunk scheduler (host only, no GPU): its prediction against numpy's
piecewise-linear interpolation, and its choice against a brute-force search."""
import numpy as np
import pytest

from quantized_linear_error_gb300 import build, spear

DENS = [0.0, 0.125, 0.5, 1.0]
TOKS = [320, 576, 1088, 2112]
MS = np.array([[10.0, 11.0, 19.0, 36.0],
               [10.5, 12.0, 20.5, 39.0],
               [12.0, 14.5, 24.0, 45.0],
               [14.0, 17.0, 29.0, 55.0]])


@pytest.fixture(scope="module")
def S():
    build.build()
    s = spear.ChunkScheduler(DENS, TOKS, MS)
    yield s
    s.close()


def _ref_predict(M, d):
    def row(i):
        t, y = np.array(TOKS, float), MS[i]
        if M <= t[0]:
            return y[0] + (y[1] - y[0]) * (M - t[0]) / (t[1] - t[0])
        if M >= t[-1]:
            return y[-2] + (y[-1] - y[-2]) * (M - t[-2]) / (t[-1] - t[-2])
        return float(np.interp(M, t, y))
    d = min(max(d, DENS[0]), DENS[-1])
    rows = np.array([row(i) for i in range(len(DENS))])
    return float(np.interp(d, DENS, rows))


@pytest.mark.parametrize("M", [64, 320, 400, 576, 1000, 1088, 2112, 3000])
@pytest.mark.parametrize("d", [0.0, 0.06, 0.125, 0.3, 0.5, 0.9, 1.0, 1.5])
def test_predict_matches_piecewise_linear(S, M, d):
    assert S.predict(M, d) == pytest.approx(_ref_predict(M, d), rel=1e-12)


def test_table_points_are_exact(S):
    for i, d in enumerate(DENS):
        for j, t in enumerate(TOKS):
            assert S.predict(t, d) == MS[i, j]


@pytest.mark.parametrize("itl", [9.0, 12.0, 16.0, 22.0, 40.0])
@pytest.mark.parametrize("d", [0.0, 0.25, 1.0])
def test_pick_is_largest_feasible_candidate(S, itl, d):
    cands = [1024, 128, 256, 512, 768, 2048]
    got = S.pick_chunk(64, d, itl, cands)
    feasible = [c for c in cands if _ref_predict(64 + c, d) <= itl]
    assert got == (max(feasible) if feasible else 0)


def test_pick_shrinks_as_density_grows(S):
    cands = list(range(0, 2049, 64))
    picks = [S.pick_chunk(64, d, 22.0, cands) for d in (0.0, 0.125, 0.5, 1.0)]
    assert picks == sorted(picks, reverse=True) and picks[0] > picks[-1]


def test_rejects_bad_tables():
    build.build()
    with pytest.raises(spear.SpearError):
        spear.ChunkScheduler([0.5, 0.2], TOKS, MS[:2])
    with pytest.raises(spear.SpearError):
        spear.ChunkScheduler(DENS, [320, 320, 1088, 2112], MS)
    with pytest.raises(spear.SpearError):
        spear.ChunkScheduler(DENS, TOKS, -MS)
    with pytest.raises(spear.SpearError):
        spear.ChunkScheduler([0.0, 1.5], TOKS, MS[:2])
