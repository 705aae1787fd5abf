"""Property-based checks of the CPU oracle on random small rows: the
invariants the mathematics fixes must hold for every input, not only for the
fixed seeds of the pin tests.  (Skipped where hypothesis is not installed.)"""
import numpy as np
import pytest

import oracle

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

IGN = -100


@st.composite
def rows(draw):
    BT = draw(st.integers(1, 5))
    V = draw(st.integers(1, 40))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    scale = draw(st.sampled_from([0.1, 1.0, 3.0, 10.0]))
    rng = np.random.default_rng(seed)
    s = rng.normal(0.0, scale, (BT, V))
    t = rng.normal(0.0, scale, (BT, V))
    tie_row = draw(st.integers(-1, BT - 1))
    if tie_row >= 0:
        t[tie_row] = s[tie_row]
    tg = rng.integers(0, V, BT)
    ign = draw(st.integers(-1, BT - 1))
    if ign >= 0:
        tg[ign] = IGN
    gce = rng.uniform(-1.0, 1.0, BT)
    gtvd = rng.uniform(-1.0, 1.0, BT)
    return s, t, tg, gce, gtvd, tie_row, ign


@settings(max_examples=150, deadline=None, derandomize=True, database=None)
@given(rows())
def test_invariants_on_random_rows(case):
    s, t, tg, gce, gtvd, tie_row, ign = case
    BT, V = s.shape
    f = oracle.fused_ce_tvd_forward(s, t, tg)
    g, status = oracle.fused_ce_tvd_backward(s, t, tg, gce, gtvd)
    assert f["status"] == 0 and status == 0
    kept = tg != IGN
    # ranges
    assert np.all(f["tvd"] >= -1e-15) and np.all(f["tvd"] <= 1 + 1e-12)
    assert np.all(np.abs(f["sigma"]) <= 1 + 1e-12)
    assert np.all(f["ce"][kept] >= -1e-12)
    # lse is at least the row maximum and at most max + log V
    mx_s, mx_t = s.max(1), t.max(1)
    assert np.all(f["student_lse"][kept] >= mx_s[kept] - 1e-12)
    assert np.all(f["student_lse"][kept] <= mx_s[kept] + np.log(V) + 1e-12)
    assert np.all(f["teacher_lse"][kept] >= mx_t[kept] - 1e-12)
    # each row of the gradient sums to zero (both terms do)
    assert np.all(np.abs(g.sum(1)) <= 1e-12 * (1 + np.abs(g).sum(1)))
    # identical rows: no TVD, no sigma, and only the CE term in the gradient
    if tie_row >= 0 and kept[tie_row]:
        assert f["tvd"][tie_row] == 0.0 and f["sigma"][tie_row] == 0.0
        p = np.exp(s[tie_row] - f["student_lse"][tie_row])
        ce_only = gce[tie_row] * (p - (np.arange(V) == tg[tie_row]))
        assert np.allclose(g[tie_row], ce_only, rtol=1e-12, atol=1e-15)
    # ignored rows: zeros everywhere
    if ign >= 0:
        for k in ("ce", "tvd", "student_lse", "teacher_lse", "sigma"):
            assert f[k][ign] == 0.0
        assert np.all(g[ign] == 0.0)


@settings(max_examples=100, deadline=None, derandomize=True, database=None)
@given(rows(), st.floats(-50.0, 50.0), st.floats(-50.0, 50.0))
def test_per_row_shift_invariance(case, cs, ct):
    s, t, tg, gce, gtvd, _, _ = case
    a = oracle.fused_ce_tvd_forward(s, t, tg)
    b = oracle.fused_ce_tvd_forward(s + cs, t + ct, tg)
    kept = tg != IGN
    for k in ("ce", "tvd"):
        assert np.allclose(a[k][kept], b[k][kept], rtol=1e-9, atol=1e-9)
    assert np.allclose(b["student_lse"][kept] - a["student_lse"][kept], cs, atol=1e-9)
    ga, _ = oracle.fused_ce_tvd_backward(s, t, tg, gce, gtvd)
    gb, _ = oracle.fused_ce_tvd_backward(s + cs, t + ct, tg, gce, gtvd)
    # sigma and the TVD gradient jump where p - q changes sign, and after a
    # shift an exact tie (p == q) rounds to either sign: compare them only on
    # rows without near-ties
    for r in np.nonzero(kept)[0]:
        p, q = oracle.row_probs(s, t, r)
        if np.min(np.abs(p - q)) > 1e-9:
            assert np.isclose(a["sigma"][r], b["sigma"][r], rtol=1e-9, atol=1e-9)
            assert np.allclose(ga[r], gb[r], rtol=1e-7, atol=1e-12)


@settings(max_examples=100, deadline=None, derandomize=True, database=None)
@given(rows())
def test_tvd_identities(case):
    s, t, tg, _, _, _, _ = case
    f = oracle.fused_ce_tvd_forward(s, t, tg)
    for r in np.nonzero(tg != IGN)[0]:
        p, q = oracle.row_probs(s, t, r)
        d = p - q
        # tvd = sum over p > q of (p - q) = sum over q > p of (q - p)
        assert np.isclose(f["tvd"][r], d[d > 0].sum(), rtol=1e-10, atol=1e-13)
        assert np.isclose(f["tvd"][r], -d[d < 0].sum(), rtol=1e-10, atol=1e-12)
        # sigma = sum of p where p > q minus sum of p where p < q
        assert np.isclose(f["sigma"][r], p[d > 0].sum() - p[d < 0].sum(),
                          rtol=1e-10, atol=1e-13)
