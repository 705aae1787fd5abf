"""Pins of the CPU fp64 oracle to facts fixed by the mathematics.

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign, p and q swapped, a transposed index, the wrong lse) fails at
least one of them.  None of them re-types the oracle's formulas: they use
closed forms, invariants, finite differences, hand-worked values and fp64
PyTorch autograd of the textbook definitions.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
IGN = -100


def _rows(seed, BT, V, scale=2.0, noise=1.0):
    rng = np.random.default_rng(seed)
    s = rng.normal(0.0, scale, (BT, V))
    t = s + rng.normal(0.0, noise, (BT, V))
    tg = rng.integers(0, V, BT)
    return s, t, tg


def _loss(s, t, tg, gce, gtvd):
    f = oracle.fused_ce_tvd_forward(s, t, tg)
    return gce * f["ce"] + gtvd * f["tvd"]


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("V", [1, 2, 7, 32, 1000])
@pytest.mark.parametrize("dtype", ["f32", "f64", "bf16"])
def test_constant_row_gives_log_v(V, dtype):
    s = torch.full((3, V), 1.75, dtype={"f32": torch.float32, "f64": torch.float64,
                                        "bf16": torch.bfloat16}[dtype])
    tg = np.array([0, V - 1, V // 2])
    out = oracle.fused_ce_tvd_forward(s, s.clone(), tg)
    np.testing.assert_allclose(out["ce"], math.log(V), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["student_lse"], 1.75 + math.log(V), atol=1e-12)
    assert np.all(out["tvd"] == 0.0) and np.all(out["sigma"] == 0.0)


def test_two_class_closed_forms():
    rng = np.random.default_rng(1)
    s = rng.normal(0, 3, (50, 2))
    t = rng.normal(0, 3, (50, 2))
    tg = rng.integers(0, 2, 50)
    out = oracle.fused_ce_tvd_forward(s, t, tg)
    other = s[np.arange(50), 1 - tg]
    mine = s[np.arange(50), tg]
    # ce = lse - s_t cancels when the target dominates: compare absolutely
    np.testing.assert_allclose(out["ce"], np.log1p(np.exp(other - mine)), rtol=1e-13, atol=1e-15)
    logistic = lambda z: 1.0 / (1.0 + np.exp(-z))
    p1, q1 = logistic(s[:, 1] - s[:, 0]), logistic(t[:, 1] - t[:, 0])
    np.testing.assert_allclose(out["tvd"], np.abs(p1 - q1), rtol=1e-12, atol=1e-15)
    # sigma = p1*sign(p1-q1) + p0*sign(p0-q0) with p0-q0 = -(p1-q1)
    np.testing.assert_allclose(out["sigma"], (2 * p1 - 1) * np.sign(p1 - q1), atol=1e-13)


def test_disjoint_peaks_reach_tvd_one():
    V = 9
    s = np.zeros((1, V)); s[0, 2] = 60.0
    t = np.zeros((1, V)); t[0, 6] = 60.0
    out = oracle.fused_ce_tvd_forward(s, t, [2])
    assert abs(out["tvd"][0] - 1.0) < 1e-12
    assert abs(out["sigma"][0] - 1.0) < 1e-12
    assert abs(out["ce"][0]) < 1e-12


def test_hand_worked_examples():
    with open(os.path.join(HERE, "golden", "hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    sym = {"ln2": math.log(2.0), "ln3": math.log(3.0), "ln4": math.log(4.0)}
    val = lambda x: sym[x] if isinstance(x, str) else (x[0] / x[1] if isinstance(x, list) else x)
    for c in cases:
        s = np.array([[val(x) for x in c["student"]]])
        t = np.array([[val(x) for x in c["teacher"]]])
        tg = [c["target"]]
        out = oracle.fused_ce_tvd_forward(s, t, tg)
        for key in ("ce", "tvd", "sigma", "student_lse", "teacher_lse"):
            assert abs(out[key][0] - val(c[key])) < 1e-14, (c["name"], key)
        g, st = oracle.fused_ce_tvd_backward(s, t, tg, c["grad_ce"], c["grad_tvd"])
        assert st == 0
        np.testing.assert_allclose(g[0], [val(x) for x in c["grad"]], atol=1e-14,
                                   err_msg=c["name"])


# ---------------------------------------------------------------- invariants

def test_identical_rows_give_exact_zero_tvd_sigma_and_tvd_grad():
    s, _, tg = _rows(2, 6, 50)
    out = oracle.fused_ce_tvd_forward(s, s.copy(), tg)
    assert np.all(out["tvd"] == 0.0) and np.all(out["sigma"] == 0.0)
    g_tvd, _ = oracle.fused_ce_tvd_backward(s, s.copy(), tg, 0.0, 1.0)
    assert np.all(g_tvd == 0.0)


def test_ranges_and_tvd_identities():
    s, t, tg = _rows(3, 40, 64, scale=3.0, noise=2.0)
    out = oracle.fused_ce_tvd_forward(s, t, tg)
    assert np.all(out["tvd"] >= 0) and np.all(out["tvd"] <= 1)
    assert np.all(np.abs(out["sigma"]) <= 1 + 1e-15)
    for r in range(40):
        p, q = oracle.row_probs(s, t, r)
        d = p - q
        assert abs(out["tvd"][r] - d[d > 0].sum()) < 1e-13       # tvd = sum_{p>q} (p-q)
        assert abs(out["tvd"][r] - (-d[d < 0]).sum()) < 1e-13    # = sum_{q>p} (q-p)
        assert abs(out["sigma"][r] - (p[d > 0].sum() - p[d < 0].sum())) < 1e-13
        assert abs(p.sum() - 1) < 1e-13 and abs(q.sum() - 1) < 1e-13


def test_shift_invariance():
    s, t, tg = _rows(4, 10, 33)
    cs = np.linspace(-7, 9, 10)[:, None]
    ct = np.linspace(5, -3, 10)[:, None]
    a = oracle.fused_ce_tvd_forward(s, t, tg)
    b = oracle.fused_ce_tvd_forward(s + cs, t + ct, tg)
    for k in ("ce", "tvd", "sigma"):
        np.testing.assert_allclose(b[k], a[k], atol=1e-12)
    np.testing.assert_allclose(b["student_lse"], a["student_lse"] + cs[:, 0], atol=1e-12)
    np.testing.assert_allclose(b["teacher_lse"], a["teacher_lse"] + ct[:, 0], atol=1e-12)
    ga, _ = oracle.fused_ce_tvd_backward(s, t, tg, 0.7, 1.3)
    gb, _ = oracle.fused_ce_tvd_backward(s + cs, t + ct, tg, 0.7, 1.3)
    np.testing.assert_allclose(gb, ga, atol=1e-13)


def test_each_gradient_term_sums_to_zero():
    s, t, tg = _rows(5, 12, 100)
    g_ce, _ = oracle.fused_ce_tvd_backward(s, t, tg, 1.0, 0.0)
    g_tvd, _ = oracle.fused_ce_tvd_backward(s, t, tg, 0.0, 1.0)
    assert np.abs(g_ce.sum(1)).max() < 1e-13
    assert np.abs(g_tvd.sum(1)).max() < 1e-14
    # the CE term alone is p - onehot: exactly -1 + p_target at the target
    for r in range(12):
        p, _ = oracle.row_probs(s, t, r)
        assert abs(g_ce[r, tg[r]] - (p[tg[r]] - 1.0)) < 1e-15


def test_ignore_rows_and_out_of_range_target():
    s, t, tg = _rows(6, 4, 20)
    tg = tg.copy(); tg[1] = IGN; tg[2] = 20
    out = oracle.fused_ce_tvd_forward(s, t, tg)
    assert out["status"] == oracle.TARGET_OUT_OF_RANGE
    for k in ("ce", "tvd", "student_lse", "teacher_lse", "sigma"):
        assert out[k][1] == 0.0
    assert math.isnan(out["ce"][2]) and not math.isnan(out["tvd"][2])
    g, st = oracle.fused_ce_tvd_backward(s, t, tg, 1.0, 1.0)
    assert st == oracle.TARGET_OUT_OF_RANGE
    assert np.all(g[1] == 0.0) and np.all(np.isnan(g[2]))
    assert np.all(np.isfinite(g[[0, 3]]))


@pytest.mark.parametrize("ignore_index", [-1, 5])
def test_ignore_index_is_the_argument(ignore_index):
    # "Backward Pass" ignore_index handling: which rows are ignored depends
    # only on the argument.  Rows whose target equals it give exactly what
    # the same rows give with target -100 and the default ignore_index; a
    # target of -100 is then an ordinary out-of-range target.
    s, t, tg = _rows(9, 6, 12)
    tg = tg.copy()
    tg[[1, 4]] = ignore_index
    ref_tg = tg.copy()
    ref_tg[[1, 4]] = IGN
    a = oracle.fused_ce_tvd_forward(s, t, tg, ignore_index)
    b = oracle.fused_ce_tvd_forward(s, t, ref_tg)
    for k in ("ce", "tvd", "student_lse", "teacher_lse", "sigma"):
        np.testing.assert_array_equal(a[k], b[k])
    ga, _ = oracle.fused_ce_tvd_backward(s, t, tg, 0.5, 0.25, ignore_index)
    gb, _ = oracle.fused_ce_tvd_backward(s, t, ref_tg, 0.5, 0.25)
    np.testing.assert_array_equal(ga, gb)
    assert np.all(ga[[1, 4]] == 0.0)
    tg[2] = IGN
    out = oracle.fused_ce_tvd_forward(s, t, tg, ignore_index)
    assert out["status"] == oracle.TARGET_OUT_OF_RANGE and math.isnan(out["ce"][2])


# ---------------------------------------------------------------- derivatives

def test_central_finite_differences():
    rng = np.random.default_rng(7)
    checked = 0
    while checked < 12:
        V = int(rng.integers(2, 17))
        s = rng.normal(0, 1.5, (1, V))
        t = rng.normal(0, 1.5, (1, V))
        tg = [int(rng.integers(0, V))]
        p, q = oracle.row_probs(s, t, 0)
        if np.min(np.abs(p - q)) < 1e-4:
            continue   # a kink of |p - q| too close for a finite difference
        gce, gtvd = rng.uniform(0.2, 2.0, 2)
        g, _ = oracle.fused_ce_tvd_backward(s, t, tg, gce, gtvd)
        h = 1e-6
        for v in range(V):
            sp, sm = s.copy(), s.copy()
            sp[0, v] += h; sm[0, v] -= h
            fd = (_loss(sp, t, tg, gce, gtvd)[0] - _loss(sm, t, tg, gce, gtvd)[0]) / (2 * h)
            assert abs(fd - g[0, v]) < 2e-8, (V, v, fd, g[0, v])
        checked += 1


def test_against_fp64_torch_autograd():
    s, t, tg = _rows(8, 16, 77, scale=2.5, noise=1.5)
    tg = tg.copy(); tg[3] = IGN
    gce = np.linspace(0.1, 1.6, 16)
    gtvd = np.linspace(2.0, 0.3, 16)
    S = torch.tensor(s, dtype=torch.float64, requires_grad=True)
    T = torch.tensor(t, dtype=torch.float64)
    TG = torch.tensor(tg)
    keep = (TG != IGN).double()
    ce = torch.nn.functional.cross_entropy(S, TG, reduction="none", ignore_index=IGN)
    tvd = 0.5 * (torch.softmax(S, -1) - torch.softmax(T, -1)).abs().sum(-1) * keep
    (torch.tensor(gce) * ce + torch.tensor(gtvd) * tvd).sum().backward()
    out = oracle.fused_ce_tvd_forward(s, t, tg)
    np.testing.assert_allclose(out["ce"], ce.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(out["tvd"], tvd.detach().numpy(), atol=1e-13)
    lse = torch.logsumexp(S.detach(), -1).numpy() * keep.numpy()
    np.testing.assert_allclose(out["student_lse"], lse, atol=1e-12)
    g, _ = oracle.fused_ce_tvd_backward(s, t, tg, gce, gtvd)
    np.testing.assert_allclose(g, S.grad.numpy(), atol=1e-14)


def test_tie_subgradient_matches_torch_abs():
    # Rows with teacher == student except a few entries: many exact ties.
    rng = np.random.default_rng(9)
    s = rng.normal(0, 1, (4, 12))
    t = s.copy()
    t[:, :3] += rng.normal(0, 1, (4, 3))
    # with unequal lse no element ties exactly; with equal lse all tie:
    t[2] = s[2]
    S = torch.tensor(s, requires_grad=True)
    tvd = 0.5 * (torch.softmax(S, -1) - torch.softmax(torch.tensor(t), -1)).abs().sum(-1)
    tvd.sum().backward()
    g, _ = oracle.fused_ce_tvd_backward(s, t, [0, 1, 2, 3], 0.0, 1.0)
    np.testing.assert_allclose(g, S.grad.numpy(), atol=1e-15)
    assert np.all(g[2] == 0.0)


# ---------------------------------------------------------------- CE subset

def test_ce_subset_matches_fused_and_torch():
    s, t, tg = _rows(10, 9, 40)
    tg = tg.copy(); tg[4] = IGN
    f = oracle.fused_ce_tvd_forward(s, t, tg)
    c = oracle.ce_forward(s, tg)
    np.testing.assert_array_equal(c["ce"], f["ce"])
    np.testing.assert_array_equal(c["lse"], f["student_lse"])
    gce = np.linspace(0.5, 1.5, 9)
    g_ce, _ = oracle.ce_backward(s, tg, gce)
    S = torch.tensor(s, requires_grad=True)
    ce = torch.nn.functional.cross_entropy(S, torch.tensor(tg), reduction="none",
                                           ignore_index=IGN)
    (ce * torch.tensor(gce)).sum().backward()
    np.testing.assert_allclose(g_ce, S.grad.numpy(), atol=1e-15)
    g_f, _ = oracle.fused_ce_tvd_backward(s, t, tg, gce, 0.0)
    np.testing.assert_allclose(g_ce, g_f, atol=0)


def test_bf16_inputs_are_widened_exactly():
    x = torch.randn(5, 19, generator=torch.Generator().manual_seed(3)).bfloat16()
    tg = np.arange(5)
    a = oracle.fused_ce_tvd_forward(x, x.roll(1, 1), tg)
    b = oracle.fused_ce_tvd_forward(x.double(), x.roll(1, 1).double(), tg)
    for k in ("ce", "tvd", "sigma", "student_lse", "teacher_lse"):
        np.testing.assert_array_equal(a[k], b[k])


def test_padded_rows_are_read_through_ld():
    s, t, tg = _rows(11, 5, 30)
    big_s = np.zeros((5, 48)); big_s[:, :30] = s
    big_t = np.full((5, 48), 99.0); big_t[:, :30] = t
    a = oracle.fused_ce_tvd_forward(s, t, tg)
    b = oracle.fused_ce_tvd_forward(big_s[:, :30], big_t[:, :30], tg)
    for k in ("ce", "tvd", "sigma", "student_lse", "teacher_lse"):
        np.testing.assert_array_equal(a[k], b[k])


# ---------------------------------------------------------------- mean over tokens

def test_mean_loss_matches_torch_reductions_and_autograd():
    s, t, tg = _rows(12, 20, 37)
    tg = tg.copy(); tg[[2, 9, 10]] = IGN
    alpha, beta = 0.7, 1.9
    f = oracle.fused_ce_tvd_forward(s, t, tg)
    loss, gce, gtvd, n = oracle.mean_loss(f["ce"], f["tvd"], tg, IGN, alpha, beta)
    assert n == 17
    S = torch.tensor(s, requires_grad=True)
    T = torch.tensor(t)
    TG = torch.tensor(tg)
    keep = TG != IGN
    ce_mean = torch.nn.functional.cross_entropy(S, TG, reduction="mean", ignore_index=IGN)
    tvd_rows = 0.5 * (torch.softmax(S, -1) - torch.softmax(T, -1)).abs().sum(-1)
    ref = alpha * ce_mean + beta * tvd_rows[keep].mean()
    ref.backward()
    assert abs(loss - ref.item()) < 1e-12
    # the upstream gradients reproduce autograd's gradient of the mean loss
    g, _ = oracle.fused_ce_tvd_backward(s, t, tg, gce, gtvd)
    np.testing.assert_allclose(g, S.grad.numpy(), atol=1e-14)


def test_mean_loss_with_no_kept_rows():
    loss, gce, gtvd, n = oracle.mean_loss([0.0, 0.0], [0.0, 0.0], [IGN, IGN])
    assert (loss, gce, gtvd, n) == (0.0, 0.0, 0.0, 0)
