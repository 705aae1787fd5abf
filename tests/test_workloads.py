"""The seeded input recipes have the sizes, distributions and structure they
are documented to have (CPU, reduced rows; statistical checks use bounds of
several standard errors, so they hold for any seed)."""
import math

import pytest
import torch

from distillation_ce_tvd_gb300 import workloads

IGN = workloads.IGNORE_INDEX


def _within(x, mean, se, k=5.0):
    return abs(x - mean) <= k * se


def _ignored_fraction_ok(target, p):
    n = target.numel()
    frac = float((target == IGN).float().mean())
    return _within(frac, p, math.sqrt(p * (1 - p) / n))


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_shapes_dtypes_and_seeding(name):
    cfg = workloads.WORKLOADS[name]
    rows = min(cfg["BT"], 16)
    a = workloads.make(name, "cpu", rows=rows, V=min(cfg["V"], 4099))
    b = workloads.make(name, "cpu", rows=rows, V=min(cfg["V"], 4099))
    c = workloads.make(name, "cpu", rows=rows, V=min(cfg["V"], 4099), seed=cfg["seed"] + 1)
    assert a.student.shape == (rows, min(cfg["V"], 4099)) and a.student.dtype == cfg["dtype"]
    assert a.teacher.shape == a.student.shape and a.teacher.dtype == a.student.dtype
    assert a.target.dtype == torch.int64 and a.grad_ce.dtype == torch.float32
    for x in (a.student, a.teacher, a.target, a.grad_ce, a.grad_tvd):
        assert x.is_contiguous()
    for x, y in ((a.student, b.student), (a.teacher, b.teacher), (a.target, b.target)):
        assert torch.equal(x, y)  # same seed, same bytes
    assert not torch.equal(a.student, c.student)
    kept = a.target[a.target != IGN]
    assert torch.all((kept >= 0) & (kept < a.V))


def test_tiny_structure():
    w = workloads.make("tiny_bt8_v32_f32", "cpu")
    assert w.student.shape == (8, 32)
    assert torch.equal(w.student[3], w.teacher[3])
    assert int(w.target[5]) == IGN
    assert torch.all(w.grad_ce == 1) and torch.all(w.grad_tvd == 1)


def test_near_teacher_recipe():
    w = workloads.make("bt1024_v32000_bf16", "cpu", rows=256)
    s, t = w.student.float(), w.teacher.float()
    assert _within(float(s.std()), 1.5, 0.01)
    assert _within(float((t - s).std()), 0.5, 0.01)  # bf16 rounding adds < 1%
    assert _ignored_fraction_ok(workloads.make("bt1024_v32000_bf16", "cpu", V=8).target, 0.05)
    assert torch.allclose(w.grad_ce, torch.full_like(w.grad_ce, 1 / 256))
    assert torch.allclose(w.grad_tvd, torch.full_like(w.grad_tvd, 0.5 / 256))


def test_peaked_teacher_recipe():
    w = workloads.make("bt1024_v151936_bf16", "cpu", rows=512, V=4096)
    s, t = w.student.float(), w.teacher.float()
    assert _within(float(s.std()), 2.0, 0.02)
    # teacher independent of the student
    assert abs(float(torch.corrcoef(torch.stack([s.flatten(), t.flatten()]))[0, 1])) < 0.01
    # +6 at the target in 80% of rows: t[target] - mean(t) averages 0.8 * 6
    full = workloads.make("bt1024_v151936_bf16", "cpu", V=4096)
    kept = full.target != IGN
    rows = torch.nonzero(kept).flatten()
    lift = full.teacher.float()[rows, full.target[rows]] - full.teacher.float()[rows].mean(1)
    n = rows.numel()
    assert _within(float(lift.mean()), 0.8 * 6.0, math.sqrt(0.16 * 36 / n + 4.0 / n))
    assert _ignored_fraction_ok(full.target, 0.05)


def test_zipf_teacher_recipe_and_sampled_targets():
    # The teacher is 0.7 s + N(0, 1) + 8 rank(v)^-1.1 over one vocabulary
    # permutation shared by all rows, and targets are draws from softmax(t).
    V = 16
    w = workloads.make("bt8192_v151936_bf16", "cpu", rows=8192, V=V)
    s, t = w.student.float(), w.teacher.float()
    resid = t - 0.7 * s
    bias = resid.mean(0)  # N(0, 1) noise averages out over rows
    ranked = torch.sort(bias, descending=True).values
    expect = 8.0 * torch.arange(1, V + 1, dtype=torch.float32).pow(-1.1)
    assert torch.all((ranked - expect).abs() < 5.0 / math.sqrt(8192) + 0.05)
    assert _within(float((resid - bias).std()), 1.0, 0.02)
    # Gumbel-max targets follow softmax(t) of the stored (rounded) teacher
    kept = w.target != IGN
    p = torch.softmax(t[kept].double(), dim=1)
    emp = torch.bincount(w.target[kept], minlength=V).double() / kept.sum()
    se = (p.mean(0) * (1 - p.mean(0)) / kept.sum()).sqrt()
    assert torch.all((emp - p.mean(0)).abs() <= 5 * se + 1e-3)
    assert _ignored_fraction_ok(w.target, 0.03)


def test_independent_with_ties_recipe():
    w = workloads.make("bt4096_v256000_f32", "cpu", V=64)
    s, t = w.student, w.teacher
    tied = (s == t).all(1)
    n = s.shape[0]
    assert _within(float(tied.float().mean()), 0.10, math.sqrt(0.09 / n))
    st, tt = s[~tied], t[~tied]
    assert _within(float(st.std()), 3.0, 0.03) and _within(float(tt.std()), 3.0, 0.03)
    assert abs(float(torch.corrcoef(torch.stack([st.flatten(), tt.flatten()]))[0, 1])) < 0.02
    assert _ignored_fraction_ok(w.target, 0.05)


def test_linear_recipe_gives_logits_of_std_two():
    w = workloads.make_linear("linear_bt8192_d4096_v151936_bf16", "cpu", rows=64, V=4096)
    assert w.h_student.shape == (64, 4096) and w.w_student.shape == (4096, 4096)
    assert w.h_teacher.shape == (64, 4096) and w.w_teacher.shape == (4096, 4096)
    for h, wt in ((w.h_student, w.w_student), (w.h_teacher, w.w_teacher)):
        logits = h.float() @ wt.float().T
        assert _within(float(logits.std()), 2.0, 0.03)
    assert _ignored_fraction_ok(
        workloads.make_linear("linear_bt8192_d4096_v151936_bf16", "cpu", V=8, d=8).target, 0.03)
    small = workloads.make_linear("linear_bt8192_d4096_v151936_bf16", "cpu", rows=4, V=40, d=16)
    assert small.w_student.shape == (40, 16) and small.h_teacher.shape == (4, 16)
