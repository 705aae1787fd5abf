"""Element-by-element comparison of the CUDA path against the CPU oracle.

Tolerances:
  * per-row ce, tvd, student_lse, teacher_lse: abs 2e-4 for bf16 logits,
    abs 1e-5 for fp32 logits;
  * sigma: the same, widened by 2 * (oracle probability mass of the row's
    near-ties), because a sign flip at an element with |p - q| < 1e-7 is
    allowed and moves sigma by at most 2 p_v;
  * gradient: abs 1e-6 + rel 2e-3, widened at a row with near-ties by
    |grad_tvd| * 0.5 * p_v * (2 [v is a near-tie] + 2 * near-tie mass),
    the most a set of allowed sign flips can move element v.  A bf16
    gradient adds half a bf16 ulp of the reference value: rel 2e-3 is finer
    than bf16's unit roundoff (2^-8), so even the correctly rounded result
    could not meet it; fp32 gradients get no such allowance.
Ignored rows must be exactly zero on both sides.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TIE_EPS = 1e-7


def row_atol(dtype) -> float:
    return 2e-4 if dtype == torch.bfloat16 else 1e-5


def to_host_rows(x: torch.Tensor, rows) -> torch.Tensor:
    return x[rows].cpu() if rows is not None else x.cpu()


def tie_info(s_rows, t_rows):
    """Per row: boolean near-tie mask, near-tie mass and the oracle's p."""
    masks, mass, probs = [], [], []
    for r in range(s_rows.shape[0]):
        p, q = oracle.row_probs(s_rows, t_rows, r)
        m = np.abs(p - q) < TIE_EPS
        masks.append(m)
        mass.append(float(p[m].sum()))
        probs.append(p)
    return masks, np.array(mass), probs


def check_forward(dtype, target, got: dict, ref: dict, tie_mass, ignore_index=-100,
                  what="", atol=None):
    """got/ref: dict of per-row arrays (ce, tvd, student_lse, teacher_lse, sigma).

    atol (scalar or per row) overrides the dtype's tolerance when the inputs
    themselves carry a known error (logits computed by a GEMM)."""
    if atol is None:
        atol = row_atol(dtype)
    tg = np.asarray(target)
    ign = tg == ignore_index
    for k in ("ce", "tvd", "student_lse", "teacher_lse", "sigma"):
        g = np.asarray(got[k], np.float64)
        r = np.asarray(ref[k], np.float64)
        assert np.all(g[ign] == 0.0), f"{what}{k}: ignored rows must be exactly 0"
        nan_r = np.isnan(r)
        assert np.array_equal(np.isnan(g), nan_r), f"{what}{k}: NaN pattern differs"
        tol = atol + (2.0 * tie_mass if k == "sigma" else 0.0)
        err = np.abs(g - r)
        err[nan_r] = 0.0
        bad = np.nonzero(err > tol)[0]
        assert bad.size == 0, (f"{what}{k}: {bad.size} rows out of tolerance, worst row "
                               f"{bad[np.argmax(err[bad])]}: got {g[bad[0]]!r} ref {r[bad[0]]!r} "
                               f"err {err[bad].max():.3e} tol {np.atleast_1d(tol)[0]:.3e}")


def bf16_half_ulp(x):
    """Half a bf16 ulp at |x| (bf16 keeps 8 significant bits)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 8)


def grad_tol(ref: np.ndarray, out_dtype) -> np.ndarray:
    tol = 1e-6 + 2e-3 * np.abs(ref)
    if out_dtype == torch.bfloat16:
        tol = tol + bf16_half_ulp(np.abs(ref) * (1 + 2e-3) + 1e-6)
    return tol


def check_grad(got: np.ndarray, ref: np.ndarray, grad_tvd_rows, tie_masks, tie_mass, probs,
               target, ignore_index=-100, what="", out_dtype=torch.float32):
    """got: gradient rows as fp64 (from bf16/fp32); ref: the oracle's fp64 rows."""
    tg = np.asarray(target)
    gtvd = np.asarray(grad_tvd_rows, np.float64)
    for r in range(ref.shape[0]):
        g, f = got[r], ref[r]
        if tg[r] == ignore_index:
            assert np.all(g == 0.0), f"{what}row {r}: ignored row gradient must be exactly 0"
            continue
        if np.isnan(f).all():
            assert np.isnan(g).all(), f"{what}row {r}: out-of-range target row must be NaN"
            continue
        tol = grad_tol(f, out_dtype)
        if tie_mass[r] > 0.0:
            tol = tol + abs(gtvd[r]) * 0.5 * probs[r] * (2.0 * tie_masks[r] + 2.0 * tie_mass[r])
        err = np.abs(g - f)
        bad = np.nonzero(err > tol)[0]
        assert bad.size == 0, (f"{what}row {r}: {bad.size} elements out of tolerance; v={bad[0]} "
                               f"got {g[bad[0]]!r} ref {f[bad[0]]!r} tol {tol[bad[0]]:.3e}")


def oracle_rows(s_rows, t_rows, tg_rows, gce_rows, gtvd_rows, ignore_index=-100):
    ref = oracle.fused_ce_tvd_forward(s_rows, t_rows, tg_rows, ignore_index)
    grad, _ = oracle.fused_ce_tvd_backward(s_rows, t_rows, tg_rows, gce_rows, gtvd_rows,
                                           ignore_index)
    return ref, grad


def check_every_row(w, fwd: dict, grad, name: str, step: int = 256):
    """Every per-row output and every gradient element of a workload against
    the oracle, streamed in blocks of `step` rows.

    fwd: dict of per-row device outputs; grad: the (BT, V) device gradient.
    Elements within a lower bound of the gradient tolerance (1e-6 + 2e-3
    |ref|, plus half a bf16 ulp of the reference for bf16, at least 2^-9 of
    it) pass at once; any other element's row is checked exactly, with the
    near-tie widening, by check_grad."""
    dtype = w.student.dtype
    atol = row_atol(dtype)
    rel_lo = 2e-3 + (2.0 ** -9 if dtype == torch.bfloat16 else 0.0)
    tg_all = w.target.cpu().numpy()
    gce_all, gtvd_all = w.grad_ce.cpu().numpy(), w.grad_tvd.cpu().numpy()
    got_all = {k: v.cpu().numpy() for k, v in fwd.items()}
    for r0 in range(0, w.BT, step):
        r1 = min(r0 + step, w.BT)
        s, t = w.student[r0:r1].cpu(), w.teacher[r0:r1].cpu()
        tg = tg_all[r0:r1]
        ref, G = oracle_rows(s, t, tg, gce_all[r0:r1], gtvd_all[r0:r1], w.ignore_index)
        ign = tg == w.ignore_index
        for k, gk in got_all.items():
            g = gk[r0:r1].astype(np.float64)
            assert np.all(g[ign] == 0.0), f"{name} {k}: ignored rows"
            err = np.abs(g - ref[k])
            bad = np.nonzero(err > atol)[0]
            if bad.size and k == "sigma":  # near-ties may move sigma (and only sigma)
                _, mass, _ = tie_info(s[bad], t[bad])
                bad = bad[err[bad] > atol + 2.0 * mass]
            assert bad.size == 0, f"{name} {k}: rows {(bad + r0)[:5]} err {err[bad].max():.3e}"
        gb = grad[r0:r1].cpu().double()
        Gt = torch.from_numpy(G)
        assert torch.all(gb[torch.from_numpy(ign)] == 0), f"{name}: ignored gradient rows"
        err = (gb - Gt).abs_()
        lo = Gt.abs().mul_(rel_lo).add_(1e-6)
        rows = torch.nonzero((err > lo).any(dim=1)).flatten().numpy()
        if rows.size:
            masks, mass, probs = tie_info(s[rows], t[rows])
            check_grad(gb[rows].numpy(), G[rows], gtvd_all[r0:r1][rows], masks, mass, probs,
                       tg[rows], w.ignore_index, f"{name} rows {r0}+{rows[:5]} ", dtype)
