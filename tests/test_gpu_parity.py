"""Parity of the CUDA path (through the C ABI) with the CPU fp64 oracle."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from distillation_ce_tvd_gb300 import binding, workloads
from parity_util import (check_every_row, check_forward, check_grad, grad_tol, oracle_rows,
                         row_atol, tie_info, to_host_rows)

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()
    yield


def same_layout_clone(x):
    """A copy with the same strides (a plain clone of a padded view would be
    contiguous and take another code path)."""
    y = torch.empty_strided(x.shape, x.stride(), dtype=x.dtype, device=x.device)
    y.copy_(x)
    return y


def run(w, cluster=0, inplace=False, stream=None, ring=0):
    """Forward + backward of a workload on the GPU (cluster: CTAs per row of
    the forward, ring: its staging, 0 = automatic)."""
    opts = binding.options(ctas_per_row=cluster, ring=ring)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ce, tvd, ls, lt, sg = binding.fused_ce_tvd_forward(
        w.student, w.teacher, w.target, w.ignore_index, dev_status=status, stream=stream,
        options=opts)
    s_in = same_layout_clone(w.student) if inplace else w.student
    grad = binding.fused_ce_tvd_backward(
        s_in, w.teacher, w.target, ls, lt, sg, w.grad_ce, w.grad_tvd, w.ignore_index,
        inplace=inplace, dev_status=status, stream=stream)
    torch.cuda.synchronize()
    fwd = {"ce": ce, "tvd": tvd, "student_lse": ls, "teacher_lse": lt, "sigma": sg}
    return fwd, grad, int(status.item())


def compare(w, fwd, grad, rows=None, what=""):
    """Check the given rows (all when None) against the oracle."""
    s = to_host_rows(w.student, rows)
    t = to_host_rows(w.teacher, rows)
    tg = to_host_rows(w.target, rows).numpy()
    gce = to_host_rows(w.grad_ce, rows).numpy()
    gtvd = to_host_rows(w.grad_tvd, rows).numpy()
    ref, ref_grad = oracle_rows(s, t, tg, gce, gtvd, w.ignore_index)
    masks, mass, probs = tie_info(s, t)
    got = {k: to_host_rows(v, rows).numpy() for k, v in fwd.items()}
    check_forward(w.student.dtype, tg, got, ref, mass, w.ignore_index, what)
    g = to_host_rows(grad, rows).double().numpy()
    check_grad(g, ref_grad, gtvd, masks, mass, probs, tg, w.ignore_index, what, grad.dtype)
    return ref


def exact_tie_rows(w):
    return torch.nonzero((w.student == w.teacher).all(dim=1)).flatten()


def assert_exact_ties(w, fwd):
    rows = exact_tie_rows(w)
    rows = rows[w.target[rows] != w.ignore_index]
    if rows.numel():
        assert torch.all(fwd["tvd"][rows] == 0) and torch.all(fwd["sigma"][rows] == 0)


# ------------------------------------------------------------------ small, all rows

def test_tiny_workload_all_rows_and_fixture():
    with open(os.path.join(HERE, "golden", "tiny_bt8_v32_f32.json")) as f:
        d = json.load(f)
    w = workloads.make("tiny_bt8_v32_f32", "cpu")
    w = workloads.Workload(w.name, w.student.to(DEV), w.teacher.to(DEV), w.target.to(DEV),
                           w.grad_ce.to(DEV), w.grad_tvd.to(DEV))
    fwd, grad, st = run(w)
    assert st == 0
    compare(w, fwd, grad)
    np.testing.assert_allclose(fwd["tvd"].cpu().numpy(), d["forward"]["tvd"], atol=1e-5)
    np.testing.assert_allclose(grad.cpu().double().numpy(), d["grad_student"], atol=1e-6, rtol=2e-3)  # fp32
    assert fwd["tvd"][3].item() == 0.0 and fwd["sigma"][3].item() == 0.0
    assert torch.all(grad[5] == 0)


@pytest.mark.parametrize("name,rows,V", [
    ("bt1024_v32000_bf16", 96, 32000),
    ("bt1024_v32000_bf16", 64, 32000 + 5),        # ragged tail, misaligned row stride
    ("bt1024_v151936_bf16", 48, 151936),
    ("bt8192_v151936_bf16", 48, 151936),
    ("bt4096_v256000_f32", 24, 256000),
    ("bt4096_v256000_f32", 24, 4099),              # fp32 ragged
])
def test_recipes_reduced_rows_all_rows(name, rows, V):
    w = workloads.make(name, DEV, rows=rows, V=V, seed=11)
    fwd, grad, st = run(w)
    assert st == 0
    compare(w, fwd, grad, what=f"{name}[{rows}x{V}] ")
    assert_exact_ties(w, fwd)


@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_every_cluster_size(cluster, dtype):
    w = workloads.make("bt4096_v256000_f32", DEV, rows=40, V=20011, dtype=dtype, seed=5)
    fwd, grad, st = run(w, cluster=cluster)
    assert st == 0
    compare(w, fwd, grad, what=f"C={cluster} ")
    assert_exact_ties(w, fwd)


# ------------------------------------------------------------------ full sizes, sampled rows

FULL = ["bt1024_v32000_bf16", "bt1024_v151936_bf16", "bt8192_v151936_bf16", "bt4096_v256000_f32"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows_and_properties(name):
    w = workloads.make(name, DEV)
    fwd, grad, st = run(w)
    assert st == 0
    BT = w.BT
    g = torch.Generator().manual_seed(123)
    sample = torch.randperm(BT, generator=g)[:40]
    ign = torch.nonzero(w.target == w.ignore_index).flatten().cpu()[:4]
    ties = exact_tie_rows(w).cpu()[:4]
    rows = torch.unique(torch.cat([sample, ign, ties, torch.tensor([0, BT - 1])]))
    compare(w, fwd, grad, rows=rows.to(DEV), what=f"{name} ")
    # properties that hold at every row
    keep = w.target != w.ignore_index
    assert torch.all(fwd["tvd"] >= 0) and torch.all(fwd["tvd"] <= 1 + 1e-6)
    assert torch.all(fwd["sigma"].abs() <= 1 + 1e-5)
    rowmax = w.student.float().amax(dim=1)
    assert torch.all(fwd["student_lse"][keep] >= rowmax[keep] - 1e-5)
    assert torch.all(fwd["ce"][keep] >= -1e-4)
    for k in fwd:
        assert torch.all(fwd[k][~keep] == 0)
    assert torch.all(grad[~keep] == 0)
    assert torch.isfinite(grad).all()
    assert_exact_ties(w, fwd)


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_extreme_rows(dtype):
    # A maximum far above everything before it (at the end of a row) and at
    # its start, rows far from zero, -inf entries in the student, in the
    # teacher and in both identically, a constant row and an ignored row:
    # the first pass's rescaling paths and -inf handling.
    V, BT = 4104, 8
    big = 100.0 if dtype == torch.bfloat16 else 50.0  # > 64 / log2(e): forces a rescale
    g = torch.Generator(device=DEV).manual_seed(81)
    s = torch.randn(BT, V, generator=g, device=DEV)
    t = s + 0.5 * torch.randn(BT, V, generator=g, device=DEV)
    tg = torch.randint(V // 2, V - 1, (BT,), generator=g, device=DEV)
    s[0, V - 1] = big
    s[1, 0] = big
    s[2] -= 200.0
    t[2] -= 200.0
    s[3, : V // 2] = float("-inf")
    t[4, ::2] = float("-inf")
    s[5, ::3] = float("-inf")
    t[5] = s[5]
    s[6] = 0.0
    tg[5] = V - 2  # a finite student entry of row 5 (every third one is -inf)
    tg[7] = -100
    w = workloads.Workload("extreme", s.to(dtype).contiguous(), t.to(dtype).contiguous(), tg,
                           torch.full((BT,), 1.0 / BT, device=DEV),
                           torch.full((BT,), 0.5 / BT, device=DEV))
    fwd, grad, st = run(w)
    f2, g2, st2 = run_single(w)
    assert st == st2 == 0
    for k in fwd:
        assert torch.equal(fwd[k], f2[k]), k
    assert torch.equal(grad, g2)
    sh, th = w.student.cpu(), w.teacher.cpu()
    tgc = tg.cpu().numpy()
    ref, ref_grad = oracle_rows(sh, th, tgc, w.grad_ce.cpu().numpy(), w.grad_tvd.cpu().numpy())
    masks, mass, probs = tie_info(sh, th)
    got = {k: v.cpu().numpy() for k, v in fwd.items()}
    # the outputs are fp32: allow a few of their own ulps at large magnitudes
    mag = np.maximum.reduce([np.abs(ref["student_lse"]), np.abs(ref["teacher_lse"]),
                             np.abs(np.nan_to_num(ref["ce"]))])
    atol = row_atol(dtype) + 8.0 * 2.0 ** -23 * mag
    check_forward(dtype, tgc, got, ref, mass, what="extreme ", atol=atol)
    check_grad(grad.cpu().double().numpy(), ref_grad, w.grad_tvd.cpu().numpy(), masks, mass,
               probs, tgc, what="extreme ", out_dtype=dtype)
    assert fwd["tvd"][5].item() == 0.0 and fwd["sigma"][5].item() == 0.0
    assert abs(fwd["ce"][6].item() - np.log(V)) <= row_atol(dtype)
    assert torch.isfinite(grad).all()


@pytest.mark.parametrize("V", [1, 2, 3, 7, 8, 9, 17, 1023])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_small_and_ragged_vocab(V, dtype):
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=13, V=V, dtype=dtype, seed=V)
    fwd, grad, st = run(w)
    assert st == 0
    compare(w, fwd, grad, what=f"V={V} ")


def padded(w, ld, off):
    """The same rows stored with row stride `ld` starting `off` elements into
    a larger buffer (junk around them), to exercise strides, alignment and
    the vector path's ragged tail."""
    BT, V = w.student.shape
    out = []
    for x, junk in ((w.student, 77.0), (w.teacher, -55.0)):
        buf = torch.full((BT * ld + off + 16,), junk, device=DEV, dtype=x.dtype)
        view = buf[off:off + BT * ld].view(BT, ld)[:, :V]
        view.copy_(x)
        out.append(view)
    return workloads.Workload(w.name, out[0], out[1], w.target, w.grad_ce, w.grad_tvd)


# (V, ld, off): aligned rows with a ragged tail use the vector path; the rest
# the scalar path.
PADDED = [(3005, 3008, 0), (3005, 3048, 8), (3000, 3001, 0), (3000, 3013, 3), (3001, 3001, 1)]


@pytest.mark.parametrize("V,ld,off", PADDED)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_padded_and_misaligned_rows(V, ld, off, dtype):
    base = workloads.make("bt1024_v32000_bf16", DEV, rows=21, V=V, dtype=dtype, seed=2)
    w = padded(base, ld, off)
    fwd, grad, st = run(w)
    assert st == 0
    compare(w, fwd, grad, what=f"V={V} ld={ld} off={off} ")


def test_row_offsets_beyond_4_gib():
    """Rows that start more than 2^32 bytes (2^31 elements) past the base
    pointer: every entry point gives bitwise the results of a compact layout
    with the same 16-byte alignment, which itself matches the oracle."""
    V, ld = 4099, (1 << 30) + 64  # bf16: row r starts r * (2 GiB + 128 B) in
    base = workloads.make("bt1024_v32000_bf16", DEV, rows=3, V=V, dtype=torch.bfloat16, seed=9)
    small = padded(base, 4104, 0)
    fwd, grad, st = run(small)
    assert st == 0
    compare(small, fwd, grad, what="compact ")

    bufs = [torch.empty(2 * ld + V, dtype=torch.bfloat16, device=DEV) for _ in range(3)]

    def far(k, x=None):
        view = bufs[k].as_strided((3, V), (ld, 1))
        if x is not None:
            view.copy_(x)
        return view

    s_b, t_b = far(0, base.student), far(1, base.teacher)
    s_s, t_s = small.student, small.teacher
    tg, gce, gtvd = base.target, base.grad_ce, base.grad_tvd
    status = torch.zeros(1, dtype=torch.int32, device=DEV)

    def same(xs, ys, what):
        torch.cuda.synchronize()
        assert status.item() == 0, what
        for k, (x, y) in enumerate(zip(xs, ys)):
            assert torch.equal(x, y), f"{what} output {k}"

    f_s = binding.fused_ce_tvd_forward(s_s, t_s, tg)
    f_b = binding.fused_ce_tvd_forward(s_b, t_b, tg, dev_status=status)
    same(f_s, f_b, "forward")
    g_s = binding.fused_ce_tvd_backward(s_s, t_s, tg, *f_s[2:], gce, gtvd,
                                        grad_student=same_layout_clone(s_s))
    g_b = binding.fused_ce_tvd_backward(s_b, t_b, tg, *f_b[2:], gce, gtvd, grad_student=far(2),
                                        dev_status=status)
    same([g_s], [g_b], "backward")
    o_s = binding.fused_ce_tvd_forward_backward(s_s, t_s, tg, gce, gtvd,
                                                grad_student=same_layout_clone(s_s))
    o_b = binding.fused_ce_tvd_forward_backward(s_b, t_b, tg, gce, gtvd, grad_student=far(2),
                                                dev_status=status)
    same(o_s, o_b, "single launch")
    w_s = binding.fused_ce_tvd_forward_signs(s_s, t_s, tg)
    w_b = binding.fused_ce_tvd_forward_signs(s_b, t_b, tg, dev_status=status)
    same(w_s, w_b, "forward with sign words")
    b_b = binding.fused_ce_tvd_backward_signs(s_b, t_b, tg, *w_b[2:], gce, gtvd,
                                              grad_student=far(2), dev_status=status)
    same([g_s], [b_b], "backward from sign words")
    c_s = binding.ce_forward_backward(s_s, tg, gce, grad_logits=same_layout_clone(s_s))
    c_b = binding.ce_forward_backward(s_b, tg, gce, grad_logits=far(2), dev_status=status)
    same(c_s, c_b, "cross-entropy single launch")


def test_empty_batch_is_a_no_op():
    s = torch.empty(0, 100, device=DEV, dtype=torch.bfloat16)
    tg = torch.empty(0, device=DEV, dtype=torch.int64)
    out = binding.fused_ce_tvd_forward(s, s.clone(), tg)
    assert all(o.numel() == 0 for o in out)
    g = binding.fused_ce_tvd_backward(s, s.clone(), tg, *out[2:], out[0], out[0])
    assert g.numel() == 0


def test_all_rows_ignored_and_out_of_range_target():
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=6, V=500, seed=4)
    w.target[:] = -100
    fwd, grad, st = run(w)
    assert st == 0 and all(torch.all(v == 0) for v in fwd.values()) and torch.all(grad == 0)
    w.target[:] = torch.tensor([3, 500, -100, -1, 7, 499], device=DEV)
    fwd, grad, st = run(w)
    assert st == binding.FCT_DEV_TARGET_OUT_OF_RANGE
    compare(w, fwd, grad, what="oob ")
    assert torch.isnan(fwd["ce"][1]) and torch.isnan(fwd["ce"][3])
    assert torch.isnan(grad[1].float()).all() and torch.isnan(grad[3].float()).all()


@pytest.mark.parametrize("ignore_index", [-1, 5])
def test_other_ignore_index_values(ignore_index):
    # ignore_index is an argument, not a constant: -1, or even a vocabulary
    # index (rows whose target is 5 are then ignored).  A target of -100 is
    # out of range for both.
    import dataclasses
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=40, V=4104, seed=71)
    w = dataclasses.replace(w, ignore_index=ignore_index)
    w.target[[2, 9, 30]] = ignore_index
    w.target[11] = -100
    fwd, grad, st = run(w)
    assert st == binding.FCT_DEV_TARGET_OUT_OF_RANGE
    compare(w, fwd, grad, what=f"ignore_index={ignore_index} ")
    assert torch.all(grad[[2, 9, 30]] == 0) and torch.isnan(fwd["ce"][11])
    f2, g2, st2 = run_single(w)
    assert st2 == st
    nan_safe = ~torch.isnan(fwd["ce"])
    for k in fwd:
        assert torch.equal(fwd[k][nan_safe], f2[k][nan_safe]), k
    assert torch.equal(grad[nan_safe], g2[nan_safe])
    # cross-entropy alone and the mean front end take the same argument
    ce, lse, gl = binding.ce_forward_backward(w.student, w.target, w.grad_ce, ignore_index)
    torch.cuda.synchronize()
    assert torch.all(ce[[2, 9, 30]] == 0) and torch.all(gl[[2, 9, 30]] == 0)
    assert torch.equal(ce[nan_safe], fwd["ce"][nan_safe])
    _, _, n = binding.fused_ce_tvd_mean_upstream(w.target, ignore_index, 1.0, 1.0)
    torch.cuda.synchronize()
    assert int(n.item()) == int((w.target != ignore_index).sum().item())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_inplace_matches_out_of_place(dtype):
    w = workloads.make("bt1024_v151936_bf16", DEV, rows=17, V=12345, dtype=dtype, seed=8)
    _, g1, _ = run(w)
    _, g2, _ = run(w, inplace=True)
    assert torch.equal(g1, g2)


def test_broadcast_upstream_gradient():
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=9, V=777, seed=3)
    fwd, _, _ = run(w)
    ls, lt, sg = fwd["student_lse"], fwd["teacher_lse"], fwd["sigma"]
    a = binding.fused_ce_tvd_backward(w.student, w.teacher, w.target, ls, lt, sg, 0.25, 1.5)
    b = binding.fused_ce_tvd_backward(w.student, w.teacher, w.target, ls, lt, sg,
                                      torch.full((9,), 0.25, device=DEV),
                                      torch.full((9,), 1.5, device=DEV))
    assert torch.equal(a, b)


def test_row_blocks_are_bitwise_independent():
    w = workloads.make("bt8192_v151936_bf16", DEV, rows=64, V=151936, seed=21)
    fwd, grad, _ = run(w)
    for lo, hi in ((0, 1), (1, 30), (30, 64)):
        sub = workloads.Workload(w.name, w.student[lo:hi], w.teacher[lo:hi], w.target[lo:hi],
                                 w.grad_ce[lo:hi], w.grad_tvd[lo:hi])
        f2, g2, _ = run(sub)
        for k in fwd:
            assert torch.equal(fwd[k][lo:hi], f2[k]), k
        assert torch.equal(grad[lo:hi], g2)


def test_non_default_stream():
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=33, V=32000, seed=6)
    ref_fwd, ref_grad, _ = run(w)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        fwd, grad, _ = run(w, stream=s)
    for k in fwd:
        assert torch.equal(fwd[k], ref_fwd[k])
    assert torch.equal(grad, ref_grad)


def test_repeat_runs_are_deterministic():
    w = workloads.make("bt4096_v256000_f32", DEV, rows=20, V=65536, seed=9)
    a, ga, _ = run(w)
    b, gb, _ = run(w)
    for k in a:
        assert torch.equal(a[k], b[k])
    assert torch.equal(ga, gb)


# ------------------------------------------------------------------ CE subset, autograd

@pytest.mark.parametrize("dtype,V,ld,cluster", [
    (torch.bfloat16, 151936, None, 0), (torch.float32, 256000, None, 0),   # fp32: 2-CTA rows
    (torch.bfloat16, 20003, 20008, 0), (torch.float32, 9001, 9004, 4),
    (torch.bfloat16, 3003, None, 0),                                        # unaligned: two launches
    (torch.bfloat16, 5, None, 0)])
def test_ce_single_launch_equals_two(dtype, V, ld, cluster):
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=10, V=V, dtype=dtype, seed=36)
    if ld is not None:
        w = padded(w, ld, 0)
    w.target[3] = w.ignore_index
    w.target[6] = -7                                   # out of range
    opts = binding.options(ctas_per_row=cluster)
    st1 = torch.zeros(1, dtype=torch.int32, device=DEV)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    ce1, lse1 = binding.ce_forward(w.student, w.target, dev_status=st1, options=opts)
    g1 = binding.ce_backward(w.student, w.target, lse1, w.grad_ce, dev_status=st1)
    ce2, lse2, g2 = binding.ce_forward_backward(w.student, w.target, w.grad_ce, dev_status=st2,
                                                options=opts)
    s_in = same_layout_clone(w.student)
    ce3, lse3, g3 = binding.ce_forward_backward(s_in, w.target, 0.25, inplace=True, options=opts)
    g4 = binding.ce_backward(w.student, w.target, lse1, 0.25)
    torch.cuda.synchronize()
    assert st1.item() == st2.item() == binding.FCT_DEV_TARGET_OUT_OF_RANGE

    def bits(x):
        x = x.contiguous()
        return x.view(torch.int32 if x.element_size() == 4 else torch.int16)

    for a, b in ((ce1, ce2), (lse1, lse2), (g1, g2), (ce1, ce3), (lse1, lse3), (g4, g3)):
        assert torch.equal(bits(a), bits(b))


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 151936), (torch.float32, 32003), (torch.bfloat16, 5)])
def test_ce_subset(dtype, V):
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=24, V=V, dtype=dtype, seed=12)
    w.target[2] = -100
    ce, lse = binding.ce_forward(w.student, w.target)
    g = binding.ce_backward(w.student, w.target, lse, w.grad_ce)
    gi = binding.ce_backward(w.student.clone(), w.target, lse, w.grad_ce, inplace=True)
    torch.cuda.synchronize()
    assert torch.equal(g, gi)
    s = w.student.cpu()
    tg = w.target.cpu().numpy()
    ref = oracle.ce_forward(s, tg)
    ref_g, _ = oracle.ce_backward(s, tg, w.grad_ce.cpu().numpy())
    atol = 2e-4 if dtype == torch.bfloat16 else 1e-5
    np.testing.assert_allclose(ce.cpu().numpy(), ref["ce"], atol=atol, rtol=0)
    np.testing.assert_allclose(lse.cpu().numpy(), ref["lse"], atol=atol, rtol=0)
    err = np.abs(g.cpu().double().numpy() - ref_g)
    assert np.all(err <= grad_tol(ref_g, dtype))


def test_autograd_wrapper_matches_direct_calls():
    from distillation_ce_tvd_gb300.autograd import fused_ce_tvd_loss
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=16, V=4000, seed=14)
    s = w.student.clone().requires_grad_(True)
    ce, tvd = fused_ce_tvd_loss(s, w.teacher, w.target)
    (ce * w.grad_ce + tvd * w.grad_tvd).sum().backward()
    fwd, grad, _ = run(w)
    assert torch.equal(ce.detach(), fwd["ce"]) and torch.equal(tvd.detach(), fwd["tvd"])
    assert torch.equal(s.grad, grad)


# ------------------------------------------------------------------ sign words

@pytest.mark.parametrize("dtype,V,ld,cluster", [
    (torch.bfloat16, 151936, None, 0),
    (torch.bfloat16, 20003, 20008, 2),     # ragged tail, aligned rows, 2-CTA clusters
    (torch.float32, 9001, 9004, 8),        # ragged tail, 8-CTA clusters
    (torch.float32, 32000, None, 0),
    (torch.bfloat16, 3003, None, 0),       # unaligned rows: flags set, signs recomputed
])
def test_sign_words_match_plain_forward_and_backward(dtype, V, ld, cluster):
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=12, V=V, dtype=dtype, seed=35)
    if ld is not None:
        w = padded(w, ld, 0)
    w.teacher[2] = w.student[2]                                   # every element ties
    w.teacher[3] = (w.student[3].float() + 1.0).to(dtype)         # near ties
    w.target[5] = w.ignore_index
    w.target[7] = V + 3                                           # out of range
    opts = binding.options(ctas_per_row=cluster)
    st1 = torch.zeros(1, dtype=torch.int32, device=DEV)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    f1 = binding.fused_ce_tvd_forward(w.student, w.teacher, w.target, dev_status=st1, options=opts)
    g1 = binding.fused_ce_tvd_backward(w.student, w.teacher, w.target, *f1[2:], w.grad_ce,
                                       w.grad_tvd, dev_status=st1)
    f2 = binding.fused_ce_tvd_forward_signs(w.student, w.teacher, w.target, dev_status=st2,
                                            options=opts)
    signs = f2[5]
    g2 = binding.fused_ce_tvd_backward_signs(w.student, w.teacher, w.target, *f2[2:5], signs,
                                             w.grad_ce, w.grad_tvd, dev_status=st2)
    s_in = same_layout_clone(w.student)
    g3 = binding.fused_ce_tvd_backward_signs(s_in, w.teacher, w.target, *f2[2:5], signs,
                                             w.grad_ce, w.grad_tvd, inplace=True)
    torch.cuda.synchronize()
    assert st1.item() == st2.item() == binding.FCT_DEV_TARGET_OUT_OF_RANGE

    def bits(x):  # compare bit patterns: the out-of-range row holds NaN
        x = x.contiguous()
        return x.view(torch.int32 if x.element_size() == 4 else torch.int16)

    for a, b in zip(f1, f2[:5]):
        assert torch.equal(bits(a), bits(b))
    assert torch.equal(bits(g1), bits(g2))
    assert torch.equal(bits(g1), bits(g3))
    flags = signs[:, :4].contiguous().view(torch.int32)[:, 0]
    assert flags[2].item() != 0               # the tied row falls back to the teacher


# ------------------------------------------------------------------ randomized layouts

def _random_case(k):
    """Seeded random shape, dtype, layout, cluster size and row structure."""
    g = np.random.default_rng(1000 + k)
    dtype = [torch.bfloat16, torch.float32][int(g.integers(2))]
    V = int(g.choice([1, 2, 7, 8, 33, 257, 1000, 4099, 20000, 70001]))
    rows = int(g.integers(1, 20))
    vec = 8 if dtype == torch.bfloat16 else 4
    layout = int(g.integers(3))          # 0 contiguous, 1 padded to a vector, 2 odd stride
    ld = {0: None, 1: (V + vec - 1) // vec * vec + vec, 2: V + 1}[layout]
    cluster = int(g.choice([0, 1, 2, 4, 8]))
    return dtype, V, rows, ld, cluster, int(g.integers(1 << 30))


@pytest.mark.parametrize("k", range(24))
def test_randomized_layouts_all_paths(k):
    dtype, V, rows, ld, cluster, seed = _random_case(k)
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=rows, V=V, dtype=dtype, seed=seed)
    if ld is not None:
        w = padded(w, ld, 0)
    if rows > 2:
        w.teacher[1] = w.student[1]
        w.target[2] = w.ignore_index
    f1, g1, st1 = run(w, cluster=cluster)
    f2, g2, st2 = run_single(w, cluster=cluster)
    assert st1 == st2 == 0
    for key in f1:
        assert torch.equal(f1[key], f2[key]), key
    assert torch.equal(g1, g2)
    f3 = binding.fused_ce_tvd_forward_signs(w.student, w.teacher, w.target,
                                            options=binding.options(ctas_per_row=cluster))
    g3 = binding.fused_ce_tvd_backward_signs(w.student, w.teacher, w.target, *f3[2:5], f3[5],
                                             w.grad_ce, w.grad_tvd)
    torch.cuda.synchronize()
    for key, x in zip(("ce", "tvd", "student_lse", "teacher_lse", "sigma"), f3[:5]):
        assert torch.equal(f1[key], x), key
    assert torch.equal(g1, g3)
    compare(w, f1, g1, what=f"case {k} ")


# ------------------------------------------------------------------ single launch

def run_single(w, cluster=0, inplace=False, grads=None, ring=0):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    s_in = same_layout_clone(w.student) if inplace else w.student
    gce, gtvd = grads if grads is not None else (w.grad_ce, w.grad_tvd)
    ce, tvd, ls, lt, sg, grad = binding.fused_ce_tvd_forward_backward(
        s_in, w.teacher, w.target, gce, gtvd, w.ignore_index, inplace=inplace,
        dev_status=status, options=binding.options(ctas_per_row=cluster, ring=ring))
    torch.cuda.synchronize()
    fwd = {"ce": ce, "tvd": tvd, "student_lse": ls, "teacher_lse": lt, "sigma": sg}
    return fwd, grad, int(status.item())


@pytest.mark.parametrize("name,rows,V,dtype,ld", [
    ("bt8192_v151936_bf16", 40, 151936, torch.bfloat16, None),
    ("bt1024_v32000_bf16", 33, 32000, torch.bfloat16, None),
    ("bt4096_v256000_f32", 12, 256000, torch.float32, None),
    ("bt4096_v256000_f32", 21, 9001, torch.bfloat16, 9008),   # ragged tail, aligned rows
    ("bt4096_v256000_f32", 21, 9001, torch.float32, 9004),    # ragged tail, aligned rows
    ("bt1024_v32000_bf16", 17, 3003, torch.bfloat16, None),   # unaligned stride: two launches
    ("bt1024_v32000_bf16", 9, 5, torch.float32, None),
])
@pytest.mark.parametrize("cluster", [0, 2, 8])
@pytest.mark.parametrize("ring", [0, 1])
def test_single_launch_equals_forward_then_backward(name, rows, V, dtype, ld, cluster, ring):
    w = workloads.make(name, DEV, rows=rows, V=V, dtype=dtype, seed=31)
    if ld is not None:
        w = padded(w, ld, 0)
    if rows > 3:
        w.target[1] = w.ignore_index
    f1, g1, st1 = run(w, cluster=cluster, ring=ring)
    f2, g2, st2 = run_single(w, cluster=cluster, ring=ring)
    assert st1 == st2 == 0
    for k in f1:
        assert torch.equal(f1[k], f2[k]), k
    assert torch.equal(g1, g2)
    _, g3, _ = run_single(w, cluster=cluster, inplace=True, ring=ring)
    assert torch.equal(g1, g3)
    if cluster == 0 and ring == 1:  # the per-thread ring at one CTA per row: the oracle too
        compare(w, f2, g2, what=f"cp.async {name} ")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("cluster", [0, 2])
def test_single_launch_ties_equal_forward_then_backward(dtype, cluster):
    # Rows with exact ties (teacher == student), near ties (teacher shifted by
    # a constant, so p and q agree to rounding and some elements tie exactly)
    # and a row tied on a block of columns only: the single launch must still
    # match forward + backward bit for bit, tie threads included.
    w = workloads.make("bt8192_v151936_bf16", DEV, rows=10, V=151936, dtype=dtype, seed=33)
    w.teacher[2] = w.student[2]
    w.teacher[3] = (w.student[3].float() + 1.0).to(dtype)
    w.teacher[4] = (w.student[4].float() - 0.5).to(dtype)
    w.teacher[6, 1000:70000] = w.student[6, 1000:70000]
    w.target[8] = w.ignore_index
    f1, g1, st1 = run(w, cluster=cluster)
    f2, g2, st2 = run_single(w, cluster=cluster)
    assert st1 == st2 == 0
    for k in f1:
        assert torch.equal(f1[k], f2[k]), k
    assert torch.equal(g1, g2)
    assert f2["tvd"][2].item() == 0.0 and f2["sigma"][2].item() == 0.0


@pytest.mark.parametrize("cluster", [0, 2])
def test_subnormal_probability_differences(cluster):
    # Elements whose p and q are normal floats just above 2^-126 and differ
    # by a subnormal amount: teacher == student except one ulp up at those
    # elements, so both rows keep the same lse and p - q is about 1e-43.
    # Step 2 then takes a fractional sign there and flags the thread for the
    # exact teacher path in step 3; the outputs stay within the oracle's
    # near-tie tolerances and the single launch equals forward + backward.
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=4, V=4096, dtype=torch.float32, seed=35)
    w.teacher.copy_(w.student)
    for r, cols in ((0, slice(100, 164)), (1, slice(0, 4096, 37)), (3, slice(4000, 4096))):
        w.student[r, cols] = -78.0
        w.teacher[r, cols] = torch.nextafter(w.student[r, cols], torch.zeros_like(w.student[r, cols]))
    w.teacher[2] = w.student[2] * 0.9 + 0.1  # a plain row beside them
    f1, g1, st1 = run(w, cluster=cluster)
    f2, g2, st2 = run_single(w, cluster=cluster)
    assert st1 == st2 == 0
    for k in f1:
        assert torch.equal(f1[k], f2[k]), k
    assert torch.equal(g1, g2)
    compare(w, f2, g2, what="subnormal differences ")


@pytest.mark.parametrize("dtype,V,ld", [(torch.bfloat16, 300003, 300008),
                                        (torch.float32, 140001, 140004)])
def test_single_launch_without_sign_words(dtype, V, ld):
    # One CTA per row over a long row: more steps per thread than the shared
    # memory keeps sign words for, so the third pass re-reads the teacher.
    # (Rows padded to 16-byte strides: the vector path, which the single
    # launch needs.)
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=6, V=V, dtype=dtype, seed=34)
    w = padded(w, ld, 0)
    w.teacher[1] = w.student[1]
    w.target[4] = w.ignore_index
    f1, g1, st1 = run(w, cluster=1)
    f2, g2, st2 = run_single(w, cluster=1)
    assert st1 == st2 == 0
    for k in f1:
        assert torch.equal(f1[k], f2[k]), k
    assert torch.equal(g1, g2)
    compare(w, f2, g2, what="long rows ")


def test_single_launch_parity_and_status():
    w = workloads.make("bt8192_v151936_bf16", DEV, rows=24, V=151936, seed=32)
    w.teacher[5] = w.student[5]
    w.target[7] = 151936          # out of range
    fwd, grad, st = run_single(w)
    assert st == binding.FCT_DEV_TARGET_OUT_OF_RANGE
    compare(w, fwd, grad, what="single ")
    assert fwd["tvd"][5].item() == 0.0 and fwd["sigma"][5].item() == 0.0
    # broadcast upstream scalars
    _, g_b, _ = run_single(w, grads=(0.125, 0.5))
    _, g_r, _ = run_single(w, grads=(torch.full((24,), 0.125, device=DEV),
                                     torch.full((24,), 0.5, device=DEV)))
    assert torch.equal(g_b[~torch.isnan(g_b.float()).any(1)], g_r[~torch.isnan(g_r.float()).any(1)])



@pytest.mark.parametrize("name", FULL)
def test_full_size_single_launch_every_row(name):
    """Each full-size workload in the bench's launch (one forward + backward
    launch per step, all rows): bitwise equal to forward then backward, and
    every per-row output and every gradient element against the oracle,
    streamed by row blocks."""
    w = workloads.make(name, DEV)
    f1, g1, st1 = run(w)
    f2, g2, st2 = run_single(w)
    assert st1 == st2 == 0
    for k in f1:
        assert torch.equal(f1[k], f2[k]), k
    assert torch.equal(g1, g2)
    del f1, g1
    check_every_row(w, f2, g2, name)


# ------------------------------------------------------------------ bulk-copy (TMA) ring

@pytest.mark.parametrize("dtype,V,ld,rows", [
    (torch.bfloat16, 151936, None, 40),
    (torch.bfloat16, 20003, 20008, 21),     # ragged tail, aligned rows
    (torch.float32, 9001, 9004, 17),        # fp32, ragged tail
    (torch.bfloat16, 300003, 300008, 6),    # more steps than sign words: teacher re-read
    (torch.bfloat16, 5, 8, 9),              # no full vector at all
    (torch.float32, 3, 4, 9),
    (torch.bfloat16, 4100, None, 200),      # several rows per CTA
    (torch.bfloat16, 1000, None, 5000),     # enough rows per CTA for the start stagger
    # step 3 takes step 2's last 3 steps from the ring: 3 steps (none left
    # to stage), 4 steps (one), and fp32 with two steps per sign word
    (torch.bfloat16, 40003, 40008, 400),
    (torch.bfloat16, 60000, None, 400),
    (torch.float32, 100003, 100004, 320),
    (torch.bfloat16, 49152, None, 300),     # last step exactly full (3 steps)
    (torch.float32, 16384, None, 300),      # last step exactly full (2 steps)
])
def test_tma_ring_single_launch_equals_forward_then_backward(dtype, V, ld, rows):
    """The producer-warp bulk-copy ring: its single launch equals its forward
    followed by the backward bit for bit (out of place and in place), both
    rings agree with the oracle, and with each other within the tolerances
    (their step-1 partial sums are grouped differently)."""
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=rows, V=V, dtype=dtype, seed=61)
    if ld is not None:
        w = padded(w, ld, 0)
    w.teacher[2] = w.student[2]                                   # exact ties
    w.teacher[3] = (w.student[3].float() + 1.0).to(dtype)         # near ties
    w.target[1] = w.ignore_index
    w.target[4] = V + 3                                           # out of range
    names = ("ce", "tvd", "student_lse", "teacher_lse", "sigma")
    opts = binding.options(ctas_per_row=1, ring=binding.RING_TMA)
    st1 = torch.zeros(1, dtype=torch.int32, device=DEV)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    single = binding.fused_ce_tvd_forward_backward(w.student, w.teacher, w.target, w.grad_ce,
                                                   w.grad_tvd, dev_status=st1, options=opts)
    s_in = same_layout_clone(w.student)
    inplace = binding.fused_ce_tvd_forward_backward(s_in, w.teacher, w.target, w.grad_ce,
                                                    w.grad_tvd, inplace=True, options=opts)
    fwd = binding.fused_ce_tvd_forward(w.student, w.teacher, w.target, dev_status=st2,
                                       options=opts)
    g2 = binding.fused_ce_tvd_backward(w.student, w.teacher, w.target, *fwd[2:], w.grad_ce,
                                       w.grad_tvd, dev_status=st2)
    torch.cuda.synchronize()
    assert st1.item() == st2.item() == binding.FCT_DEV_TARGET_OUT_OF_RANGE
    for x, y in zip(single[:5], fwd):
        assert torch.equal(_bits(x), _bits(y))
    assert torch.equal(_bits(single[5]), _bits(g2))
    assert torch.equal(_bits(single[5]), _bits(inplace[5]))
    for x, y in zip(single[:5], inplace[:5]):
        assert torch.equal(_bits(x), _bits(y))
    # the sign-word pair on the same ring
    f3 = binding.fused_ce_tvd_forward_signs(w.student, w.teacher, w.target, options=opts)
    g3 = binding.fused_ce_tvd_backward_signs(w.student, w.teacher, w.target, *f3[2:5], f3[5],
                                             w.grad_ce, w.grad_tvd)
    torch.cuda.synchronize()
    for x, y in zip(single[:5], f3[:5]):
        assert torch.equal(_bits(x), _bits(y))
    assert torch.equal(_bits(single[5]), _bits(g3))
    compare(w, dict(zip(names, single[:5])), single[5], what=f"tma {V} ")
    # the per-thread ring on the same rows: the oracle's tolerances apart at most
    fa, ga, _ = run_single(w, cluster=1, ring=binding.RING_CP_ASYNC)
    compare(w, fa, ga, what=f"cp.async {V} ")
    if V >= 8 and rows == 40:  # same tie pattern, so identical NaN and zero rows
        assert torch.equal(torch.isnan(ga.float()), torch.isnan(single[5].float()))


def test_tma_ring_randomised_shapes():
    """Seeded random row lengths (many near a step boundary of the ring),
    dtypes, row strides and row counts: the bulk-copy ring's single launch
    equals its forward + backward bit for bit, out of place and in place,
    and the oracle on sampled rows (including an exact-tie row and an
    ignored row)."""
    import random
    rng = random.Random(20261203)
    opts = binding.options(ctas_per_row=1, ring=binding.RING_TMA)
    names = ("ce", "tvd", "student_lse", "teacher_lse", "sigma")
    for i in range(20):
        dtype = rng.choice([torch.bfloat16, torch.float32])
        ve = 8 if dtype == torch.bfloat16 else 4
        if rng.random() < 0.5:
            V = max(1, rng.randint(1, 20) * 2048 * ve + rng.randint(-9, 9))
        else:
            V = rng.randint(1, 320000)
        ld = (V + ve - 1) // ve * ve + ve * rng.randint(0, 3)
        rows = rng.randint(4, 600)
        w = padded(workloads.make("bt1024_v32000_bf16", DEV, rows=rows, V=V, dtype=dtype,
                                  seed=300 + i), ld, 0)
        w.teacher[rows // 2] = w.student[rows // 2]
        w.target[rows // 3] = w.ignore_index
        single = binding.fused_ce_tvd_forward_backward(w.student, w.teacher, w.target, w.grad_ce,
                                                       w.grad_tvd, options=opts)
        s_in = same_layout_clone(w.student)
        inplace = binding.fused_ce_tvd_forward_backward(s_in, w.teacher, w.target, w.grad_ce,
                                                        w.grad_tvd, inplace=True, options=opts)
        fwd = binding.fused_ce_tvd_forward(w.student, w.teacher, w.target, options=opts)
        g2 = binding.fused_ce_tvd_backward(w.student, w.teacher, w.target, *fwd[2:], w.grad_ce,
                                           w.grad_tvd)
        torch.cuda.synchronize()
        what = f"random {i} (V {V}, ld {ld}, rows {rows}) "
        for x, y in zip(single[:5], fwd):
            assert torch.equal(_bits(x), _bits(y)), what
        assert torch.equal(_bits(single[5]), _bits(g2)), what
        assert torch.equal(_bits(single[5]), _bits(inplace[5])), what
        sample = sorted({rows // 2, rows // 3, rows - 1, *rng.sample(range(rows), min(rows, 8))})
        compare(w, dict(zip(names, single[:5])), single[5], rows=torch.tensor(sample), what=what)


def test_tma_ring_falls_back_on_clusters():
    # A row split over a cluster has no bulk-copy form: the call takes the
    # per-thread ring and gives its results.
    w = workloads.make("bt4096_v256000_f32", DEV, rows=10, V=20011, seed=62)
    r1 = binding.fused_ce_tvd_forward_backward(w.student, w.teacher, w.target, w.grad_ce,
                                               w.grad_tvd, options=binding.options(2, ring=1))
    r2 = binding.fused_ce_tvd_forward_backward(w.student, w.teacher, w.target, w.grad_ce,
                                               w.grad_tvd, options=binding.options(2, ring=2))
    torch.cuda.synchronize()
    for x, y in zip(r1, r2):
        assert torch.equal(x, y)


# ------------------------------------------------------------------ mean over tokens

def test_mean_front_end_and_autograd_loss():
    from distillation_ce_tvd_gb300.autograd import fused_ce_tvd_mean_loss
    w = workloads.make("bt1024_v151936_bf16", DEV, rows=30, V=20000, seed=41)
    w.target[[3, 4]] = w.ignore_index
    alpha, beta = 0.8, 1.7
    gce, gtvd, n = binding.fused_ce_tvd_mean_upstream(w.target, w.ignore_index, alpha, beta)
    fwd, grad, st = run_single(w, grads=(gce, gtvd))
    loss = binding.fused_ce_tvd_mean_loss(fwd["ce"], fwd["tvd"], w.target, w.ignore_index,
                                          alpha, beta)
    torch.cuda.synchronize()
    n_kept = int((w.target != w.ignore_index).sum().item())
    assert st == 0 and int(n.item()) == n_kept
    # fp32 results of alpha/n and beta/n: exact to one rounding
    assert abs(gce.item() - alpha / n_kept) <= 1e-7 * alpha / n_kept
    assert abs(gtvd.item() - beta / n_kept) <= 1e-7 * beta / n_kept
    ref = oracle.mean_loss(fwd["ce"].cpu().numpy(), fwd["tvd"].cpu().numpy(),
                           w.target.cpu().numpy(), w.ignore_index, alpha, beta)
    assert abs(loss.item() - ref[0]) < 1e-6
    # the gradient of the mean loss against the oracle's, row by row
    s, t = w.student.cpu(), w.teacher.cpu()
    tg = w.target.cpu().numpy()
    ref_grad, _ = oracle.fused_ce_tvd_backward(s, t, tg, ref[1], ref[2], w.ignore_index)
    masks, mass, probs = tie_info(s, t)
    check_grad(grad.cpu().double().numpy(), ref_grad, np.full(30, ref[2]), masks, mass, probs,
               tg, w.ignore_index, "mean ", grad.dtype)
    # autograd wrapper: same loss and gradient
    sv = w.student.clone().requires_grad_(True)
    lv = fused_ce_tvd_mean_loss(sv, w.teacher, w.target, w.ignore_index, alpha, beta)
    lv.backward()
    assert torch.equal(lv.detach().reshape(1), loss)
    assert torch.equal(sv.grad, grad)


def test_mean_front_end_all_ignored():
    tg = torch.full((5,), -100, device=DEV, dtype=torch.int64)
    gce, gtvd, n = binding.fused_ce_tvd_mean_upstream(tg, -100, 1.0, 1.0)
    z = torch.zeros(5, device=DEV)
    loss = binding.fused_ce_tvd_mean_loss(z, z, tg)
    torch.cuda.synchronize()
    assert n.item() == 0 and gce.item() == 0 and gtvd.item() == 0 and loss.item() == 0


def _bits(x):
    x = x.contiguous()
    return x.view(torch.int32 if x.element_size() == 4 else torch.int16)


@pytest.mark.parametrize("dtype,V,host_ld,block_rows,scalar", [
    (torch.bfloat16, 32000, None, 16, False),
    (torch.bfloat16, 32003, 32010, 7, True),      # ragged V, padded host rows, broadcast grads
    (torch.float32, 9001, None, 64, False),       # block larger than the batch
    (torch.bfloat16, 151936, None, 32, False),
])
def test_host_entry_point_equals_device_call(dtype, V, host_ld, block_rows, scalar):
    """The host-buffer entry point (copies in and out on its own streams, row
    blocks through a three-slot device ring) gives bit for bit the device
    single launch's outputs, the gradient included, and the status bits."""
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=45, V=V, dtype=dtype, seed=51)
    w.target[3] = w.ignore_index
    w.target[9] = V + 4                       # out of range: NaN row, status bit
    w.teacher[5] = w.student[5]               # exact ties
    grads = (0.125, 0.5) if scalar else (w.grad_ce, w.grad_tvd)
    # the device reference on rows padded to a 16-byte stride, as the
    # entry point's device slots are (the same kernel and reduction order)
    vec = 16 // w.student.element_size()
    ld_dev = (V + vec - 1) // vec * vec
    ref_w = padded(w, ld_dev, 0) if ld_dev != V else w
    f1, g1, st1 = run_single(ref_w, grads=grads)
    assert st1 == binding.FCT_DEV_TARGET_OUT_OF_RANGE

    def host(x, ld=None):
        if ld is None:
            return x.cpu().pin_memory()
        buf = torch.full((x.shape[0], ld), 3.0, dtype=x.dtype).pin_memory()
        buf[:, :x.shape[1]] = x.cpu()
        return buf[:, :x.shape[1]]

    hs, ht = host(w.student, host_ld), host(w.teacher, host_ld)
    htg = w.target.cpu().pin_memory()
    if scalar:
        hgce, hgtvd = torch.tensor([0.125]), torch.tensor([0.5])
    else:
        hgce, hgtvd = w.grad_ce.cpu().pin_memory(), w.grad_tvd.cpu().pin_memory()
    status = torch.zeros(1, dtype=torch.int32).pin_memory()
    grad_h = torch.full((45, host_ld or V), 9.0, dtype=dtype).pin_memory()[:, :V]
    out = binding.fused_ce_tvd_forward_backward_host(
        hs, ht, htg, hgce, hgtvd, w.ignore_index, block_rows=block_rows, grad_student=grad_h,
        status=status)
    torch.cuda.synchronize()
    assert status.item() == st1
    for k, v in zip(("ce", "tvd", "student_lse", "teacher_lse", "sigma"), out[:5]):
        assert torch.equal(_bits(f1[k].cpu()), _bits(v)), k
    assert torch.equal(_bits(g1.cpu()), _bits(out[5]))
    if host_ld is not None:  # the padding of the host gradient rows is untouched
        assert torch.all(grad_h.as_strided((45, host_ld - V), (host_ld, 1), V) == 9.0)


def test_host_entry_point_without_gradient_and_tiny_workspace_checks():
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=10, V=4000, seed=52)
    f1, _, _ = run_single(w)
    hs, ht, htg = (x.cpu().pin_memory() for x in (w.student, w.teacher, w.target))
    hg = w.grad_ce.cpu().pin_memory(), w.grad_tvd.cpu().pin_memory()
    out = binding.fused_ce_tvd_forward_backward_host(hs, ht, htg, *hg, want_grad=False,
                                                     block_rows=3)
    torch.cuda.synchronize()
    assert out[5] is None
    assert torch.equal(_bits(f1["ce"].cpu()), _bits(out[0]))
    need = binding.fused_ce_tvd_host_workspace_size(4000, torch.bfloat16, 3)
    small = torch.empty(need - 256, device=DEV, dtype=torch.uint8)
    with pytest.raises(binding.FctError) as e:
        binding.fused_ce_tvd_forward_backward_host(hs, ht, htg, *hg, block_rows=3,
                                                   workspace=small)
    assert e.value.status == 1


# ------------------------------------------------------------------ fused linear (chunked)

def _linear_case(BT, ds, dt, V, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    hs = torch.randn(BT, ds, generator=g, device=DEV).bfloat16()
    ht = torch.randn(BT, dt, generator=g, device=DEV).bfloat16()
    ws = (torch.randn(V, ds, generator=g, device=DEV) * (2.0 / ds ** 0.5)).bfloat16()
    wt = (torch.randn(V, dt, generator=g, device=DEV) * (2.0 / dt ** 0.5)).bfloat16()
    tg = torch.randint(0, V, (BT,), generator=g, device=DEV)
    tg[::7] = -100
    return hs, ws, ht, wt, tg


@pytest.mark.parametrize("BT,ds,dt,V,chunk", [(50, 128, 96, 1003, 16), (64, 256, 256, 4096, 64),
                                              (33, 64, 128, 2048, 100)])
def test_fused_linear_against_fp64(BT, ds, dt, V, chunk):
    hs, ws, ht, wt, tg = _linear_case(BT, ds, dt, V, seed=BT + V)
    gce = torch.full((BT,), 1.0 / BT, device=DEV)
    gtvd = torch.full((BT,), 0.7 / BT, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ce, tvd, ls, lt, sg, gh, gw = binding.fused_linear_ce_tvd_forward_backward(
        hs, ws, ht, wt, tg, gce, gtvd, chunk_rows=chunk, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    # fp64 reference: library matmuls for the logits, the oracle for the loss
    Hs, Ws, Ht, Wt = (x.cpu().double() for x in (hs, ws, ht, wt))
    Ls, Lt = Hs @ Ws.T, Ht @ Wt.T
    tgc = tg.cpu().numpy()
    ref = oracle.fused_ce_tvd_forward(Ls, Lt, tgc)
    G, _ = oracle.fused_ce_tvd_backward(Ls, Lt, tgc, gce.cpu().numpy(), gtvd.cpu().numpy())
    masks, mass, probs = tie_info(Ls, Lt)
    got = {"ce": ce, "tvd": tvd, "student_lse": ls, "teacher_lse": lt, "sigma": sg}
    # The GPU's logits are fp32 sums of D exact bf16 products: each is off by
    # at most D * 2^-24 * sum_k |h_k w_vk|; every per-row output moves by at
    # most twice the largest logit error on top of the fp32 tolerance.
    bound = np.maximum((np.abs(Hs.numpy()) @ np.abs(Ws.numpy()).T).max(1) * ds,
                       (np.abs(Ht.numpy()) @ np.abs(Wt.numpy()).T).max(1) * dt) * 2.0 ** -24
    check_forward(torch.float32, tgc, {k: v.cpu().numpy() for k, v in got.items()}, ref, mass,
                  what="linear ", atol=1e-5 + 2.0 * bound)
    check_linear_grads(gh, gw, G, Hs.numpy(), Ws.numpy())


def check_linear_grads(gh, gw, G, Hs, Ws, what=""):
    """d hidden and d weight against G @ Ws and G.T @ Hs in fp64 (G: the
    oracle's logit gradient).  Bounds: the logit gradient is rounded to bf16
    (2^-8 relative) on top of its own tolerance (2e-3 relative, 1e-6
    absolute), the GEMMs sum in fp32, and d hidden is itself rounded to bf16."""
    BT, V = G.shape
    G_abs = np.abs(G)
    e_rel = 2.0 ** -8 + 2e-3 + V * 2.0 ** -24
    ref_gh = G @ Ws
    tol_gh = e_rel * (G_abs @ np.abs(Ws)) + 1e-6 * np.abs(Ws).sum(0) \
        + 2.0 ** -8 * np.abs(ref_gh) + 1e-9
    err_gh = np.abs(gh.cpu().double().numpy() - ref_gh)
    assert np.all(err_gh <= tol_gh), f"{what}grad_h {float((err_gh / tol_gh).max())}"
    ref_gw = G.T @ Hs
    e_rel_w = 2.0 ** -8 + 2e-3 + BT * 2.0 ** -24
    tol_gw = e_rel_w * (G_abs.T @ np.abs(Hs)) + 1e-6 * np.abs(Hs).sum(0) + 1e-9
    err_gw = np.abs(gw.cpu().double().numpy() - ref_gw)
    assert np.all(err_gw <= tol_gw), f"{what}grad_w {float((err_gw / tol_gw).max())}"


def _dyadic_linear_case(BT, ds, dt, V, seed, wden=16.0):
    """Hidden states in quarters up to 3/4 and weights in multiples of 1/wden
    up to 7/wden: every product is a multiple of 1/(4 wden) and every partial
    sum stays below 2^24 / (4 wden) in magnitude (d * 3/4 * 7/wden * 4 wden =
    21 d < 2^24), so the GEMMs' fp32 sums are exact in any order and the
    logits the loss kernel reads are known exactly on the host."""
    assert 21 * max(ds, dt) < 2 ** 24
    g = torch.Generator(device=DEV).manual_seed(seed)

    def q(shape, k, den):
        x = torch.randint(-k, k + 1, shape, generator=g, device=DEV, dtype=torch.int16)
        return x.to(torch.bfloat16).div_(den)
    hs, ht = q((BT, ds), 3, 4.0), q((BT, dt), 3, 4.0)
    ws, wt = q((V, ds), 7, wden), q((V, dt), 7, wden)
    tg = torch.randint(0, V, (BT,), generator=g, device=DEV)
    tg[::7] = -100
    return hs, ws, ht, wt, tg


@pytest.mark.parametrize("logits_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("BT,ds,dt,V,chunk", [(50, 128, 96, 1003, 16), (33, 64, 256, 2048, 100),
                                              (20, 256, 128, 151936, 8)])
def test_fused_linear_exact_logits(logits_dtype, BT, ds, dt, V, chunk):
    # With exact GEMMs the loss sees known logits (rounded once to bf16 for
    # bf16 blocks), so the per-row outputs meet the logit-level tolerances of
    # that element type, and they do not depend on the block size.
    hs, ws, ht, wt, tg = _dyadic_linear_case(BT, ds, dt, V, seed=3 * BT + V)
    gce = torch.full((BT,), 1.0 / BT, device=DEV)
    gtvd = torch.full((BT,), 0.7 / BT, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = binding.fused_linear_ce_tvd_forward_backward(
        hs, ws, ht, wt, tg, gce, gtvd, chunk_rows=chunk, logits_dtype=logits_dtype,
        dev_status=status)
    other = binding.fused_linear_ce_tvd_forward_backward(
        hs, ws, ht, wt, tg, gce, gtvd, chunk_rows=BT, logits_dtype=logits_dtype)
    torch.cuda.synchronize()
    assert status.item() == 0
    for k in range(5):
        assert torch.equal(out[k], other[k]), k
    Hs, Ws, Ht, Wt = (x.cpu().double() for x in (hs, ws, ht, wt))
    Ls, Lt = (Hs @ Ws.T), (Ht @ Wt.T)
    assert torch.equal(Ls, Ls.float().double()) and torch.equal(Lt, Lt.float().double())
    if logits_dtype == torch.bfloat16:
        Ls, Lt = Ls.float().bfloat16().double(), Lt.float().bfloat16().double()
    Ls, Lt = Ls.numpy(), Lt.numpy()
    tgc = tg.cpu().numpy()
    ref = oracle.fused_ce_tvd_forward(Ls, Lt, tgc)
    G, _ = oracle.fused_ce_tvd_backward(Ls, Lt, tgc, gce.cpu().numpy(), gtvd.cpu().numpy())
    masks, mass, probs = tie_info(Ls, Lt)
    got = dict(zip(("ce", "tvd", "student_lse", "teacher_lse", "sigma"),
                   (x.cpu().numpy() for x in out[:5])))
    check_forward(logits_dtype, tgc, got, ref, mass, what="linear exact ")
    check_linear_grads(out[5], out[6], G, Hs.numpy(), Ws.numpy(), what="linear exact ")


def test_fused_linear_chunking_is_invisible():
    hs, ws, ht, wt, tg = _linear_case(70, 128, 128, 3000, seed=5)
    a = binding.fused_linear_ce_tvd_forward_backward(hs, ws, ht, wt, tg, 0.01, 0.02, chunk_rows=70)
    b = binding.fused_linear_ce_tvd_forward_backward(hs, ws, ht, wt, tg, 0.01, 0.02, chunk_rows=9)
    torch.cuda.synchronize()
    # The GEMMs may pick other algorithms (summation orders) for other block
    # sizes, so results agree to fp32 rounding rather than bit for bit.
    for x, y in zip(a[:5], b[:5]):
        assert torch.allclose(x, y, rtol=0, atol=2e-5)
    assert torch.allclose(a[5].float(), b[5].float(), rtol=2 ** -7, atol=1e-7)
    assert torch.allclose(a[6], b[6], rtol=1e-3, atol=1e-7)


def test_fused_linear_autograd_wrapper_matches_direct_calls():
    from distillation_ce_tvd_gb300.autograd import fused_linear_ce_tvd_mean_loss
    hs, ws, ht, wt, tg = _linear_case(90, 128, 96, 3001, seed=11)
    alpha, beta = 0.6, 1.3
    gce, gtvd, _ = binding.fused_ce_tvd_mean_upstream(tg, -100, alpha, beta)
    direct = binding.fused_linear_ce_tvd_forward_backward(hs, ws, ht, wt, tg, gce, gtvd,
                                                          chunk_rows=32)
    ref_loss = binding.fused_ce_tvd_mean_loss(direct[0], direct[1], tg, -100, alpha, beta)

    h = hs.clone().requires_grad_(True)
    w = ws.clone().requires_grad_(True)
    loss = fused_linear_ce_tvd_mean_loss(h, w, ht, wt, tg, -100, alpha, beta, chunk_rows=32)
    (2.0 * loss).backward()
    torch.cuda.synchronize()
    assert loss.shape == () and torch.equal(loss.detach(), ref_loss.reshape(()))
    assert torch.equal(h.grad, direct[5] * 2.0)
    assert w.grad.dtype == torch.bfloat16
    assert torch.equal(w.grad, (direct[6] * 2.0).to(torch.bfloat16))

    # only the hidden states need a gradient: the weight-gradient GEMM is skipped
    h2 = hs.clone().requires_grad_(True)
    fused_linear_ce_tvd_mean_loss(h2, ws, ht, wt, tg, -100, alpha, beta, chunk_rows=32).backward()
    torch.cuda.synchronize()
    assert torch.equal(h2.grad, direct[5])

    # bf16 logit blocks through the wrapper
    direct = binding.fused_linear_ce_tvd_forward_backward(hs, ws, ht, wt, tg, gce, gtvd,
                                                          chunk_rows=32,
                                                          logits_dtype=torch.bfloat16)
    h3 = hs.clone().requires_grad_(True)
    loss = fused_linear_ce_tvd_mean_loss(h3, ws, ht, wt, tg, -100, alpha, beta, chunk_rows=32,
                                         logits_dtype=torch.bfloat16)
    loss.backward()
    torch.cuda.synchronize()
    assert torch.equal(h3.grad, direct[5])
    assert torch.equal(loss.detach(), binding.fused_ce_tvd_mean_loss(
        direct[0], direct[1], tg, -100, alpha, beta).reshape(()))


def test_fused_linear_other_ignore_index():
    BT, d, V = 40, 64, 1003
    hs, ws, ht, wt, tg = _dyadic_linear_case(BT, d, d, V, seed=13)
    tg[tg == -100] = 3
    tg[::5] = -1
    gce = torch.full((BT,), 1.0 / BT, device=DEV)
    gtvd = torch.full((BT,), 0.5 / BT, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = binding.fused_linear_ce_tvd_forward_backward(hs, ws, ht, wt, tg, gce, gtvd, -1,
                                                       chunk_rows=16, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    Ls = (hs.cpu().double() @ ws.cpu().double().T).numpy()
    Lt = (ht.cpu().double() @ wt.cpu().double().T).numpy()
    tgc = tg.cpu().numpy()
    ref = oracle.fused_ce_tvd_forward(Ls, Lt, tgc, -1)
    G, _ = oracle.fused_ce_tvd_backward(Ls, Lt, tgc, gce.cpu().numpy(), gtvd.cpu().numpy(), -1)
    _, mass, _ = tie_info(Ls, Lt)
    got = dict(zip(("ce", "tvd", "student_lse", "teacher_lse", "sigma"),
                   (x.cpu().numpy() for x in out[:5])))
    check_forward(torch.float32, tgc, got, ref, mass, -1, what="linear ignore -1 ")
    assert torch.all(out[5][::5] == 0)
    check_linear_grads(out[5], out[6], G, hs.cpu().double().numpy(), ws.cpu().double().numpy(),
                       what="linear ignore -1 ")


@pytest.mark.parametrize("logits_dtype", [torch.float32, torch.bfloat16])
def test_fused_linear_full_size_sampled_rows(logits_dtype):
    # The fused-linear bench workload's shapes and block size (8192 rows,
    # hidden 4096, V = 151936, 2048-row blocks) with exact GEMMs.  The
    # upstream gradients are nonzero on sampled rows only (block edges, an
    # ignored row, the last row), so every other logit-gradient row is
    # exactly 0 and the whole (V, d) weight gradient is a sum over the sampled
    # rows, which the oracle gives.
    BT, d, V, chunk = 8192, 4096, 151936, 2048
    hs, ws, ht, wt, tg = _dyadic_linear_case(BT, d, d, V, seed=41, wden=64.0)
    rows = torch.tensor([0, 7, 2047, 2048, 4095, 6001, 8191])
    assert int(tg[7]) == -100
    rows_d = rows.to(DEV)
    gce = torch.zeros(BT, device=DEV)
    gtvd = torch.zeros(BT, device=DEV)
    gce[rows_d], gtvd[rows_d] = 1.0 / 8, 0.5 / 8
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ce, tvd, ls, lt, sg, gh, gw = binding.fused_linear_ce_tvd_forward_backward(
        hs, ws, ht, wt, tg, gce, gtvd, chunk_rows=chunk, logits_dtype=logits_dtype,
        dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0

    Ws_h, Wt_h = ws.cpu(), wt.cpu()
    Hs_r, Ht_r = hs[rows_d].cpu().double(), ht[rows_d].cpu().double()
    n = rows.numel()
    Ls, Lt = torch.empty(n, V, dtype=torch.float64), torch.empty(n, V, dtype=torch.float64)
    step = 16384
    for v0 in range(0, V, step):
        Ls[:, v0:v0 + step] = Hs_r @ Ws_h[v0:v0 + step].double().T
        Lt[:, v0:v0 + step] = Ht_r @ Wt_h[v0:v0 + step].double().T
    assert torch.equal(Ls, Ls.float().double()) and torch.equal(Lt, Lt.float().double())
    if logits_dtype == torch.bfloat16:
        Ls, Lt = Ls.float().bfloat16().double(), Lt.float().bfloat16().double()
    Ls, Lt = Ls.numpy(), Lt.numpy()
    tgc = tg[rows_d].cpu().numpy()
    ref = oracle.fused_ce_tvd_forward(Ls, Lt, tgc)
    G, _ = oracle.fused_ce_tvd_backward(Ls, Lt, tgc, np.full(n, 1.0 / 8), np.full(n, 0.5 / 8))
    masks, mass, probs = tie_info(Ls, Lt)
    got = {k: v[rows_d].cpu().numpy()
           for k, v in zip(("ce", "tvd", "student_lse", "teacher_lse", "sigma"),
                           (ce, tvd, ls, lt, sg))}
    check_forward(logits_dtype, tgc, got, ref, mass, what="linear full size ")

    # d hidden: zero outside the sampled rows; on them, the bounds of
    # check_linear_grads with the fp64 products summed over vocabulary slices
    others = torch.ones(BT, dtype=torch.bool, device=DEV)
    others[rows_d] = False
    assert torch.all(gh[others] == 0)
    Hs_abs = np.abs(Hs_r.numpy())
    ref_gh = np.zeros((n, d))
    abs_gh = np.zeros((n, d))
    w_abs_sum = np.zeros(d)
    for v0 in range(0, V, step):
        Wc = Ws_h[v0:v0 + step].double().numpy()
        ref_gh += G[:, v0:v0 + step] @ Wc
        abs_gh += np.abs(G[:, v0:v0 + step]) @ np.abs(Wc)
        w_abs_sum += np.abs(Wc).sum(0)
    e_rel = 2.0 ** -8 + 2e-3 + V * 2.0 ** -24
    tol_gh = e_rel * abs_gh + 1e-6 * w_abs_sum + 2.0 ** -8 * np.abs(ref_gh) + 1e-9
    err_gh = np.abs(gh[rows_d].cpu().double().numpy() - ref_gh)
    assert np.all(err_gh <= tol_gh), float((err_gh / tol_gh).max())

    # d weight, all V x d entries, against G.T @ H of the sampled rows
    gw_h = gw.cpu()
    e_rel_w = 2.0 ** -8 + 2e-3 + BT * 2.0 ** -24
    h_abs_sum = Hs_abs.sum(0)
    worst = 0.0
    for v0 in range(0, V, step):
        Gc = G[:, v0:v0 + step]
        ref_gw = Gc.T @ Hs_r.numpy()
        tol_gw = e_rel_w * (np.abs(Gc).T @ Hs_abs) + 1e-6 * h_abs_sum + 1e-9
        err_gw = np.abs(gw_h[v0:v0 + step].double().numpy() - ref_gw)
        worst = max(worst, float((err_gw / tol_gw).max()))
    assert worst <= 1.0, worst
