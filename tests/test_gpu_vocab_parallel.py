"""The vocabulary-parallel split on one GPU: the vocabulary cut into 2-4
column shards, each shard's passes through the C ABI, the partials merged by
the library, and every per-row output and every gradient element compared
with the oracle (which sees whole rows)."""
import numpy as np
import pytest
import torch

from distillation_ce_tvd_gb300 import binding, vocab_parallel, workloads
from parity_util import check_every_row, tie_info
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"
NAMES = ("ce", "tvd", "student_lse", "teacher_lse", "sigma")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def run_vp(w, n_shards):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = vocab_parallel.forward_backward_local(w.student, w.teacher, w.target, n_shards,
                                                w.grad_ce, w.grad_tvd, w.ignore_index,
                                                dev_status=status)
    torch.cuda.synchronize()
    return dict(zip(NAMES, out[:5])), out[5], int(status.item())


@pytest.mark.parametrize("name,n_shards", [("bt1024_v151936_bf16", 2), ("bt1024_v151936_bf16", 3),
                                           ("bt4096_v256000_f32", 4)])
def test_vocab_shards_every_row_full_size(name, n_shards):
    """Full-size workloads, every row and every gradient element against the
    oracle; the single launch on whole rows agrees within the same tolerances."""
    w = workloads.make(name, DEV)
    fwd, grad, st = run_vp(w, n_shards)
    assert st == 0
    check_every_row(w, fwd, grad, f"{name}/{n_shards} shards")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V,bounds", [
    (20003, None),                   # even split, ragged last shard
    (20000, [0, 1001, 20000]),       # a shard starting off a 16-byte boundary: element loads
    (5000, [0, 8, 16, 5000]),        # tiny shards
    (7, None),                       # fewer columns than a vector
])
def test_vocab_shards_layouts_ties_and_status(dtype, V, bounds):
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=40, V=V, dtype=dtype, seed=71)
    w.teacher[2] = w.student[2]                                   # exact ties
    w.teacher[3] = (w.student[3].float() + 1.0).to(dtype)         # near ties
    w.target[5] = w.ignore_index
    w.target[6] = V + 9                                           # out of range
    w.target[7] = V - 1                                           # the last column
    w.target[8] = 0
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    if bounds is None:
        fwd, grad, st = run_vp(w, 3)
    else:
        # explicit shard bounds through the step's building blocks
        views = [(w.student[:, b:e], w.teacher[:, b:e], b, e) for b, e in zip(bounds, bounds[1:])]
        p1 = torch.stack([binding.fused_ce_tvd_vp_lse(s, t, w.target, b) for s, t, b, _ in views])
        ce, ls, lt = binding.fused_ce_tvd_vp_merge_lse(p1, w.target, V, dev_status=status)
        p2 = torch.stack([binding.fused_ce_tvd_vp_tvd(s, t, w.target, ls, lt) for s, t, _, _ in views])
        tvd, sg = binding.fused_ce_tvd_vp_merge_tvd(p2, w.target)
        grad = torch.empty_like(w.student)
        for s, t, b, e in views:
            binding.fused_ce_tvd_vp_backward(s, t, w.target, b, V, ls, lt, sg, w.grad_ce,
                                             w.grad_tvd, grad_student=grad[:, b:e],
                                             dev_status=status)
        torch.cuda.synchronize()
        fwd, st = dict(zip(NAMES, (ce, tvd, ls, lt, sg))), int(status.item())
    assert st == binding.FCT_DEV_TARGET_OUT_OF_RANGE
    # teacher == student: identical shard code on identical bytes, exact zeros
    assert fwd["tvd"][2].item() == 0.0 and fwd["sigma"][2].item() == 0.0
    assert torch.isnan(fwd["ce"][6]) and torch.isnan(grad[6].float()).all()
    check_every_row(w, fwd, grad, f"vp {V} {dtype}")


def test_vocab_shards_in_place_and_broadcast_grads():
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=24, V=10000, seed=72)
    V = w.V
    fwd, grad, _ = run_vp(w, 2)
    # in place over each shard's student columns, broadcast upstream grads
    s_copy = w.student.clone()
    views = [(s_copy[:, b:e], w.teacher[:, b:e], b) for b, e in
             (vocab_parallel.shard_bounds(V, 2, k) for k in range(2))]
    for s, t, b in views:
        binding.fused_ce_tvd_vp_backward(s, t, w.target, b, V, fwd["student_lse"],
                                         fwd["teacher_lse"], fwd["sigma"], w.grad_ce, w.grad_tvd,
                                         inplace=True)
    torch.cuda.synchronize()
    assert torch.equal(s_copy, grad)
    g_b = [binding.fused_ce_tvd_vp_backward(w.student[:, b:e], w.teacher[:, b:e], w.target, b, V,
                                            fwd["student_lse"], fwd["teacher_lse"], fwd["sigma"],
                                            0.25, 0.5)
           for b, e in (vocab_parallel.shard_bounds(V, 2, k) for k in range(2))]
    g_r = [binding.fused_ce_tvd_vp_backward(w.student[:, b:e], w.teacher[:, b:e], w.target, b, V,
                                            fwd["student_lse"], fwd["teacher_lse"], fwd["sigma"],
                                            torch.full((24,), 0.25, device=DEV),
                                            torch.full((24,), 0.5, device=DEV))
           for b, e in (vocab_parallel.shard_bounds(V, 2, k) for k in range(2))]
    torch.cuda.synchronize()
    for a, b in zip(g_b, g_r):
        assert torch.equal(a, b)


def test_vocab_shards_argument_checks():
    w = workloads.make("bt1024_v32000_bf16", DEV, rows=4, V=100, seed=73)
    p = torch.zeros(2, 4, 3, device=DEV)
    flat = p.view(-1)
    with pytest.raises(binding.FctError):        # an output inside the partials
        binding.fused_ce_tvd_vp_merge_lse(p, w.target, 100, ce=flat[:4])
    with pytest.raises(ValueError):
        binding.fused_ce_tvd_vp_merge_lse(p[:, :, :2].contiguous(), w.target, 100)
    with pytest.raises(binding.FctError):        # the shard must lie inside the vocabulary
        binding.fused_ce_tvd_vp_backward(w.student[:, 50:], w.teacher[:, 50:], w.target, 60, 100,
                                         *(torch.zeros(4, device=DEV) for _ in range(3)), 1.0, 1.0)
