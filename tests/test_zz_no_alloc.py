"""The no-allocation fused-linear entry point against the oracle (fp64
logits, the fp64 loss) and against the regular fused-linear entry point.

The file name sorts last, so in a full run this also exercises the entry point
after every other GPU test in the same process; it passes alone as well.
"""
import numpy as np
import pytest
import torch

import oracle
from distillation_ce_tvd_gb300 import binding
from parity_util import tie_info

pytestmark = pytest.mark.gpu

DEV = "cuda"
FCT_ERR_UNSUPPORTED = 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def _case(BT, ds, dt, V, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    hs = torch.randn(BT, ds, generator=g, device=DEV).bfloat16()
    ht = torch.randn(BT, dt, generator=g, device=DEV).bfloat16()
    ws = (torch.randn(V, ds, generator=g, device=DEV) * (2.0 / ds ** 0.5)).bfloat16()
    wt = (torch.randn(V, dt, generator=g, device=DEV) * (2.0 / dt ** 0.5)).bfloat16()
    tg = torch.randint(0, V, (BT,), generator=g, device=DEV)
    tg[::7] = -100
    gce = torch.full((BT,), 1.0 / BT, device=DEV)
    gtvd = torch.full((BT,), 0.7 / BT, device=DEV)
    return hs, ws, ht, wt, tg, gce, gtvd


def _outputs(BT, V, ds):
    """Caller-owned outputs, pre-filled with NaN so that an unwritten value shows."""
    outs = [torch.full((BT,), float("nan"), device=DEV) for _ in range(5)]
    grad_h = torch.full((BT, ds), float("nan"), device=DEV, dtype=torch.bfloat16)
    grad_w = torch.zeros(V, ds, device=DEV)
    return outs, grad_h, grad_w


def _reference(case):
    """The fp64 reference of a case (library matmuls for the logits, the
    oracle for the loss) and the fused-linear tests' tolerances around it:
    per-row outputs, sigma, d hidden and d weight."""
    hs, ws, ht, wt, tg, gce, gtvd = case
    ds, dt = hs.shape[1], ht.shape[1]
    BT, V = hs.shape[0], ws.shape[0]
    Hs, Ws, Ht, Wt = (x.cpu().double().numpy() for x in (hs, ws, ht, wt))
    Ls, Lt = Hs @ Ws.T, Ht @ Wt.T
    tgc = tg.cpu().numpy()
    gce_h = np.broadcast_to(gce.cpu().numpy(), (BT,)).copy()
    gtvd_h = np.broadcast_to(gtvd.cpu().numpy(), (BT,)).copy()
    fwd = oracle.fused_ce_tvd_forward(Ls, Lt, tgc)
    G, _ = oracle.fused_ce_tvd_backward(Ls, Lt, tgc, gce_h, gtvd_h)
    _, mass, _ = tie_info(Ls, Lt)
    # logits are fp32 sums of D exact bf16 products (error <= D 2^-24 sum |h w|);
    # a per-row output moves by at most twice the largest logit error
    bound = np.maximum((np.abs(Hs) @ np.abs(Ws).T).max(1) * ds,
                       (np.abs(Ht) @ np.abs(Wt).T).max(1) * dt) * 2.0 ** -24
    row = 1e-5 + 2.0 * bound
    sigma = row + 2.0 * mass
    G_abs = np.abs(G)
    e_rel = 2.0 ** -8 + 2e-3 + V * 2.0 ** -24
    ref_gh = G @ Ws
    tol_gh = (e_rel * (G_abs @ np.abs(Ws)) + 1e-6 * np.abs(Ws).sum(0)
              + 2.0 ** -8 * np.abs(ref_gh) + 1e-9)
    e_rel_w = 2.0 ** -8 + 2e-3 + BT * 2.0 ** -24
    ref_gw = G.T @ Hs
    tol_gw = e_rel_w * (G_abs.T @ np.abs(Hs)) + 1e-6 * np.abs(Hs).sum(0) + 1e-9
    names = ("ce", "tvd", "student_lse", "teacher_lse", "sigma")
    ref = tuple(fwd[k] for k in names) + (ref_gh, ref_gw)
    return tgc, ref, (row, sigma, tol_gh, tol_gw)


def _compare(got, ref, tgc, tols, what, factor=1.0):
    """got against ref within factor x the tolerances (2 when ref is another
    GPU result: each is within them of the fp64 result).  grad_h / grad_w
    entries of None are skipped."""
    row, sigma, tol_gh, tol_gw = (factor * t for t in tols)
    ign = tgc == -100
    names = ("ce", "tvd", "student_lse", "teacher_lse", "sigma")
    as_np = lambda x: x.cpu().double().numpy() if torch.is_tensor(x) else np.asarray(x)  # noqa: E731
    for k, name in enumerate(names):
        a, b = as_np(got[k]), as_np(ref[k])
        assert np.all(a[ign] == 0.0) and np.all(b[ign] == 0.0), f"{what}{name}: ignored rows"
        tol = sigma if name == "sigma" else row
        err = np.abs(a - b)
        assert np.all(err <= tol), f"{what}{name}: worst err/tol {(err / tol).max():.3g}"
    if got[5] is not None and ref[5] is not None:
        gh_a, gh_b = as_np(got[5]), as_np(ref[5])
        assert np.all(gh_a[ign] == 0.0), f"{what}grad_h: ignored rows must be 0"
        err = np.abs(gh_a - gh_b)
        assert np.all(err <= tol_gh), f"{what}grad_h: worst err/tol {(err / tol_gh).max():.3g}"
    if got[6] is not None and ref[6] is not None:
        err = np.abs(as_np(got[6]) - as_np(ref[6]))
        assert np.all(err <= tol_gw), f"{what}grad_w: worst err/tol {(err / tol_gw).max():.3g}"


# (50, 128, 96, 1003): the rows fit in one block of the fixed scratch.
# (120, 64, 64, 151936): 64 MiB holds 55 rows of 2 x 151936 fp32 logits, so
# three blocks, the last one ragged (10 rows).
@pytest.mark.parametrize("BT,ds,dt,V", [(50, 128, 96, 1003), (120, 64, 64, 151936)])
def test_noalloc_matches_regular_entry_point(BT, ds, dt, V):
    cases = [_case(BT, ds, dt, V, seed=BT + V + k) for k in range(2)]
    bufs = [_outputs(BT, V, ds) for _ in cases]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)

    # two calls in a row; the second finds the first one's data in the scratch
    def call(case, buf):
        hs, ws, ht, wt, tg, gce, gtvd = case
        outs, grad_h, grad_w = buf
        return binding.fused_linear_ce_tvd_forward_backward_noalloc(
            hs, ws, ht, wt, tg, gce, gtvd, *outs, grad_h=grad_h, grad_w=grad_w,
            dev_status=status)

    got = [call(cases[0], bufs[0])]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    got.append(call(cases[1], bufs[1]))
    torch.cuda.synchronize()
    # set-up happened in the first call; the second allocates nothing
    assert torch.cuda.mem_get_info()[0] == free_before
    assert status.item() == 0

    for k, (case, g) in enumerate(zip(cases, got)):
        hs, ws, ht, wt, tg, gce, gtvd = case
        tgc, ref64, tols = _reference(case)
        # against the oracle (fp64 logits and loss) ...
        _compare(g, ref64, tgc, tols, what=f"call {k} vs oracle: ")
        # ... and against the regular entry point
        ref = binding.fused_linear_ce_tvd_forward_backward(hs, ws, ht, wt, tg, gce, gtvd)
        torch.cuda.synchronize()
        _compare(g, ref, tgc, tols, what=f"call {k} vs regular: ", factor=2.0)


@pytest.mark.parametrize("grads,want_h,want_w", [
    ("scalar", True, True),      # one broadcast upstream value each (grad_stride 0)
    ("rows", False, True),       # no d hidden
    ("rows", True, False),       # no d weight
    ("rows", False, False),      # the loss alone
])
def test_noalloc_optional_outputs_and_broadcast_grads(grads, want_h, want_w):
    BT, ds, dt, V = 70, 64, 96, 2051
    case = list(_case(BT, ds, dt, V, seed=77))
    if grads == "scalar":
        case[5] = torch.full((1,), 0.25, device=DEV)
        case[6] = torch.full((1,), 0.125, device=DEV)
    hs, ws, ht, wt, tg, gce, gtvd = case
    outs, grad_h, grad_w = _outputs(BT, V, ds)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.fused_linear_ce_tvd_forward_backward_noalloc(
        hs, ws, ht, wt, tg, gce, gtvd, *outs, grad_h=grad_h if want_h else None,
        grad_w=grad_w if want_w else None, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert (got[5] is None) == (not want_h) and (got[6] is None) == (not want_w)
    tgc, ref64, tols = _reference(case)
    _compare(got, ref64, tgc, tols, what=f"{grads} h={want_h} w={want_w}: ")


def test_noalloc_refuses_multi_dim_upstream_grads():
    # A (B, T) view of the per-row upstream gradient would be read in storage
    # order; the binding takes 1-D vectors only and copies nothing.
    BT, ds, V = 12, 32, 300
    hs, ws, ht, wt, tg, gce, gtvd = _case(BT, ds, ds, V, seed=5)
    outs, grad_h, grad_w = _outputs(BT, V, ds)
    g2 = torch.ones(4, 3, device=DEV).t()           # non-contiguous, 12 values
    with pytest.raises(ValueError):
        binding.fused_linear_ce_tvd_forward_backward_noalloc(hs, ws, ht, wt, tg, g2, gtvd, *outs)
    with pytest.raises(ValueError):
        binding.fused_linear_ce_tvd_forward_backward_noalloc(
            hs, ws, ht, wt, tg, gce.reshape(3, 4), gtvd, *outs)


def test_noalloc_rejects_vocab_beyond_scratch():
    # 8 * round8(V) bytes (one student + one teacher fp32 row) must fit in
    # 64 MiB: V = 8,388,609 does not.  The buffers are real and sized for V,
    # and the refusal comes before any launch, leaving the outputs untouched.
    BT, d, V = 2, 8, 8 * 1024 * 1024 + 1
    hs = torch.zeros(BT, d, device=DEV, dtype=torch.bfloat16)
    w = torch.zeros(V, d, device=DEV, dtype=torch.bfloat16)
    tg = torch.zeros(BT, dtype=torch.int64, device=DEV)
    g = torch.ones(BT, device=DEV)
    outs = [torch.full((BT,), 7.0, device=DEV) for _ in range(5)]
    with pytest.raises(binding.FctError) as e:
        binding.fused_linear_ce_tvd_forward_backward_noalloc(hs, w, hs, w, tg, g, g, *outs)
    assert e.value.status == FCT_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert all(bool((o == 7.0).all()) for o in outs)


def test_noalloc_takes_unaligned_layouts_the_regular_entry_refuses():
    # Hidden size 100 (rows of 200 bytes): not a TMA layout, so the regular
    # entry point refuses it with FCT_ERR_ALIGNMENT and this one runs its
    # CUDA-core GEMMs; the results still meet the oracle's tolerances.
    BT, ds, dt, V = 40, 100, 60, 1003
    case = _case(BT, ds, dt, V, seed=91)
    hs, ws, ht, wt, tg, gce, gtvd = case
    outs, grad_h, grad_w = _outputs(BT, V, ds)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.fused_linear_ce_tvd_forward_backward_noalloc(
        hs, ws, ht, wt, tg, gce, gtvd, *outs, grad_h=grad_h, grad_w=grad_w, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    tgc, ref64, tols = _reference(case)
    _compare(got, ref64, tgc, tols, what="unaligned: ")
    with pytest.raises(binding.FctError) as e:
        binding.fused_linear_ce_tvd_forward_backward(hs, ws, ht, wt, tg, gce, gtvd)
    assert e.value.status == 3  # FCT_ERR_ALIGNMENT
