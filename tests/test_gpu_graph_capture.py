"""The entry points inside a CUDA graph: a captured step, replayed on new
inputs copied into the captured buffers, gives bitwise the eager results.

The calls are stream-ordered, allocate nothing when their outputs are passed
in and never synchronise the host, so a training step that includes them can
be captured whole.  The per-device set-up (kernel attributes, occupancy) is
done by an eager call before the capture.
"""
import pytest
import torch

from distillation_ce_tvd_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def _single(s, t, tg, gce, gtvd, outs):
    ce, tvd, ls, lt, sg, grad, status = outs
    binding.fused_ce_tvd_forward_backward(s, t, tg, gce, gtvd, ce=ce, tvd=tvd, student_lse=ls,
                                          teacher_lse=lt, sigma=sg, grad_student=grad,
                                          dev_status=status)
    return ce, tvd, ls, lt, sg, grad


def _signs_pair(s, t, tg, gce, gtvd, outs):
    ce, tvd, ls, lt, sg, grad, status, signs = outs
    binding.fused_ce_tvd_forward_signs(s, t, tg, ce=ce, tvd=tvd, student_lse=ls, teacher_lse=lt,
                                       sigma=sg, signs=signs, dev_status=status)
    binding.fused_ce_tvd_backward_signs(s, t, tg, ls, lt, sg, signs, gce, gtvd, grad_student=grad,
                                        dev_status=status)
    return ce, tvd, ls, lt, sg, grad


def _ce_single(s, t, tg, gce, gtvd, outs):
    ce, lse, grad, status = outs
    binding.ce_forward_backward(s, tg, gce, ce=ce, lse=lse, grad_logits=grad, dev_status=status)
    return ce, lse, grad


def _buffers(path, BT, V, s):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    vec = [torch.empty(BT, device=DEV) for _ in range(5)]
    grad = torch.empty_like(s)
    if path == "single":
        return (*vec, grad, status)
    if path == "signs_pair":
        nb = binding.fused_ce_tvd_signs_row_bytes(V, s.dtype)
        signs = torch.empty(BT, nb, device=DEV, dtype=torch.uint8)
        return (*vec, grad, status, signs)
    return (vec[0], vec[1], grad, status)


PATHS = {"single": _single, "signs_pair": _signs_pair, "ce_single": _ce_single}


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("V", [151936, 3001])
def test_captured_step_replays_bitwise(path, V):
    # 300 rows: more than one per SM, so the persistent grid loops over rows;
    # V = 3001 (rows not 16-byte aligned) takes the scalar path and, for sign
    # words, the flag-setting memset.
    BT = 300
    fn = PATHS[path]
    cases = [workloads.make("bt8192_v151936_bf16", DEV, rows=BT, V=V, seed=61 + k)
             for k in range(2)]
    a = cases[0]
    s, t, tg = a.student.clone(), a.teacher.clone(), a.target.clone()
    gce, gtvd = a.grad_ce.clone(), a.grad_tvd.clone()
    outs = _buffers(path, BT, V, s)
    status = outs[-2] if path == "signs_pair" else outs[-1]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn(s, t, tg, gce, gtvd, outs)  # eager: per-device set-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        results = fn(s, t, tg, gce, gtvd, outs)

    for w in (cases[1], cases[0], cases[1]):
        for dst, src in ((s, w.student), (t, w.teacher), (tg, w.target), (gce, w.grad_ce),
                         (gtvd, w.grad_tvd)):
            dst.copy_(src)
        graph.replay()
        eager = fn(w.student, w.teacher, w.target, w.grad_ce, w.grad_tvd,
                   _buffers(path, BT, V, w.student))
        torch.cuda.synchronize()
        for k, (x, y) in enumerate(zip(results, eager)):
            assert torch.equal(x, y), f"{path} output {k}"
    assert status.item() == 0


@pytest.mark.parametrize("logits_dtype", [torch.bfloat16, torch.float32])
def test_captured_fused_linear_step_replays_bitwise(logits_dtype):
    # The fused-linear entry point: cluster launches of the tensor-core GEMM
    # with tensor maps built at capture time, the loss started from the
    # GEMM's log-sum-exp partials, d hidden's K split and d weight's
    # accumulation (zeroed inside the graph), over 3 row blocks (the last
    # one ragged).
    BT, D, V, chunk = 300, 128, 3000, 128
    g = torch.Generator(device=DEV).manual_seed(71)

    def case():
        hs = torch.randn(BT, D, generator=g, device=DEV).bfloat16()
        ht = torch.randn(BT, D, generator=g, device=DEV).bfloat16()
        ws = (torch.randn(V, D, generator=g, device=DEV) * 0.2).bfloat16()
        wt = (torch.randn(V, D, generator=g, device=DEV) * 0.2).bfloat16()
        tg = torch.randint(0, V, (BT,), generator=g, device=DEV)
        tg[::9] = -100
        gce = torch.full((BT,), 1.0 / BT, device=DEV)
        return [hs, ws, ht, wt, tg, gce, gce * 0.5]

    def buffers():
        ws_bytes = binding.fused_linear_ce_tvd_workspace_size(V, chunk, logits_dtype)
        return (torch.empty(BT, D, device=DEV, dtype=torch.bfloat16),
                torch.zeros(V, D, device=DEV),
                torch.empty(ws_bytes, device=DEV, dtype=torch.uint8),
                torch.zeros(1, dtype=torch.int32, device=DEV))

    def step_all(inp, bufs):
        gh, gw, work, status = bufs
        gw.zero_()
        # (the per-row outputs come from the caching allocator: inside the
        # capture, from the graph's own pool)
        return binding.fused_linear_ce_tvd_forward_backward(
            *inp, chunk_rows=chunk, logits_dtype=logits_dtype, workspace=work, grad_h=gh,
            grad_w=gw, dev_status=status)

    cases = [case() for _ in range(2)]
    inp = [x.clone() for x in cases[0]]
    bufs = buffers()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step_all(inp, bufs)  # eager: per-device set-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        results = step_all(inp, bufs)

    for c in (cases[1], cases[0], cases[1]):
        for dst, src in zip(inp, c):
            dst.copy_(src)
        graph.replay()
        eager = step_all(c, buffers())
        torch.cuda.synchronize()
        for k, (x, y) in enumerate(zip(results, eager)):
            assert torch.equal(x, y), f"output {k}"
    assert bufs[-1].item() == 0
