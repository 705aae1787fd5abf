"""The library's tcgen05 bf16 GEMM (the fused-linear path's four products)
through the C ABI, against fp64 products on the host.

Exactness: with operands that are small multiples of powers of two, every
partial sum is an integer multiple of the products' common unit and stays
far below 2^24 units, so an fp32 accumulator is exact in any order and the
GPU result must equal the fp64 product bit for bit.  Random normal operands
check the general case against the fp32 accumulation bound."""
import itertools

import numpy as np
import pytest
import torch

from distillation_ce_tvd_gb300 import binding

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()
    yield


def dyadic(shape, k, den, g):
    x = torch.randint(-k, k + 1, shape, generator=g, device=DEV, dtype=torch.int16)
    return x.to(torch.bfloat16).div_(den)


def round8(n: int) -> int:
    return (n + 7) // 8 * 8


def operand(x_rowmajor: torch.Tensor, mn_major: bool, pad: int = 0,
            fill=float("nan")) -> torch.Tensor:
    """The (rows, K) operand x as a K-major view (row-major, row stride
    round8(K) + pad) or an MN-major one (the transpose of a row-major
    (K, rows) tensor with row stride round8(rows) + pad); pad is a multiple
    of 8, so the strides meet the 16-byte rule.  The padding holds NaN: a
    tile load that read past the matrix instead of filling zeros would turn
    the result into NaN."""
    rows, K = x_rowmajor.shape
    if mn_major:
        base = torch.full((K, round8(rows) + pad), fill, dtype=x_rowmajor.dtype, device=DEV)
        base[:, :rows] = x_rowmajor.t()
        return base[:, :rows].t()
    base = torch.full((rows, round8(K) + pad), fill, dtype=x_rowmajor.dtype, device=DEV)
    base[:, :K] = x_rowmajor
    return base[:, :K]


SHAPES = [(128, 256, 64), (1, 8, 1), (200, 300, 100), (129, 257, 65), (300, 1003, 777),
          (64, 4096, 256)]


@pytest.mark.parametrize("a_mn,b_mn", list(itertools.product([False, True], repeat=2)))
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_exact_all_layouts(a_mn, b_mn, M, N, K):
    g = torch.Generator(device=DEV).manual_seed(M * 7 + N * 3 + K)
    a = dyadic((M, K), 3, 4.0, g)
    b = dyadic((N, K), 7, 16.0, g)
    ref = a.double().cpu() @ b.double().cpu().T
    A = operand(a, a_mn, pad=8 if a_mn else 16)
    B = operand(b, b_mn, pad=16 if b_mn else 8)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    c = binding.fct_gemm_bf16(A, B, dev_status=status)
    cb = binding.fct_gemm_bf16(A, B, out_dtype=torch.bfloat16)
    c0 = dyadic((M, N), 5, 8.0, g).float()
    cacc = binding.fct_gemm_bf16(A, B, c0.clone(), accumulate=True)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(c.cpu().double(), ref)
    assert torch.equal(cb.cpu(), ref.float().bfloat16())  # one rounding of the exact sum
    assert torch.equal(cacc.cpu().double(), ref + c0.cpu().double())


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True)])
def test_gemm_random_within_fp32_bound(a_mn, b_mn):
    M, N, K = 333, 700, 2500
    g = torch.Generator(device=DEV).manual_seed(17)
    a = torch.randn(M, K, generator=g, device=DEV).bfloat16()
    b = torch.randn(N, K, generator=g, device=DEV).bfloat16()
    c = binding.fct_gemm_bf16(operand(a, a_mn), operand(b, b_mn))
    torch.cuda.synchronize()
    A, B = a.double().cpu().numpy(), b.double().cpu().numpy()
    ref = A @ B.T
    # products of bf16 are exact in fp32; K fp32 additions each add at most
    # 2^-23 of the running magnitude (a truncating adder included), bounded
    # by sum |a||b|
    bound = K * 2.0 ** -23 * (np.abs(A) @ np.abs(B).T) + 1e-30
    err = np.abs(c.cpu().double().numpy() - ref)
    assert np.all(err <= bound), float((err / bound).max())
    # far tighter in practice than the worst case
    assert float(np.median(err / bound)) < 0.05


def test_gemm_is_deterministic_and_tile_independent():
    # a row of A gives the same bits whether it falls in the first tile or a
    # later one, and on every call
    g = torch.Generator(device=DEV).manual_seed(5)
    a = torch.randn(300, 1000, generator=g, device=DEV).bfloat16()
    b = torch.randn(600, 1000, generator=g, device=DEV).bfloat16()
    c1 = binding.fct_gemm_bf16(a, b)
    c2 = binding.fct_gemm_bf16(a, b)
    c3 = binding.fct_gemm_bf16(a[170:171], b[300:])
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
    assert torch.equal(c1[170:171, 300:], c3)


@pytest.mark.parametrize("r0,c0", [(3, 5), (8, 8)])
def test_gemm_ragged_output_leaves_neighbours_alone(r0, c0):
    # C as a view inside a larger buffer: nothing outside M x N is written.
    # At (3, 5) the view is not 16-byte aligned (per-thread stores); at
    # (8, 8) it is, and C goes out through TMA stores whose last boxes are
    # clipped at the view's edge.
    g = torch.Generator(device=DEV).manual_seed(9)
    a = dyadic((130, 72), 3, 4.0, g)
    b = dyadic((259, 72), 7, 16.0, g)
    ref64 = a.double() @ b.double().T
    for dtype in (torch.float32, torch.bfloat16):
        for accumulate in ((False, True) if dtype == torch.float32 else (False,)):
            big = torch.full((140, 272), 7.0, device=DEV, dtype=dtype)
            view = big[r0:r0 + 130, c0:c0 + 259]
            binding.fct_gemm_bf16(a, b, view, accumulate=accumulate)
            torch.cuda.synchronize()
            ref = (ref64 + (7.0 if accumulate else 0.0)).to(dtype)
            assert torch.equal(view, ref), (dtype, accumulate)
            mask = torch.ones_like(big, dtype=torch.bool)
            mask[r0:r0 + 130, c0:c0 + 259] = False
            assert torch.all(big[mask] == 7.0), (dtype, accumulate)


def test_gemm_fused_linear_shapes_sampled():
    # The fused-linear bench's three product shapes (2048-row block, hidden
    # 4096, V = 151936), exact operands, checked on sampled rows and columns.
    g = torch.Generator(device=DEV).manual_seed(23)
    R, D, V = 2048, 4096, 151936
    h = dyadic((R, D), 3, 4.0, g)
    w = dyadic((V, D), 7, 64.0, g)
    G = dyadic((R, V), 3, 256.0, g)
    rows = torch.tensor([0, 1, 127, 128, 1000, 2047])
    cols = torch.tensor([0, 255, 256, 70001, 151935])
    logits = binding.fct_gemm_bf16(h, w)                            # R x V
    dh = binding.fct_gemm_bf16(G, w.t(), out_dtype=torch.float32)   # R x D: W MN-major
    dw = binding.fct_gemm_bf16(G.t(), h.t())                        # V x D: both MN-major
    torch.cuda.synchronize()
    dcols = torch.tensor([0, 63, 64, 2049, 4095])
    vrows = torch.tensor([0, 1, 127, 128, 99999, 151935])
    rows_d, cols_d, dcols_d, vrows_d = (x.to(DEV) for x in (rows, cols, dcols, vrows))
    ref_l = h[rows_d].cpu().double() @ w[cols_d].cpu().double().T
    assert torch.equal(logits[rows_d][:, cols_d].cpu().double(), ref_l)
    # d hidden sums V = 151936 products in units of 2^-14 of at most 21
    # units each: partial sums stay below 2^24 units, so fp32 is exact
    ref_dh = G[rows_d].cpu().double() @ w[:, dcols_d].cpu().double()
    assert torch.equal(dh[rows_d][:, dcols_d].cpu().double(), ref_dh)
    ref_dw = G[:, vrows_d].cpu().double().T @ h[:, dcols_d].cpu().double()
    assert torch.equal(dw[vrows_d][:, dcols_d].cpu().double(), ref_dw)


@pytest.mark.parametrize("M,N,K", [(300, 1003, 4000), (64, 256, 8192), (513, 520, 3000)])
def test_gemm_split_k_exact_and_deterministic(M, N, K):
    # Few output tiles and a long K: with a workspace the GEMM splits K and
    # adds the parts' fp32 slabs in order.  Exact operands: every split gives
    # the exact product; random operands: repeated calls give the same bits.
    g = torch.Generator(device=DEV).manual_seed(M + N + K)
    a = dyadic((M, K), 3, 4.0, g)
    b = dyadic((N, K), 7, 16.0, g)
    ws = torch.empty(binding.fct_gemm_bf16_workspace_size(M, N), dtype=torch.uint8, device=DEV)
    ref = a.double().cpu() @ b.double().cpu().T
    big = torch.full((M + 16, N + 24), 7.0, device=DEV)
    view = big[8:8 + M, 8:8 + N]
    binding.fct_gemm_bf16(a, operand(b, True), view, workspace=ws)
    cb = binding.fct_gemm_bf16(a, b, out_dtype=torch.bfloat16, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(view.cpu().double(), ref)
    assert torch.equal(cb.cpu(), ref.float().bfloat16())
    mask = torch.ones_like(big, dtype=torch.bool)
    mask[8:8 + M, 8:8 + N] = False
    assert torch.all(big[mask] == 7.0)

    x = torch.randn(M, K, generator=g, device=DEV).bfloat16()
    y = torch.randn(N, K, generator=g, device=DEV).bfloat16()
    c1 = binding.fct_gemm_bf16(x, y, workspace=ws)
    c2 = binding.fct_gemm_bf16(x, y, workspace=ws)
    c0 = binding.fct_gemm_bf16(x, y)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
    X, Y = x.double().cpu().numpy(), y.double().cpu().numpy()
    bound = K * 2.0 ** -23 * (np.abs(X) @ np.abs(Y).T) + 1e-30
    for c in (c0, c1):
        assert np.all(np.abs(c.cpu().double().numpy() - X @ Y.T) <= bound)


def test_gemm_split_k_fused_linear_d_hidden_shape():
    # d hidden of a 2048-row block: 8 x 16 output tiles over K = 151936
    g = torch.Generator(device=DEV).manual_seed(31)
    R, D, V = 2048, 4096, 151936
    w = dyadic((V, D), 7, 64.0, g)
    G = dyadic((R, V), 3, 256.0, g)
    ws = torch.empty(binding.fct_gemm_bf16_workspace_size(R, D), dtype=torch.uint8, device=DEV)
    dh = binding.fct_gemm_bf16(G, w.t(), out_dtype=torch.bfloat16, workspace=ws)
    dh32 = binding.fct_gemm_bf16(G, w.t(), workspace=ws)
    torch.cuda.synchronize()
    rows = torch.tensor([0, 255, 256, 1999, 2047], device=DEV)
    cols = torch.tensor([0, 127, 128, 4000, 4095], device=DEV)
    ref = G[rows].cpu().double() @ w[:, cols].cpu().double()
    assert torch.equal(dh32[rows][:, cols].cpu().double(), ref)
    assert torch.equal(dh[rows][:, cols].cpu(), ref.float().bfloat16())
