"""Parity of the plain tcgen05 GEMM (identity epilogue) with the float64 oracle,
all four operand layouts, shapes spanning several tiles with ragged tails."""
import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, dev_bf16, f64

pytestmark = pytest.mark.gpu

SHAPES = [
    (128, 256, 64),     # one tile, one k-block
    (256, 512, 512),    # 2 x 2 tiles, 8 k-blocks
    (300, 520, 200),    # ragged M, N, K
    (64, 8, 8),         # smaller than one tile in every dimension
    (1, 264, 136),      # single row
    (640, 1024, 2048),  # 5 x 4 tiles, 32 k-blocks
    (2560, 4096, 128),  # 320 tiles: two or three tiles per persistent CTA
    (4096, 3072, 264),  # 384 tiles, ragged K
    (200, 264, 72),     # transposed operands with M, N not multiples of 64 (one 2-D box per 64 columns)
]


def _operands(M, N, K, ta, tb, seed):
    rngs = [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(2)]
    A = gen.normal_bf16(rngs[0], (K, M) if ta else (M, K))
    B = gen.normal_bf16(rngs[1], (N, K) if tb else (K, N), std=1.0 / np.sqrt(max(K, 1)))
    return A, B


@pytest.fixture(params=[1, 2], ids=["cta1", "cta2"])
def cta_group(coda, request):
    """Run the test with the single-SM (128 x 256) and the SM-pair (256 x 256)
    tile variant."""
    coda.coda_set_cta_group(request.param)
    yield request.param
    coda.coda_set_cta_group(0)


@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_parity(coda, cta_group, M, N, K, ta, tb):
    if ta and M % 8:
        pytest.skip("transposed A needs M % 8 == 0 (16-byte rows)")
    A, B = _operands(M, N, K, ta, tb, seed=M * 7 + N * 3 + K + ta * 2 + tb)
    C = coda.coda_gemm(dev_bf16(A), dev_bf16(B), transA=bool(ta), transB=bool(tb))
    a = O.bf16(A).T if ta else O.bf16(A)
    b = O.bf16(B).T if tb else O.bf16(B)
    assert_bf16(f64(C), O.matmul(a, b), f"gemm {M}x{N}x{K} ta={ta} tb={tb}")


def test_gemm_k_zero_and_empty(coda, cta_group):
    import torch
    A = torch.zeros((16, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((0, 24), dtype=torch.bfloat16, device="cuda")
    C = torch.full((16, 24), 7.0, dtype=torch.bfloat16, device="cuda")
    coda.coda_gemm(A, B, out=C)
    assert float(C.float().abs().max()) == 0.0
    E = coda.coda_gemm(torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"),
                       torch.zeros((64, 16), dtype=torch.bfloat16, device="cuda"))
    assert E.shape == (0, 16)


def test_gemm_leading_dims(coda, cta_group):
    """Row strides larger than the logical width (views into wider buffers)."""
    M, N, K = 200, 136, 72
    A, B = _operands(M, N + 24, K + 40, 0, 0, seed=5)
    dA, dB = dev_bf16(A), dev_bf16(B)
    import torch
    out = torch.zeros((M, N + 56), dtype=torch.bfloat16, device="cuda")
    coda.coda_gemm(dA[:, :K], dB[:K, :N], out=out[:, :N])
    assert_bf16(f64(out[:, :N]), O.matmul(O.bf16(A)[:, :K], O.bf16(B)[:K, :N]), "gemm strided")
    assert float(out[:, N:].float().abs().max()) == 0.0, "wrote past the logical columns"


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 0), (1, 1)])
def test_gemm_leading_dimensions(coda, cta_group, ta, tb):
    """Operands that are column slices of wider arrays (lda, ldb above the row
    length), for the 3-D (multiple of 64) and the 2-D operand maps."""
    M, N, K = 384, 320, 200
    A, B = _operands(M, N, K, ta, tb, seed=11 + ta + 2 * tb)
    pad = 72
    Aw = np.zeros((A.shape[0], A.shape[1] + pad), np.uint16)
    Aw[:, :A.shape[1]] = A
    Bw = np.zeros((B.shape[0], B.shape[1] + pad), np.uint16)
    Bw[:, :B.shape[1]] = B
    dA = dev_bf16(Aw)[:, :A.shape[1]]
    dB = dev_bf16(Bw)[:, :B.shape[1]]
    assert dA.stride(0) == A.shape[1] + pad
    C = coda.coda_gemm(dA, dB, transA=bool(ta), transB=bool(tb))
    a = O.bf16(A).T if ta else O.bf16(A)
    b = O.bf16(B).T if tb else O.bf16(B)
    assert_bf16(f64(C), O.matmul(a, b), f"strided gemm ta={ta} tb={tb}")


def test_gemm_random_shapes(coda):
    """Seeded sweep: random sizes (multiples of 8; some multiples of 64, which
    take the 3-D operand boxes), random operand layouts, all three tile variants."""
    R = np.random.default_rng(2024)
    for i in range(24):
        M = int(R.integers(1, 96)) * 8
        N = int(R.integers(1, 96)) * 8
        K = int(R.integers(1, 64)) * 8
        if i % 3 == 0:
            M, N = 64 * max(1, M // 64), 64 * max(1, N // 64)
        ta, tb, cg = int(R.integers(0, 2)), int(R.integers(0, 2)), (1, 2)[int(R.integers(0, 2))]
        A, B = _operands(M, N, K, ta, tb, seed=1000 + i)
        try:
            coda.coda_set_cta_group(cg)
            C = coda.coda_gemm(dev_bf16(A), dev_bf16(B), transA=bool(ta), transB=bool(tb))
        finally:
            coda.coda_set_cta_group(0)
        a = O.bf16(A).T if ta else O.bf16(A)
        b = O.bf16(B).T if tb else O.bf16(B)
        assert_bf16(f64(C), O.matmul(a, b), f"random gemm {M}x{N}x{K} ta={ta} tb={tb} cta{cg}")
