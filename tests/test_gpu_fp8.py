"""Parity of the FP8 (E4M3) mainloop variants with the float64 oracle.

The oracle decodes the exact E4M3 operand bytes (oracle.e4m3), multiplies by
the per-tensor scales and applies the same operator definitions as the bf16
kernels' oracle (matmul, rope, swiglu, ce_fwd, ce_bwd). Products of E4M3 values
are exact in fp32, so the tolerances are the bf16 ones (outputs are bf16,
statistics fp32)."""
import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, assert_stat, f64

pytestmark = pytest.mark.gpu

THETA = 10000.0


def dev_u8(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).cuda()


def _ops(M, K, N, seed, labels=False):
    p = gen.fp8_problem(M, K, N, seed=seed, labels=labels)
    a = O.e4m3(p["A"]) * p["sA"]
    b = O.e4m3(p["B"]) * p["sB"]          # [N, K]
    return p, a, b, p["sA"] * p["sB"]


@pytest.fixture(params=[1, 2], ids=["cta1", "cta2"])
def cta_group(coda, request):
    coda.coda_set_cta_group(request.param)
    yield request.param
    coda.coda_set_cta_group(0)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 520, 208), (640, 1024, 2048), (1, 264, 16), (2560, 4096, 384)])
def test_gemm_fp8(coda, cta_group, M, N, K):
    p, a, b, alpha = _ops(M, K, N, seed=M + N + K)
    C = coda.coda_gemm_fp8(dev_u8(p["A"]), dev_u8(p["B"]), alpha)
    assert_bf16(f64(C), O.matmul(a, b.T), f"fp8 gemm {M}x{N}x{K}")


def test_gemm_fp8_accepts_float8_dtype_and_k_zero(coda):
    import torch
    p, a, b, alpha = _ops(256, 512, 384, seed=3)
    A8 = dev_u8(p["A"]).view(torch.float8_e4m3fn)
    B8 = dev_u8(p["B"]).view(torch.float8_e4m3fn)
    C = coda.coda_gemm_fp8(A8, B8, alpha)
    assert_bf16(f64(C), O.matmul(a, b.T), "fp8 gemm from float8_e4m3fn tensors")
    Z = coda.coda_gemm_fp8(torch.zeros((64, 0), dtype=torch.uint8, device="cuda"),
                           torch.zeros((32, 0), dtype=torch.uint8, device="cuda"), 1.0)
    assert float(Z.float().abs().max()) == 0.0


@pytest.mark.parametrize("M,K,N,S", [(300, 208, 768, 128), (256, 512, 1536, 100)])
def test_rope_fp8(coda, cta_group, M, K, N, S):
    hd, rc = 128, 2 * N // 3
    p, a, b, alpha = _ops(M, K, N, seed=11)
    c, s = coda.coda_rope_tables(S, hd, THETA)
    out = coda.coda_gemm_rope_fp8(dev_u8(p["A"]), dev_u8(p["B"]), alpha, c, s, hd, rc)
    assert_bf16(f64(out), O.gemm_rope(a, b.T, np.arange(M) % S, hd, THETA, rc), "fp8 GEMM+RoPE")


@pytest.mark.parametrize("want_gu", [False, True])
def test_swiglu_fp8(coda, cta_group, want_gu):
    M, K, F = 300, 400, 264
    p, a, b, alpha = _ops(M, K, 2 * F, seed=12)
    A, GU = coda.coda_gemm_swiglu_fp8(dev_u8(p["A"]), dev_u8(p["B"]), alpha, want_gu=want_gu)
    ref = O.gemm_swiglu(a, b.T)
    assert_bf16(f64(A), ref["A"], "fp8 SwiGLU A")
    if want_gu:
        assert_bf16(f64(GU), ref["GU"], "fp8 SwiGLU GU")
    else:
        assert GU is None


def test_ce_fp8(coda, cta_group):
    import torch
    M, K, V = 300, 256, 1000
    p, a, b, alpha = _ops(M, K, V, seed=13, labels=True)
    y = torch.from_numpy(p["labels"]).cuda()
    H8, W8 = dev_u8(p["A"]), dev_u8(p["B"])
    pmax, psum, parg, tgt = coda.coda_gemm_ce_lse_fp8(H8, W8, alpha, y)
    lse, loss_row, loss_mean, am = coda.coda_ce_reduce(pmax, psum, parg, tgt)
    L = O.matmul(a, b.T)
    ref = O.ce_fwd(L, p["labels"])
    assert_stat(f64(lse), ref["lse"], "fp8 lse")
    assert_stat(f64(loss_row), ref["loss_row"], "fp8 loss rows")
    top2 = np.sort(L, axis=1)[:, -2:]
    sure = (top2[:, 1] - top2[:, 0]) > 1e-5 * np.sqrt(K) * np.max(np.abs(L), axis=1) + 1e-6
    assert np.array_equal(am.cpu().numpy()[sure], ref["argmax"][sure])
    dl = coda.coda_gemm_ce_bwd_fp8(H8, W8, alpha, y, lse, 1.0 / M)
    assert_bf16(f64(dl), O.ce_bwd(L, p["labels"], f64(lse), 1.0 / M), "fp8 dl")


def _rows(M, n=40, seed=0):
    r = np.random.default_rng(seed).choice(M, size=n - 2, replace=False)
    return np.unique(np.concatenate([[0, M - 1], r]))


def test_fp8_fullsize_workloads(coda):
    """The three FP8 workloads at full size (automatic tile choice), sampled rows."""
    import torch
    w = gen.WORKLOADS["fp8_rope_qkv_4096"]
    p, a, b, alpha = _ops(w["M"], w["K"], w["N"], seed=0)
    c, s = coda.coda_rope_tables(w["S"], w["head_dim"], w["theta"])
    out = coda.coda_gemm_rope_fp8(dev_u8(p["A"]), dev_u8(p["B"]), alpha, c, s, w["head_dim"], w["rope_cols"])
    rows = _rows(w["M"])
    assert_bf16(f64(out[rows]), O.gemm_rope(a[rows], b.T, rows % w["S"], w["head_dim"], THETA, w["rope_cols"]),
                "fp8 QKV rows")

    w = gen.WORKLOADS["fp8_swiglu_up_4096"]
    p, a, b, alpha = _ops(w["M"], w["K"], w["N"], seed=0)
    A, GU = coda.coda_gemm_swiglu_fp8(dev_u8(p["A"]), dev_u8(p["B"]), alpha, want_gu=True)
    rows = _rows(w["M"], seed=1)
    ref = O.gemm_swiglu(a[rows], b.T)
    assert_bf16(f64(A[rows]), ref["A"], "fp8 SwiGLU A rows")
    assert_bf16(f64(GU[rows]), ref["GU"], "fp8 SwiGLU GU rows")

    w = gen.WORKLOADS["fp8_lm_head_ce_8192"]
    p, a, b, alpha = _ops(w["M"], w["K"], w["N"], seed=0, labels=True)
    y = torch.from_numpy(p["labels"]).cuda()
    H8, W8 = dev_u8(p["A"]), dev_u8(p["B"])
    pmax, psum, parg, tgt = coda.coda_gemm_ce_lse_fp8(H8, W8, alpha, y)
    lse, loss_row, _, _ = coda.coda_ce_reduce(pmax, psum, parg, tgt)
    dl = coda.coda_gemm_ce_bwd_fp8(H8, W8, alpha, y, lse, 1.0 / w["M"])
    rows = _rows(w["M"], seed=2)
    L = O.matmul(a[rows], b.T)
    ref = O.ce_fwd(L, p["labels"][rows])
    assert_stat(f64(lse[rows]), ref["lse"], "fp8 lse rows")
    assert_stat(f64(loss_row[rows]), ref["loss_row"], "fp8 loss rows")
    assert_bf16(f64(dl[rows]), O.ce_bwd(L, p["labels"][rows], f64(lse[rows]), 1.0 / w["M"]), "fp8 dl rows")
    assert coda.coda_device_status(clear=True) == 0
