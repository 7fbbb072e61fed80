"""Outputs past 2^31 elements.

The plain GEMM, the unfused in-place RoPE and the fused RoPE GEMM write a
[65568, 33024] bf16 output (2.17e9 elements, 4.3 GB), ragged in both
dimensions (M is 32 rows past a 256-row tile, N 256 columns past a 512-column
block). Sampled rows, among them
rows whose flat offsets lie past 2^31, are checked against the float64 oracle
(positions = row mod S for RoPE, so the tables wrap 16 times). This guards
every offset on the path (TMA coordinates, tile and item counters, the
epilogue's row index) against 32-bit overflow. K is small to keep the
contraction short: the test is about addressing, not throughput."""
import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, dev_bf16, f64

pytestmark = pytest.mark.gpu


def test_output_past_2_31_elements(coda):
    import torch
    M, K, N, hd, rc, S = 65568, 64, 33024, 128, 32768, 4096
    assert M * N > 2 ** 31
    p = gen.rope_problem(M, K, N, seed=7, with_bwd=False)
    X, W = dev_bf16(p["X"]), dev_bf16(p["W"])
    first_past = (2 ** 31) // N  # first row with elements past 2^31
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 1, S - 1, S, first_past, first_past + 1, M - 33, M - 32, M - 1],
                                     rng.choice(M, size=23, replace=False)]))
    X64, W64 = O.bf16(p["X"][rows]), O.bf16(p["W"])
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    coda.coda_gemm(X, W, out=out)
    plain = f64(out[rows])
    assert_bf16(plain, O.matmul(X64, W64), "plain GEMM rows")

    # the unfused comparison path's in-place rotation over the same buffer
    c, s = coda.coda_rope_tables(S, hd, 10000.0)
    coda.coda_unfused_rope(out, c, s, hd, rc)
    assert_bf16(f64(out[rows]), O.rope(plain, rows % S, hd, 10000.0, rc), "unfused RoPE rows")

    out.fill_(float("nan"))
    coda.coda_gemm_rope(X, W, c, s, hd, rc, out=out)
    assert_bf16(f64(out[rows]), O.gemm_rope(X64, W64, rows % S, hd, 10000.0, rc), "RoPE GEMM rows")
    # the last row and column were written (a clipped store past 2^31 would leave the NaN fill)
    assert torch.isfinite(out[-1]).all() and torch.isfinite(out[:, -1]).all()
    del out
    assert coda.coda_device_status(clear=True) == 0
