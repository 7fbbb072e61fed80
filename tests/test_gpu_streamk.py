"""The stream-K split of the fused GEMMs against the float64 oracle.

Shapes here have between one and two waves of tiles (1800 rows: 112 SM-pair
tiles of 256 x 256 or 210 single-SM tiles of 128 x 256 at N = 3400), so with
the split forced on (coda_set_stream_k(2)) every tile is shared out as k-block
ranges and most tiles are accumulated in two pieces that meet through the
workspace. Ragged M, N and K. For every epilogue kind (identity, RoPE,
SwiGLU with its side output, SwiGLU backward and RMSNorm backward with their
TMA input boxes, the residual / row-statistic epilogues, cross-entropy
forward and dlogits, FP8) the test checks:
  * the outputs against the oracle on the exact tensors the kernel consumed;
  * two stream-K launches give the same bits (the sum of two fp32 pieces does
    not depend on which piece arrives second);
  * the stream-K result differs from the data-parallel schedule's somewhere
    (fp32 accumulation order), so the split really ran.
"""
import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, assert_stat, col_tile_sums, dev_bf16, f64

pytestmark = pytest.mark.gpu

EPS = 1e-6
THETA = 10000.0
M, K = 1800, 1096


@pytest.fixture(params=[0, 1], ids=["pair", "cta1"])
def cta_group(coda, request):
    coda.coda_set_cta_group(request.param)
    yield request.param
    coda.coda_set_cta_group(0)
    coda.coda_set_stream_k(1)


def _modes(coda, fn):
    """fn() under the data-parallel schedule and twice under the stream-K split;
    returns (dp, sk) as lists of float64 arrays, after checking that the two
    stream-K runs agree bit for bit."""
    import torch
    out = {}
    for mode, key in ((0, "dp"), (2, "sk"), (2, "sk2")):
        coda.coda_set_stream_k(mode)
        res = fn()
        torch.cuda.synchronize()
        out[key] = [r.clone() for r in (res if isinstance(res, (tuple, list)) else (res,)) if r is not None]
    coda.coda_set_stream_k(1)
    for a, b in zip(out["sk"], out["sk2"]):
        assert torch.equal(a, b), "two stream-K launches differ"
    assert any(not torch.equal(a, b) for a, b in zip(out["dp"], out["sk"])), \
        "stream-K and data-parallel results are bit-identical: the split did not run"
    return [f64(t) for t in out["dp"]], [f64(t) for t in out["sk"]]


def test_plain_gemm_layouts(coda, cta_group):
    N = 3400
    p = gen.rope_problem(M, K, N, seed=41, with_bwd=False)
    X, W = dev_bf16(p["X"]), dev_bf16(p["W"])
    ref = O.matmul(O.bf16(p["X"]), O.bf16(p["W"]))
    _, (C,) = _modes(coda, lambda: coda.coda_gemm(X, W))
    assert_bf16(C, ref, "C = X W (stream-K)")
    # transposed operands: X stored [K, M], W stored [N, K]
    Xt, Wt = X.t().contiguous(), W.t().contiguous()
    _, (Ct,) = _modes(coda, lambda: coda.coda_gemm(Xt, Wt, transA=True, transB=True))
    assert_bf16(Ct, ref, "C = (X^T)^T (W^T)^T (stream-K)")
    assert coda.coda_device_status(clear=True) == 0


def test_rope(coda, cta_group):
    N, hd, rc, S = 3328, 128, 2048, 1024
    p = gen.rope_problem(M, K, N, seed=42)
    c, s = coda.coda_rope_tables(S, hd, THETA)
    pos = np.arange(M) % S
    X, W, A, B = (dev_bf16(p[k]) for k in ("X", "W", "A", "B"))
    _, (out,) = _modes(coda, lambda: coda.coda_gemm_rope(X, W, c, s, hd, rc))
    assert_bf16(out, O.gemm_rope(O.bf16(p["X"]), O.bf16(p["W"]), pos, hd, THETA, rc), "rope fwd (stream-K)")
    _, (g,) = _modes(coda, lambda: coda.coda_gemm_rope_bwd(A, B, c, s, hd, rc))
    assert_bf16(g, O.gemm_rope_bwd(O.bf16(p["A"]), O.bf16(p["B"]), pos, hd, THETA, rc), "rope bwd (stream-K)")


def test_swiglu_fwd_bwd(coda, cta_group):
    F = 1696
    p = gen.swiglu_problem(M, K, F, seed=43)
    X, Wgu = dev_bf16(p["X"]), dev_bf16(p["Wgu"])
    _, (A, GU) = _modes(coda, lambda: coda.coda_gemm_swiglu(X, Wgu, want_gu=True))
    ref = O.gemm_swiglu(O.bf16(p["X"]), O.bf16(p["Wgu"]))
    assert_bf16(GU, ref["GU"], "GU side output (stream-K)")
    assert_bf16(A, ref["A"], "A (stream-K)")
    # the backward reads GU through the epilogue's TMA input ring: pieces that
    # arrive first drop the boxes issued for them (GU here is the GPU's own
    # forward side output at F2, the tensor the backward consumes)
    F2 = 3400
    q = gen.swiglu_problem(M, K, F2, seed=44)
    coda.coda_set_stream_k(0)
    _, GU2 = coda.coda_gemm_swiglu(dev_bf16(q["X"]), dev_bf16(q["Wgu"]), want_gu=True)
    coda.coda_set_stream_k(1)
    dY, Wd = dev_bf16(q["dY"]), dev_bf16(q["Wd"])
    _, (dGU,) = _modes(coda, lambda: coda.coda_gemm_swiglu_bwd(dY, Wd, GU2))
    rb = O.gemm_swiglu_bwd(O.bf16(q["dY"]), O.bf16(q["Wd"]), f64(GU2))
    assert_bf16(dGU, rb["dGU"], "dGU (stream-K)")


def test_rms_chain(coda, cta_group):
    d, N2, Kn = 3400, 3400, 1096
    p = gen.rms_chain(M, K, d, N2, seed=45, bwd_K=Kn)
    x, W0, z, g, W1 = (dev_bf16(p[k]) for k in ("x", "W0", "z", "gamma", "W1"))
    _, (h1, h2, psq) = _modes(coda, lambda: coda.coda_gemm_res_rmsprep(x, W0, z, g))
    ref = O.res_rmsprep(O.bf16(p["x"]), O.bf16(p["W0"]), O.bf16(p["z"]), O.bf16(p["gamma"]))
    assert_bf16(h1, ref["h1"], "h1 (stream-K)")
    assert_bf16(h2, ref["h2"], "h2 (stream-K)")
    assert_stat(psq, col_tile_sums(ref["h1"] ** 2), "psq (stream-K)")
    # downstream kernels on the data-parallel h1/h2 (same tensors for both schedules)
    coda.coda_set_stream_k(0)
    h1t, h2t, psqt = coda.coda_gemm_res_rmsprep(x, W0, z, g)
    coda.coda_set_stream_k(1)
    r = coda.coda_rms_reduce(psqt, d, EPS)
    _, (Y,) = _modes(coda, lambda: coda.coda_gemm_rowscale(h2t, W1, r))
    assert_bf16(Y, O.rowscale(f64(h2t), O.bf16(p["W1"]), f64(r)), "Y rowscale (stream-K)")
    Yt = coda.coda_gemm_rowscale(h2t, W1, r)
    dO, Wn = dev_bf16(p["dO"]), dev_bf16(p["Wn"])
    _, (dY, dYr, pdot) = _modes(coda, lambda: coda.coda_gemm_rowdot(dO, Wn, Yt, r))
    rd = O.gemm_rowdot(O.bf16(p["dO"]), O.bf16(p["Wn"]), f64(Yt), f64(r), N2)
    assert_bf16(dY, rd["dY"], "dY (stream-K)")
    assert_bf16(dYr, rd["dYr"], "dYr (stream-K)")
    assert_stat(pdot, col_tile_sums(rd["dY"] * f64(Yt)), "pdot (stream-K)")
    coda.coda_set_stream_k(0)
    dYt, _, pdott = coda.coda_gemm_rowdot(dO, Wn, Yt, r)
    coda.coda_set_stream_k(1)
    s = coda.coda_rowdot_reduce(pdott, N2)
    _, (dh1, pdg) = _modes(coda, lambda: coda.coda_gemm_rmsnorm_bwd(dYt, W1, h1t, g, r, s))
    rb = O.gemm_rmsnorm_bwd(f64(dYt), O.bf16(p["W1"]), f64(h1t), O.bf16(p["gamma"]), f64(r), f64(s))
    assert_bf16(dh1, rb["dh1"], "dh1 (stream-K)")
    rows = np.arange(M)
    part = f64(r)[:, None] * rb["G"] * f64(h1t)
    ref_pdg = np.stack([part[rows // 32 == b].sum(axis=0) for b in range(pdg.shape[0])])
    assert_stat(pdg, ref_pdg, "pdg column partials (stream-K)")


def test_ce(coda, cta_group):
    import torch
    V = 3400
    p = gen.ce_problem(M, K, V, seed=46)
    H, W = dev_bf16(p["H"]), dev_bf16(p["W"])
    y = torch.from_numpy(p["labels"]).cuda()
    L = O.matmul(O.bf16(p["H"]), O.bf16(p["W"]))
    ref = O.ce_fwd(L, p["labels"])
    _, (pmax, psum, parg, tgt) = _modes(coda, lambda: coda.coda_gemm_ce_lse(H, W, y))
    nb = coda.coda_num_col_tiles(V)
    tiles = [(t * 128, min(V, t * 128 + 128)) for t in range(nb)]
    assert_stat(pmax, np.stack([L[:, a:b].max(axis=1) for a, b in tiles], axis=1), "pmax (stream-K)")
    assert_stat(tgt, ref["tgt"], "target logit (stream-K)")
    coda.coda_set_stream_k(2)
    lse, loss_row, _, _ = coda.coda_ce_reduce(*coda.coda_gemm_ce_lse(H, W, y))
    assert_stat(f64(lse), ref["lse"], "lse (stream-K)")
    assert_stat(f64(loss_row), ref["loss_row"], "loss_row (stream-K)")
    coda.coda_set_stream_k(1)
    _, (dl,) = _modes(coda, lambda: coda.coda_gemm_ce_bwd(H, W, y, lse, 1.0 / M))
    assert_bf16(dl, O.ce_bwd(L, p["labels"], f64(lse), 1.0 / M), "dl (stream-K)")


def test_fp8(coda, cta_group):
    import torch
    N, K8, hd, rc, S = 3328, 2192, 128, 2048, 4096
    p = gen.fp8_problem(M, K8, N, seed=47)
    a = O.e4m3(p["A"]) * p["sA"]
    b = O.e4m3(p["B"]) * p["sB"]
    alpha = p["sA"] * p["sB"]
    A8 = torch.from_numpy(np.ascontiguousarray(p["A"], np.uint8)).cuda()
    B8 = torch.from_numpy(np.ascontiguousarray(p["B"], np.uint8)).cuda()
    _, (C,) = _modes(coda, lambda: coda.coda_gemm_fp8(A8, B8, alpha))
    assert_bf16(C, O.matmul(a, b.T), "fp8 gemm (stream-K)")
    c, s = coda.coda_rope_tables(S, hd, THETA)
    _, (R,) = _modes(coda, lambda: coda.coda_gemm_rope_fp8(A8, B8, alpha, c, s, hd, rc))
    assert_bf16(R, O.rope(O.matmul(a, b.T), np.arange(M) % S, hd, THETA, rc), "fp8 rope (stream-K)")
    assert coda.coda_device_status(clear=True) == 0


@pytest.mark.parametrize("seed", range(6))
def test_split_matches_data_parallel_on_random_shapes(coda, cta_group, seed):
    """Random ragged shapes with one to three waves of tiles and 16-80 k-blocks:
    the split changes only the fp32 accumulation order, so every bf16 output
    equals the data-parallel one or differs by one bf16 rounding step (the two
    fp32 sums of O(1) outputs agree to far better than 2^-8), and the two runs
    under the split agree bit for bit."""
    import torch
    rng = np.random.default_rng(1000 + seed)
    tile_m = 256 if cta_group == 0 else 128
    clusters = 76 if cta_group == 0 else 152
    for _ in range(4):
        M = int(rng.integers(2, 17)) * tile_m - int(rng.integers(0, 100))
        mb = -(-M // tile_m)
        nb = int(rng.integers(clusters // mb + 1, 3 * clusters // mb + 2))
        N = max(8, (nb * 256 - int(rng.integers(0, 32)) * 8))
        K = int(rng.integers(16, 81)) * 64 - int(rng.integers(0, 8)) * 8
        g = torch.Generator(device="cuda").manual_seed(seed)
        A = torch.randn(M, K, device="cuda", generator=g).bfloat16()
        B = (torch.randn(K, N, device="cuda", generator=g) * K ** -0.5).bfloat16()
        dp, sk = _modes_raw(coda, lambda: coda.coda_gemm(A, B))
        d = (sk.float() - dp.float()).abs()
        # one bf16 step of the output, with an absolute floor for outputs near zero,
        # where the fp32 sums' (K^(1/2) 2^-24-sized) difference can exceed a step
        step = (dp.float().abs() * 2.0 ** -7).clamp_min(1e-4)
        assert bool((d <= step).all()), f"{M}x{N}x{K}: split and data-parallel differ by more than one bf16 step"
    assert coda.coda_device_status(clear=True) == 0


def _modes_raw(coda, fn):
    """fn() without the split and with it (twice, checked equal); raw tensors."""
    import torch
    coda.coda_set_stream_k(0)
    dp = fn().clone()
    coda.coda_set_stream_k(2)
    sk = fn().clone()
    sk2 = fn().clone()
    coda.coda_set_stream_k(1)
    torch.cuda.synchronize()
    assert torch.equal(sk, sk2), "two stream-K launches differ"
    return dp, sk


@pytest.mark.parametrize("K", [1024, 1032], ids=["kb16", "kb17_ragged"])
@pytest.mark.parametrize("cg,M,N", [
    (0, 1790, 2808),     # SM pairs: 7 x 11 = 77 tiles, one past a wave (rem 1, every tile split)
    (0, 200, 38656),     # 1 x 151 = 151 tiles, rem 75 (one short of two waves)
    (0, 768, 32504),     # 3 x 127 = 381 tiles, five waves + 1
    (1, 1150, 4352),     # single SMs: 9 x 17 = 153 tiles, rem 1
    (1, 384, 25856),     # 3 x 101 = 303 tiles, rem 151
], ids=["pair_rem1", "pair_rem75", "pair_5waves_rem1", "cta1_rem1", "cta1_rem151"])
def test_split_at_wave_boundaries(coda, cg, M, N, K):
    """The split's edge cases on a GB300 with 76 SM pairs / 152 SMs: one tile
    past a wave, one tile short of two waves, five whole waves before the
    split, and the shortest reduction the split takes (16 k-blocks) with and
    without a ragged last k-block. Against the data-parallel schedule within one
    bf16 step, and repeatable."""
    import torch
    try:
        coda.coda_set_cta_group(cg)
        g = torch.Generator(device="cuda").manual_seed(M + N + K)
        A = torch.randn(M, K, device="cuda", generator=g).bfloat16()
        B = (torch.randn(K, N, device="cuda", generator=g) * K ** -0.5).bfloat16()
        dp, sk = _modes_raw(coda, lambda: coda.coda_gemm(A, B))
    finally:
        coda.coda_set_cta_group(0)
    d = (sk.float() - dp.float()).abs()
    step = (dp.float().abs() * 2.0 ** -7).clamp_min(1e-4)
    assert bool((d <= step).all()), f"{M}x{N}x{K}: split and data-parallel differ by more than one bf16 step"
    assert not torch.equal(sk, dp), "the split did not run"
    assert coda.coda_device_status(clear=True) == 0


def test_workspace_follows_stream_handles(coda):
    """Streams created and destroyed one after another (through the driver API):
    each one's first split launch finds or creates the stream's workspace. A
    destroyed stream's handle may come back for a new stream; the library then
    waits for the old stream's launches before reusing the workspace. Every
    launch must give the bits of the same split launch on torch's stream."""
    import ctypes
    import torch
    cu = ctypes.CDLL("libcuda.so.1")
    g = torch.Generator(device="cuda").manual_seed(3)
    A = torch.randn(1800, 1096, device="cuda", generator=g).bfloat16()
    B = (torch.randn(1096, 3400, device="cuda", generator=g) * 1096 ** -0.5).bfloat16()
    try:
        coda.coda_set_stream_k(2)
        ref = coda.coda_gemm(A, B).clone()
        torch.cuda.synchronize()
        for _ in range(4):
            h = ctypes.c_void_p()
            assert cu.cuStreamCreate(ctypes.byref(h), 1) == 0  # CU_STREAM_NON_BLOCKING
            s = torch.cuda.ExternalStream(h.value)
            outs = [coda.coda_gemm(A, B, stream=s) for _ in range(2)]
            s.synchronize()
            for o in outs:
                assert torch.equal(o, ref)
            assert cu.cuStreamDestroy_v2(h) == 0
    finally:
        coda.coda_set_stream_k(1)
    assert coda.coda_device_status(clear=True) == 0



@pytest.mark.parametrize("M,N,K", [
    (2048, 2552, 16376),   # 8 x 10 = 80 tiles, rem 4: every range is a tail piece and a head piece
    (2048, 4344, 16376),   # 8 x 17 = 136 tiles, rem 60: ranges of 1.8 tiles (tail, whole tile, head)
], ids=["rem4", "rem60"])
def test_split_rotated_walk(coda, M, N, K):
    """Long reductions whose split tiles' operands exceed half of L2 (eight row
    blocks and ten or more column blocks of 256 over K = 16376: 151-210 MB), so each
    cluster walks its range from its first tile boundary and takes the piece
    before it last, as the long-K dX GEMM does; B is K-major as there. Against
    the data-parallel schedule within one bf16 step, repeatable, and sampled
    rows and columns against the float64 oracle."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(N + K)
    A = torch.randn(M, K, device="cuda", generator=g).bfloat16()
    B = (torch.randn(N, K, device="cuda", generator=g) * K ** -0.5).bfloat16()
    dp, sk = _modes_raw(coda, lambda: coda.coda_gemm(A, B, transB=True))
    d = (sk.float() - dp.float()).abs()
    step = (dp.float().abs() * 2.0 ** -7).clamp_min(1e-4)
    assert bool((d <= step).all()), f"{M}x{N}x{K}: split and data-parallel differ by more than one bf16 step"
    assert not torch.equal(sk, dp), "the split did not run"
    rng = np.random.default_rng(N)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, 30, replace=False)]))
    cols = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 30, replace=False)]))
    ref = O.matmul(f64(A[rows]), f64(B[cols]).T)
    assert_bf16(f64(sk[rows][:, cols]), ref, "split GEMM, sampled rows and columns")
    assert coda.coda_device_status(clear=True) == 0
