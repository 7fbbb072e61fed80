"""Parity of every fused GEMM-epilogue kernel and auxiliary reduction with the
float64 oracle, on seeded inputs at sizes the oracle finishes in seconds that
span several 128 x 256 tiles with ragged tails in M, N and K.

Each kernel is compared with the oracle evaluated on exactly the bf16/fp32
tensors that kernel consumed (a chained input such as h2 or GU is the GPU's
own stored output). Chains are additionally compared end to end with the pure
float64 chain at the bf16 tolerances.
"""
import math

import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, assert_stat, col_tile_sums, dev_bf16, f64

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _dev_f32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


# ---------------------------------------------------------------- RMSNorm chain

@pytest.fixture(params=[0, 1], ids=["auto", "cta1"])
def cta_group(coda, request):
    """Automatic tile choice (SM pairs once M > 128) and forced single-SM tiles."""
    coda.coda_set_cta_group(request.param)
    yield request.param
    coda.coda_set_cta_group(0)


@pytest.mark.parametrize("M,K,d,N2", [(256, 512, 512, 512), (300, 200, 520, 264), (1, 64, 8, 8)])
def test_rms_chain_forward(coda, cta_group, M, K, d, N2):
    p = gen.rms_chain(M, K, d, N2, seed=0)
    x, W0, z, g, W1 = (p[k] for k in ("x", "W0", "z", "gamma", "W1"))
    h1, h2, psq = coda.coda_gemm_res_rmsprep(dev_bf16(x), dev_bf16(W0), dev_bf16(z), dev_bf16(g))
    ref = O.res_rmsprep(O.bf16(x), O.bf16(W0), O.bf16(z), O.bf16(g))
    assert_bf16(f64(h1), ref["h1"], "h1")
    assert_bf16(f64(h2), ref["h2"], "h2")
    assert psq.shape == (M, coda.coda_num_col_tiles(d))
    assert_stat(f64(psq), col_tile_sums(ref["h1"] ** 2), "psq tile partials")

    r = coda.coda_rms_reduce(psq, d, EPS)
    assert_stat(f64(r), O.rms_reduce(f64(psq), d, EPS), "r from the GPU partials")
    Y = coda.coda_gemm_rowscale(h2, dev_bf16(W1), r)
    assert_bf16(f64(Y), O.rowscale(f64(h2), O.bf16(W1), f64(r)), "Y (rowscale on its own inputs)")

    chain = O.gemm_rms_gemm_fwd(O.bf16(x), O.bf16(W0), O.bf16(z), O.bf16(g), O.bf16(W1), EPS)
    assert_stat(f64(r), chain["r"], "r vs the float64 chain")
    assert_bf16(f64(Y), chain["Y"], "Y vs the float64 chain")


def test_rms_chain_k_zero(coda):
    """Empty contraction: h1 = z exactly (zero accumulator), the epilogue still runs."""
    import torch
    M, d = 130, 264
    p = gen.rms_chain(M, 8, d, 8, seed=3)
    x = torch.zeros((M, 0), dtype=torch.bfloat16, device="cuda")
    W0 = torch.zeros((0, d), dtype=torch.bfloat16, device="cuda")
    h1, h2, psq = coda.coda_gemm_res_rmsprep(x, W0, dev_bf16(p["z"]), dev_bf16(p["gamma"]))
    assert np.array_equal(f64(h1), O.bf16(p["z"]))
    assert_stat(f64(psq).sum(axis=1), np.sum(O.bf16(p["z"]) ** 2, axis=1), "psq K=0")


def test_rms_chain_backward(coda, cta_group):
    M, K, d, N2, Kn = 300, 200, 264, 520, 136
    p = gen.rms_chain(M, K, d, N2, seed=1, bwd_K=Kn)
    x, W0, z, g, W1 = (p[k] for k in ("x", "W0", "z", "gamma", "W1"))
    h1, h2, psq = coda.coda_gemm_res_rmsprep(dev_bf16(x), dev_bf16(W0), dev_bf16(z), dev_bf16(g))
    r = coda.coda_rms_reduce(psq, d, EPS)
    Y = coda.coda_gemm_rowscale(h2, dev_bf16(W1), r)

    # the GEMM producing dY carries the row statistic (and dYr = r dY)
    dY, dYr, pdot = coda.coda_gemm_rowdot(dev_bf16(p["dO"]), dev_bf16(p["Wn"]), Y, r)
    ref = O.gemm_rowdot(O.bf16(p["dO"]), O.bf16(p["Wn"]), f64(Y), f64(r), d)
    assert_bf16(f64(dY), ref["dY"], "dY")
    assert_bf16(f64(dYr), ref["dYr"], "dYr")
    assert_stat(f64(pdot), col_tile_sums(ref["dY"] * f64(Y)), "pdot tile partials")
    s = coda.coda_rowdot_reduce(pdot, d)
    assert_stat(f64(s), ref["s"], "s")

    # RMSNorm backward in the data-gradient GEMM of the second projection
    # (the forward weight W1 is [d, N2]; G = dY W1^T)
    dh1, pdg = coda.coda_gemm_rmsnorm_bwd(dY, dev_bf16(W1), h1, dev_bf16(g), r, s)
    rb = O.gemm_rmsnorm_bwd(f64(dY), O.bf16(W1), f64(h1), O.bf16(g), f64(r), f64(s))
    assert_bf16(f64(dh1), rb["dh1"], "dh1")
    assert pdg.shape == (coda.coda_num_row_tiles(M), d)
    rows = np.arange(M)
    part = f64(r)[:, None] * rb["G"] * f64(h1)
    ref_pdg = np.stack([part[rows // 32 == b].sum(axis=0) for b in range(pdg.shape[0])])
    assert_stat(f64(pdg), ref_pdg, "pdg column partials", tol=1e-4)
    dg = coda.coda_colsum_reduce(pdg)
    assert_stat(f64(dg), rb["dgamma"], "dgamma")

    # end to end against the float64 chain gradient for upstream dY (the GPU's dY)
    full = O.gemm_rms_gemm_bwd(O.bf16(x), O.bf16(W0), O.bf16(z), O.bf16(g), O.bf16(W1), EPS, f64(dY))
    assert_bf16(f64(dh1), full["dh1"], "dh1 vs the float64 chain")
    # dgamma is a 300-row reduction over bf16-rounded h1 and dY: against the
    # unrounded float64 chain only a norm bound at the bf16 level applies
    # (the 1e-4 gate above is on the exact inputs the kernel consumed)
    rel = np.linalg.norm(f64(dg) - full["dgamma"]) / np.linalg.norm(full["dgamma"])
    assert rel <= 5e-3, f"dgamma vs the float64 chain: relative norm error {rel:.3e}"
    # the remaining gradients are plain GEMMs
    dW1 = coda.coda_gemm(h2, dYr, transA=True)
    assert_bf16(f64(dW1), O.matmul(f64(h2).T, f64(dYr)), "dW1 = h2^T dYr")
    dx = coda.coda_gemm(dh1, dev_bf16(W0), transB=True)
    assert_bf16(f64(dx), O.matmul(f64(dh1), O.bf16(W0).T), "dx = dh1 W0^T")
    dW0 = coda.coda_gemm(dev_bf16(x), dh1, transA=True)
    assert_bf16(f64(dW0), O.matmul(O.bf16(x).T, f64(dh1)), "dW0 = x^T dh1")


def test_rowdot_without_dyr(coda):
    M, N, K = 200, 264, 72
    p = gen.rms_chain(M, K, 8, N, seed=4, bwd_K=K)
    Y = dev_bf16(gen.rms_chain(M, 8, N, 8, seed=5)["z"])
    dY, dYr, pdot = coda.coda_gemm_rowdot(dev_bf16(p["dO"]), dev_bf16(p["Wn"]), Y, None, want_dyr=False)
    assert dYr is None
    ref = O.gemm_rowdot(O.bf16(p["dO"]), O.bf16(p["Wn"]), f64(Y), np.ones(M), N)
    assert_bf16(f64(dY), ref["dY"], "dY")
    assert_stat(f64(coda.coda_rowdot_reduce(pdot, N)), ref["s"], "s")


# ---------------------------------------------------------------- SwiGLU

@pytest.mark.parametrize("M,K,F", [(300, 200, 264), (256, 512, 512), (5, 64, 8)])
def test_swiglu_fwd_bwd(coda, M, K, F):
    p = gen.swiglu_problem(M, K, F, seed=2)
    A, GU = coda.coda_gemm_swiglu(dev_bf16(p["X"]), dev_bf16(p["Wgu"]), want_gu=True)
    ref = O.gemm_swiglu(O.bf16(p["X"]), O.bf16(p["Wgu"]))
    assert_bf16(f64(GU), ref["GU"], "GU side output")
    assert_bf16(f64(A), ref["A"], "A = silu(G) U")
    A2, none = coda.coda_gemm_swiglu(dev_bf16(p["X"]), dev_bf16(p["Wgu"]))
    assert none is None and np.array_equal(f64(A2), f64(A))

    dGU = coda.coda_gemm_swiglu_bwd(dev_bf16(p["dY"]), dev_bf16(p["Wd"]), GU)
    rb = O.gemm_swiglu_bwd(O.bf16(p["dY"]), O.bf16(p["Wd"]), f64(GU))
    assert_bf16(f64(dGU), rb["dGU"], "dGU")
    dX = coda.coda_gemm(dGU, dev_bf16(p["Wgu"]), transB=True)
    assert_bf16(f64(dX), O.matmul(f64(dGU), O.bf16(p["Wgu"]).T), "dX = dGU Wgu^T")
    dW = coda.coda_gemm(dev_bf16(p["X"]), dGU, transA=True)
    assert_bf16(f64(dW), O.matmul(O.bf16(p["X"]).T, f64(dGU)), "dWgu = X^T dGU")


# ---------------------------------------------------------------- RoPE

@pytest.mark.parametrize("M,K,N,hd,rope_cols,S", [
    (300, 200, 768, 128, 512, 256),   # positions wrap (row mod S), V columns pass through
    (256, 512, 1536, 128, 1024, 4096),
    (130, 72, 320, 64, 256, 100),     # S % 32 != 0: every row loads its own table values
    (192, 96, 576, 96, 384, 96),      # 12 table granules per row (swizzled shared copy)
    (160, 64, 256, 32, 128, 64),      # the smallest head
    (200, 128, 1024, 256, 512, 512),  # head_dim > 128: rows load their own values
])
def test_rope_fwd_bwd(coda, M, K, N, hd, rope_cols, S):
    theta = 10000.0
    c, s = coda.coda_rope_tables(S, hd, theta)
    ang = O.rope_angles(np.arange(S), hd, theta)
    assert np.max(np.abs(f64(c) - np.cos(ang))) < 1e-6
    assert np.max(np.abs(f64(s) - np.sin(ang))) < 1e-6
    p = gen.rope_problem(M, K, N, seed=3)
    pos = np.arange(M) % S
    out = coda.coda_gemm_rope(dev_bf16(p["X"]), dev_bf16(p["W"]), c, s, hd, rope_cols)
    assert_bf16(f64(out), O.gemm_rope(O.bf16(p["X"]), O.bf16(p["W"]), pos, hd, theta, rope_cols), "rope fwd")
    g = coda.coda_gemm_rope_bwd(dev_bf16(p["A"]), dev_bf16(p["B"]), c, s, hd, rope_cols)
    assert_bf16(f64(g), O.gemm_rope_bwd(O.bf16(p["A"]), O.bf16(p["B"]), pos, hd, theta, rope_cols), "rope bwd")
    # the pass-through (V) columns are the plain GEMM bit for bit
    plain = coda.coda_gemm(dev_bf16(p["X"]), dev_bf16(p["W"]))
    assert np.array_equal(f64(out)[:, rope_cols:], f64(plain)[:, rope_cols:])


# ---------------------------------------------------------------- cross-entropy

@pytest.mark.parametrize("M,K,V", [(300, 200, 1000), (256, 512, 2048), (3, 64, 8)])
def test_ce_fwd_bwd(coda, M, K, V):
    import torch
    p = gen.ce_problem(M, K, V, seed=4)
    H, W = dev_bf16(p["H"]), dev_bf16(p["W"])
    y = torch.from_numpy(p["labels"]).cuda()
    pmax, psum, parg, tgt = coda.coda_gemm_ce_lse(H, W, y)
    L = O.matmul(O.bf16(p["H"]), O.bf16(p["W"]))
    ref = O.ce_fwd(L, p["labels"])
    nb = coda.coda_num_col_tiles(V)
    tiles = [(t * 128, min(V, t * 128 + 128)) for t in range(nb)]
    ref_pmax = np.stack([L[:, a:b].max(axis=1) for a, b in tiles], axis=1)
    assert_stat(f64(pmax), ref_pmax, "pmax")
    ref_psum = np.stack([np.exp(L[:, a:b] - f64(pmax)[:, [t]]).sum(axis=1) for t, (a, b) in enumerate(tiles)], axis=1)
    assert_stat(f64(psum), ref_psum, "psum (relative to the GPU's own tile max)")
    assert_stat(f64(tgt), ref["tgt"], "target logit")
    lse, loss_row, loss_mean, argmax = coda.coda_ce_reduce(pmax, psum, parg, tgt)
    assert_stat(f64(lse), ref["lse"], "lse")
    assert_stat(f64(loss_row), ref["loss_row"], "loss_row")
    assert abs(float(loss_mean.item()) - ref["loss_mean"]) <= 1e-4 * abs(ref["loss_mean"])
    # argmax: exact wherever the top-2 gap exceeds the fp32 accumulation bound
    top2 = np.sort(L, axis=1)[:, -2:] if V > 1 else np.concatenate([L, L], axis=1)
    gap = top2[:, 1] - top2[:, 0]
    bound = 1e-5 * np.sqrt(K) * np.max(np.abs(L), axis=1) + 1e-6
    sure = gap > bound
    am = argmax.cpu().numpy()
    assert np.array_equal(am[sure], ref["argmax"][sure])
    assert np.all(np.abs(L[np.arange(M), am] - L.max(axis=1)) <= bound)

    g = 1.0 / M
    dl = coda.coda_gemm_ce_bwd(H, W, y, lse, g)
    assert_bf16(f64(dl), O.ce_bwd(L, p["labels"], f64(lse), g), "dl")
    dH = coda.coda_gemm(dl, W, transB=True)
    dW = coda.coda_gemm(H, dl, transA=True)
    full = O.gemm_ce_bwd(O.bf16(p["H"]), O.bf16(p["W"]), p["labels"], ref["lse"], g)
    assert_bf16(f64(dH), full["dH"], "dH vs the float64 chain")
    assert_bf16(f64(dW), full["dW"], "dW vs the float64 chain")


def test_ce_bad_label_sets_status(coda):
    import torch
    M, K, V = 64, 64, 512
    p = gen.ce_problem(M, K, V, seed=6)
    labels = p["labels"].copy()
    labels[5] = V          # out of range
    labels[9] = -1
    coda.coda_device_status(clear=True)
    pmax, psum, parg, tgt = coda.coda_gemm_ce_lse(dev_bf16(p["H"]), dev_bf16(p["W"]), torch.from_numpy(labels).cuda())
    st = coda.coda_device_status(clear=True)
    assert st & 2, f"status {st}"
    t = f64(tgt)
    assert math.isnan(t[5]) and math.isnan(t[9])
    assert np.all(np.isfinite(np.delete(t, [5, 9])))


def test_single_slot_input_ring_long_k(coda):
    """K > 3072: the two-box input epilogues (SwiGLU backward with its GU
    pre-activations; RMSNorm backward with the residual gradient) keep one chunk
    of inputs in their ring, and each CTA's last tile takes its remaining input
    boxes from the idle mainloop stages instead. Ragged shapes with more tiles
    than one wave, both tile variants, with and without the stream-K split (whose
    split pieces can be a CTA's last unit), against the oracle."""
    import torch
    M, F, K, d = 1800, 3400, 3208, 3400
    p = gen.swiglu_problem(M, K, F, seed=61)
    GU = gen.normal_bf16(np.random.default_rng(61), (M, 2 * F))
    dY, Wd, gu = dev_bf16(p["dY"]), dev_bf16(p["Wd"]), dev_bf16(GU)
    ref = O.gemm_swiglu_bwd(O.bf16(p["dY"]), O.bf16(p["Wd"]), O.bf16(GU))["dGU"]
    R = np.random.default_rng(62)
    dYr = gen.normal_bf16(R, (M, K))
    W1 = gen.normal_bf16(R, (d, K), std=K ** -0.5)
    h = gen.normal_bf16(R, (M, d))
    gamma = gen.normal_bf16(R, (d,), std=0.1, mean=1.0)
    dres = gen.normal_bf16(R, (M, d))
    r = (R.random(M) + 0.5).astype(np.float32)
    s = R.standard_normal(M).astype(np.float32)
    rr = O.gemm_rmsnorm_bwd_res(O.bf16(dYr), O.bf16(W1), O.bf16(h), O.bf16(gamma), r.astype(np.float64),
                                s.astype(np.float64), O.bf16(dres))
    dr, ds = _dev_f32(r), _dev_f32(s)
    try:
        for cg in (0, 1):
            for sk in (0, 2):
                coda.coda_set_cta_group(cg)
                coda.coda_set_stream_k(sk)
                out = coda.coda_gemm_swiglu_bwd(dY, Wd, gu)
                dh, pdg = coda.coda_gemm_rmsnorm_bwd_res(dev_bf16(dYr), dev_bf16(W1), dev_bf16(h), dev_bf16(gamma),
                                                         dr, ds, dev_bf16(dres))
                torch.cuda.synchronize()
                assert_bf16(f64(out), ref, f"SwiGLU bwd dGU (cta group {cg}, split {sk})")
                assert_bf16(f64(dh), rr["dh"], f"RMSNorm bwd + residual dh (cta group {cg}, split {sk})")
                assert_stat(f64(coda.coda_colsum_reduce(pdg)), rr["dgamma"], f"dgamma (cta group {cg}, split {sk})")
    finally:
        coda.coda_set_cta_group(0)
        coda.coda_set_stream_k(1)
    assert coda.coda_device_status(clear=True) == 0

