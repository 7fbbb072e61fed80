"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (automatic tile choice: SM-pair 256 x 256 tiles), checked on
sampled rows (row-local outputs) or sampled columns (weight and gamma
gradients) that the float64 oracle computes one by one."""
import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, assert_stat, dev_bf16, f64

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _rows(M, n=48, seed=0):
    r = np.random.default_rng(seed).choice(M, size=n - 2, replace=False)
    return np.unique(np.concatenate([[0, M - 1], r]))


def test_rope_qkv_4096(coda):
    M, K, N, hd, rc = 4096, 4096, 12288, 128, 8192
    p = gen.rope_problem(M, K, N, seed=0)
    X, W, A, B = (dev_bf16(p[k]) for k in ("X", "W", "A", "B"))
    c, s = coda.coda_rope_tables(4096, hd, 10000.0)
    out = coda.coda_gemm_rope(X, W, c, s, hd, rc)
    dP = coda.coda_gemm_rope_bwd(A, B, c, s, hd, rc)
    dX = coda.coda_gemm(dP, W, transB=True)
    dW = coda.coda_gemm(X, dP, transA=True)
    rows = _rows(M)
    W64 = O.bf16(p["W"])
    assert_bf16(f64(out[rows]), O.gemm_rope(O.bf16(p["X"][rows]), W64, rows, hd, 10000.0, rc), "QKV rows")
    assert_bf16(f64(dP[rows]), O.gemm_rope_bwd(O.bf16(p["A"][rows]), O.bf16(p["B"]), rows, hd, 10000.0, rc),
                "dP rows")
    dP64 = f64(dP)
    assert_bf16(f64(dX[rows]), O.matmul(dP64[rows], W64.T), "dX rows")
    cols = _rows(N, seed=1)
    assert_bf16(f64(dW[:, cols]), O.matmul(O.bf16(p["X"]).T, dP64[:, cols]), "dW columns")


def test_swiglu_up_4096(coda):
    M, K, F = 4096, 4096, 14336
    p = gen.swiglu_problem(M, K, F, seed=0)
    A, GU = coda.coda_gemm_swiglu(dev_bf16(p["X"]), dev_bf16(p["Wgu"]), want_gu=True)
    dGU = coda.coda_gemm_swiglu_bwd(dev_bf16(p["dY"]), dev_bf16(p["Wd"]), GU)
    rows = _rows(M)
    ref = O.gemm_swiglu(O.bf16(p["X"][rows]), O.bf16(p["Wgu"]))
    assert_bf16(f64(GU[rows]), ref["GU"], "GU rows")
    assert_bf16(f64(A[rows]), ref["A"], "A rows")
    rb = O.gemm_swiglu_bwd(O.bf16(p["dY"][rows]), O.bf16(p["Wd"]), f64(GU[rows]))
    assert_bf16(f64(dGU[rows]), rb["dGU"], "dGU rows")


def test_rmsnorm_chain_8192(coda):
    M = K = d = N2 = 8192
    p = gen.rms_chain(M, K, d, N2, seed=0, bwd_K=8192)
    x, W0, z, g, W1, dO, Wn = (dev_bf16(p[k]) for k in ("x", "W0", "z", "gamma", "W1", "dO", "Wn"))
    h1, h2, psq = coda.coda_gemm_res_rmsprep(x, W0, z, g)
    r = coda.coda_rms_reduce(psq, d, EPS)
    Y = coda.coda_gemm_rowscale(h2, W1, r)
    dY, dYr, pdot = coda.coda_gemm_rowdot(dO, Wn, Y, r)
    s = coda.coda_rowdot_reduce(pdot, d)
    dh1, pdg = coda.coda_gemm_rmsnorm_bwd(dY, W1, h1, g, r, s)
    dg = coda.coda_colsum_reduce(pdg)

    rows = _rows(M, n=32)
    W0_64, W1_64, g64 = O.bf16(p["W0"]), O.bf16(p["W1"]), O.bf16(p["gamma"])
    # forward, row-local: per kernel on its own inputs, and the float64 chain
    pr = O.res_rmsprep(O.bf16(p["x"][rows]), W0_64, O.bf16(p["z"][rows]), g64)
    assert_bf16(f64(h1[rows]), pr["h1"], "h1 rows")
    assert_bf16(f64(h2[rows]), pr["h2"], "h2 rows")
    assert_stat(f64(psq[rows]).sum(axis=1), pr["sumsq"], "sum of the psq partials")
    assert_stat(f64(r[rows]), O.rms_reduce(f64(psq[rows]), d, EPS), "r on the GPU partials")
    assert_bf16(f64(Y[rows]), O.rowscale(f64(h2[rows]), W1_64, f64(r[rows])), "Y rows (rowscale)")
    chain = O.gemm_rms_gemm_fwd(O.bf16(p["x"][rows]), W0_64, O.bf16(p["z"][rows]), g64, W1_64, EPS)
    assert_stat(f64(r[rows]), chain["r"], "r vs the float64 chain")
    assert_bf16(f64(Y[rows]), chain["Y"], "Y vs the float64 chain")
    # backward, row-local
    rd = O.gemm_rowdot(O.bf16(p["dO"][rows]), O.bf16(p["Wn"]), f64(Y[rows]), f64(r[rows]), d)
    assert_bf16(f64(dY[rows]), rd["dY"], "dY rows")
    assert_bf16(f64(dYr[rows]), rd["dYr"], "dYr rows")
    assert_stat(f64(s[rows]), rd["s"], "s rows")
    rb = O.gemm_rmsnorm_bwd(f64(dY[rows]), W1_64, f64(h1[rows]), g64, f64(r[rows]), f64(s[rows]))
    assert_bf16(f64(dh1[rows]), rb["dh1"], "dh1 rows")
    # dgamma on sampled columns: sum over all rows of r G h1, G[:, cols] = dY W1[cols]^T
    cols = _rows(d, n=32, seed=2)
    Gc = O.matmul(f64(dY), W1_64[cols].T)
    ref_dg = np.sum(f64(r)[:, None] * Gc * f64(h1)[:, cols], axis=0)
    assert_stat(f64(dg)[cols], ref_dg, "dgamma columns")


def test_lm_head_ce_8192(coda):
    import torch
    M, K, V = 8192, 4096, 32768
    p = gen.ce_problem(M, K, V, seed=0)
    H, W = dev_bf16(p["H"]), dev_bf16(p["W"])
    y = torch.from_numpy(p["labels"]).cuda()
    pmax, psum, parg, tgt = coda.coda_gemm_ce_lse(H, W, y)
    lse, loss_row, loss_mean, am = coda.coda_ce_reduce(pmax, psum, parg, tgt)
    dl = coda.coda_gemm_ce_bwd(H, W, y, lse, 1.0 / M)
    rows = _rows(M)
    L = O.matmul(O.bf16(p["H"][rows]), O.bf16(p["W"]))
    ref = O.ce_fwd(L, p["labels"][rows])
    assert_stat(f64(lse[rows]), ref["lse"], "lse rows")
    assert_stat(f64(loss_row[rows]), ref["loss_row"], "loss rows")
    lr = f64(loss_row)
    assert abs(float(loss_mean.item()) - lr.mean()) <= 1e-4 * abs(lr.mean()), "mean of the per-row losses"
    top2 = np.sort(L, axis=1)[:, -2:]
    sure = (top2[:, 1] - top2[:, 0]) > 1e-5 * np.sqrt(K) * np.max(np.abs(L), axis=1) + 1e-6
    assert np.array_equal(am.cpu().numpy()[rows][sure], ref["argmax"][sure])
    assert_bf16(f64(dl[rows]), O.ce_bwd(L, p["labels"][rows], f64(lse[rows]), 1.0 / M), "dl rows")


def test_block_chain_d4096(coda):
    """One period of the block-level chain at 16384 tokens, d = 4096, F = 14336:
    every kernel of the fused forward and backward on sampled rows (row-local
    outputs) or sampled columns (weight and gamma gradients), against the
    float64 oracle evaluated on the tensors that kernel consumed."""
    c = gen.WORKLOADS["block_d4096"]
    M, d, F, hd, rc, S = c["M"], c["d"], c["F"], c["head_dim"], c["rope_cols"], c["S"]
    p = gen.block_problem(M, d, F, seed=0)
    t = {k: dev_bf16(v) for k, v in p.items()}
    cos, sin = coda.coda_rope_tables(S, hd, c["theta"])
    blk = coda.CodaBlock(t, hd, rc, cos, sin, c["eps"]).fwd().bwd()
    b = {k: O.bf16(v) for k, v in p.items()}
    rows = _rows(M, n=24)
    pos = rows % S
    g = lambda x, r=rows: f64(x[r])  # noqa: E731

    # forward, row-local
    a1 = O.res_rmsprep(b["P"][rows], b["Wd"], b["x"][rows], b["gamma1"])
    assert_bf16(g(blk.h1), a1["h1"], "h1 rows")
    assert_bf16(g(blk.h1g), a1["h2"], "h1g rows")
    assert_stat(g(blk.r1), O.rms_scale(a1["h1"], c["eps"]), "r1 rows")
    assert_bf16(g(blk.qkv), O.gemm_rowscale_rope(g(blk.h1g), b["Wqkv"], g(blk.r1), pos, hd, c["theta"], rc),
                "QKV rows")
    a2 = O.res_rmsprep(b["O"][rows], b["Wo"], g(blk.h1), b["gamma2"])
    assert_bf16(g(blk.h2), a2["h1"], "h2 rows")
    assert_stat(g(blk.r2), O.rms_scale(a2["h1"], c["eps"]), "r2 rows")
    sw = O.gemm_rowscale_swiglu(g(blk.h2g), b["Wgu"], g(blk.r2))
    assert_bf16(g(blk.gu), sw["GU"], "GU rows")
    assert_bf16(g(blk.a), sw["A"], "A rows")

    # backward, row-local
    b1 = O.gemm_swiglu_bwd_rowdot(b["gh"][rows], b["Wdn"], g(blk.gu), g(blk.r2), d)
    assert_bf16(g(blk.dgur), b1["dGUr"], "dGUr rows")
    assert_stat(g(blk.s2), b1["s"], "s2 rows")
    b3 = O.gemm_rmsnorm_bwd_res(g(blk.dgur), b["Wgu"], g(blk.h2), b["gamma2"], g(blk.r2), g(blk.s2), b["gh"][rows])
    assert_bf16(g(blk.dh2), b3["dh"], "dh2 rows")
    assert_bf16(g(blk.dO), O.matmul(g(blk.dh2), b["Wo"].T), "dO rows")
    gl = O.rope_bwd_rowdot(b["dQKV"][rows], g(blk.qkv), g(blk.r1), pos, hd, c["theta"], rc, d)
    assert_bf16(g(blk.dqr), gl["dYqr"], "dYqr rows")
    assert_stat(g(blk.s1), gl["s"], "s1 rows")
    b10 = O.gemm_rmsnorm_bwd_res(g(blk.dqr), b["Wqkv"], g(blk.h1), b["gamma1"], g(blk.r1), g(blk.s1), g(blk.dh2))
    assert_bf16(g(blk.dh1), b10["dh"], "dh1 rows")

    # column outputs: sums over all 16384 rows, in row chunks
    cols = _rows(d, n=16, seed=3)
    cols_gu = _rows(2 * F, n=16, seed=4)
    cols_qkv = _rows(3 * d, n=16, seed=5)
    acc = {k: 0.0 for k in ("dg2", "dg1", "dWgu", "dWo", "dWqkv", "dWd")}
    for r0 in range(0, M, 2048):
        rr = np.arange(r0, min(M, r0 + 2048))
        dgur, dqr, dh1, dh2 = g(blk.dgur, rr), g(blk.dqr, rr), g(blk.dh1, rr), g(blk.dh2, rr)
        acc["dg2"] = acc["dg2"] + np.sum(O.matmul(dgur, b["Wgu"][cols].T) * g(blk.h2, rr)[:, cols], axis=0)
        acc["dg1"] = acc["dg1"] + np.sum(O.matmul(dqr, b["Wqkv"][cols].T) * g(blk.h1, rr)[:, cols], axis=0)
        acc["dWgu"] = acc["dWgu"] + O.matmul(g(blk.h2g, rr).T, dgur[:, cols_gu])
        acc["dWo"] = acc["dWo"] + O.matmul(b["O"][rr].T, dh2[:, cols])
        acc["dWqkv"] = acc["dWqkv"] + O.matmul(g(blk.h1g, rr).T, dqr[:, cols_qkv])
        acc["dWd"] = acc["dWd"] + O.matmul(b["P"][rr].T, dh1[:, cols])
    assert_stat(f64(blk.dgamma2[cols]), acc["dg2"], "dgamma2 columns")
    assert_stat(f64(blk.dgamma1[cols]), acc["dg1"], "dgamma1 columns")
    assert_bf16(f64(blk.dWgu[:, cols_gu]), acc["dWgu"], "dWgu columns")
    assert_bf16(f64(blk.dWo[:, cols]), acc["dWo"], "dWo columns")
    assert_bf16(f64(blk.dWqkv[:, cols_qkv]), acc["dWqkv"], "dWqkv columns")
    assert_bf16(f64(blk.dWd[:, cols]), acc["dWd"], "dWd columns")
    assert coda.coda_device_status(clear=True) == 0
