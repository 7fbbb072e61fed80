"""Parity at the edges of the method, where the epilogues' hardware
approximations (ex2.approx.ftz, rcp.approx.ftz) and the online rescaling are
most likely to go wrong while ordinary N(0,1) inputs stay well inside:

* cross-entropy with logits spanning about +-60: row maxima in the last
  32-column chunk of the last, ragged vocabulary tile (so the running max is
  raised chunk after chunk and the running sum rescaled), far tails that
  underflow exp, and labels at column 0, at V-1 and at the first column of
  the ragged block (CODA note, Key design 4: the online log-sum-exp);
* SwiGLU forward and backward with gates |G| up to about 200 in both signs,
  where sigmoid saturates to exactly 0 or 1 and no 0 * inf may appear (CODA
  note, Key design 2; pith page, Figure 7 caption);
* GEMM-residual-RMSNorm-GEMM with all-zero residual rows, where r reaches its
  largest value eps^-1/2 = 1000, through forward and backward (CODA note, Key
  designs 1 and 3; eps inside the square root as in the pith page's Figure 5
  caption);
* RoPE at the last positions S-32 .. S-1 of S = 4096 on the angle-addition
  table path (CODA note, Key design 2).

Every comparison is element by element against the float64 oracle on the
exact tensors the kernel consumed, at the same tolerances as the other parity
tests (tests/_util.py)."""
import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, assert_stat, col_tile_sums, dev_bf16, f64

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _rngs(seed, n):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


# ---------------------------------------------------------------- cross-entropy

def _ce_edge_problem(M=320, K=64, V=1000, seed=11):
    """Logits L = H W built from K pattern rows of W: row i of H selects pattern
    k_i with weight a_i in {60, 40} plus noise of std 0.002 on the other rows,
    so L[i] = a_i W[k_i] + (small). Patterns: a ramp rising to its peak at V-1
    (the running max grows in every chunk), a ramp falling from column 0 (the
    far tail underflows exp), and uniform(-1, 0.9) rows with a single 1.0 spike
    at a chosen column (last chunk of the ragged last tile, the tile's first
    column, block edges, column 0)."""
    r = _rngs(seed, 4)
    cols = np.arange(V)
    spikes = [999, 995, 992, 896, 0, 127, 128, 991, 500, 31, 32, 897]
    Wf = np.empty((K, V), np.float32)
    for k in range(K):
        kind = k % 4
        if kind == 0:
            Wf[k] = -1.0 + 1.8 * cols / (V - 1)
            Wf[k, V - 1] = 1.0
        elif kind == 1:
            Wf[k] = 0.8 - 1.8 * cols / (V - 1)
            Wf[k, 0] = 1.0
        else:
            Wf[k] = r[0].uniform(-1.0, 0.9, V)
            Wf[k, spikes[k % len(spikes)]] = 1.0
    Hf = (0.002 * r[1].standard_normal((M, K))).astype(np.float32)
    ki = r[2].integers(0, K, M)
    Hf[np.arange(M), ki] = np.where(np.arange(M) % 3 == 0, 40.0, 60.0)
    return gen.f32_to_bf16_bits(Hf), gen.f32_to_bf16_bits(Wf), r[3]


def test_ce_wide_logits_ragged_vocab(coda):
    import torch
    M, K, V = 320, 64, 1000          # V = 7 x 128 + 104: the last tile is ragged
    Hb, Wb, rl = _ce_edge_problem(M, K, V)
    L = O.matmul(O.bf16(Hb), O.bf16(Wb))
    assert L.max() > 55 and L.min() < -55, "the construction must span about +-60"
    am_ref = np.argmax(L, axis=1)
    assert np.sum(am_ref >= 992) >= M // 8, "many row maxima in the last chunk of the last tile"
    # labels: column 0, V-1, the first column of the ragged block, the row's argmax, random
    choice = np.stack([np.zeros(M, np.int64), np.full(M, V - 1), np.full(M, 896), am_ref,
                       rl.integers(0, V, M)], axis=1)
    labels = choice[np.arange(M), np.arange(M) % 5].astype(np.int32)

    H, W = dev_bf16(Hb), dev_bf16(Wb)
    y = torch.from_numpy(labels).cuda()
    pmax, psum, parg, tgt = coda.coda_gemm_ce_lse(H, W, y)
    ref = O.ce_fwd(L, labels)
    nb = coda.coda_num_col_tiles(V)
    tiles = [(t * 128, min(V, t * 128 + 128)) for t in range(nb)]
    assert_stat(f64(pmax), np.stack([L[:, a:b].max(axis=1) for a, b in tiles], axis=1), "pmax")
    ref_psum = np.stack([np.exp(L[:, a:b] - f64(pmax)[:, [t]]).sum(axis=1) for t, (a, b) in enumerate(tiles)],
                        axis=1)
    assert_stat(f64(psum), ref_psum, "psum (relative to the GPU's own tile max)")
    assert_stat(f64(tgt), ref["tgt"], "target logit at columns 0, V-1, 896")
    lse, loss_row, loss_mean, argmax = coda.coda_ce_reduce(pmax, psum, parg, tgt)
    assert_stat(f64(lse), ref["lse"], "lse")
    assert_stat(f64(loss_row), ref["loss_row"], "loss_row")
    assert abs(float(loss_mean.item()) - ref["loss_mean"]) <= 1e-4 * abs(ref["loss_mean"])
    # every row's top-2 gap is at least 40 x 0.1 by construction: argmax exact on all rows
    top2 = np.sort(L, axis=1)[:, -2:]
    assert np.min(top2[:, 1] - top2[:, 0]) > 1.0
    assert np.array_equal(argmax.cpu().numpy(), ref["argmax"])

    g = 1.0 / M
    dl = coda.coda_gemm_ce_bwd(H, W, y, lse, g)
    dl_ref = O.ce_bwd(L, labels, f64(lse), g)
    assert_bf16(f64(dl), dl_ref, "dl")
    # the label entries, where exp(l - lse) - 1 cancels
    rows = np.arange(M)
    assert_bf16(f64(dl)[rows, labels], dl_ref[rows, labels], "dl at the labels")
    dH = coda.coda_gemm(dl, W, transB=True)
    assert_bf16(f64(dH), O.matmul(f64(dl), O.bf16(Wb).T), "dH = dl W^T")


# ---------------------------------------------------------------- SwiGLU

def _saturated_swiglu(M, K, F, seed):
    """X ~ N(0,1); gate columns (even) of Wgu ~ N(0, 50^2 / K), up columns
    N(0, 1/K): gates G ~ N(0, 50^2), |G| up to about 200."""
    r = _rngs(seed, 4)
    X = gen.normal_bf16(r[0], (M, K))
    Wf = (r[1].standard_normal((K, 2 * F)) / np.sqrt(K)).astype(np.float32)
    Wf[:, 0::2] *= 50.0
    dY = gen.normal_bf16(r[2], (M, K))
    Wd = gen.normal_bf16(r[3], (F, K), std=1.0 / np.sqrt(F))
    return X, gen.f32_to_bf16_bits(Wf), dY, Wd


def test_swiglu_saturated_gates(coda):
    M, K, F = 300, 64, 264
    Xb, Wb, dYb, Wdb = _saturated_swiglu(M, K, F, seed=12)
    A, GU = coda.coda_gemm_swiglu(dev_bf16(Xb), dev_bf16(Wb), want_gu=True)
    ref = O.gemm_swiglu(O.bf16(Xb), O.bf16(Wb))
    G = ref["GU"][:, 0::2]
    assert np.sum(G > 88) > 100 and np.sum(G < -88) > 100, "gates must reach the saturated range"
    assert_bf16(f64(GU), ref["GU"], "GU")
    assert_bf16(f64(A), ref["A"], "A = silu(G) U")
    # saturated negative gates give exactly zero (no 0 * inf)
    Gg = f64(GU)[:, 0::2]
    assert np.all(f64(A)[Gg < -100] == 0.0)

    dGU = coda.coda_gemm_swiglu_bwd(dev_bf16(dYb), dev_bf16(Wdb), GU)
    rb = O.gemm_swiglu_bwd(O.bf16(dYb), O.bf16(Wdb), f64(GU))
    assert_bf16(f64(dGU), rb["dGU"], "dGU")
    sat = np.abs(Gg) > 88
    assert_bf16(f64(dGU)[:, 0::2][sat], rb["dGU"][:, 0::2][sat], "dG where the gate saturates")
    assert_bf16(f64(dGU)[:, 1::2][sat], rb["dGU"][:, 1::2][sat], "dU where the gate saturates")


def test_swiglu_saturated_gates_rowscale_rowdot(coda):
    """The block chain's SwiGLU pair (row-scaled forward, backward with the
    row statistic), whose fp32 statistic depends on the saturated sigmoid."""
    import torch
    M, K, F, d = 300, 64, 264, 64
    Xb, Wb, dYb, Wdb = _saturated_swiglu(M, K, F, seed=13)
    r = 0.5 + _rngs(14, 1)[0].random(M)
    rd = torch.from_numpy(r.astype(np.float32)).cuda()
    r32 = f64(rd)
    A, GU = coda.coda_gemm_rowscale_swiglu(dev_bf16(Xb), dev_bf16(Wb), rd, want_gu=True)
    ref = O.gemm_rowscale_swiglu(O.bf16(Xb), O.bf16(Wb), r32)
    assert_bf16(f64(GU), ref["GU"], "GU")
    assert_bf16(f64(A), ref["A"], "A")
    dgur, pdot = coda.coda_gemm_swiglu_bwd_rowdot(dev_bf16(dYb), dev_bf16(Wdb), GU, rd)
    rb = O.gemm_swiglu_bwd_rowdot(O.bf16(dYb), O.bf16(Wdb), f64(GU), r32, d)
    assert_bf16(f64(dgur), rb["dGUr"], "dGUr")
    assert_stat(f64(pdot), col_tile_sums(rb["dGU"] * f64(GU), 256), "row-statistic partials")
    assert_stat(f64(coda.coda_rowdot_reduce(pdot, d)), rb["s"], "s")


# ---------------------------------------------------------------- RMSNorm chain

def test_rms_chain_zero_residual_rows(coda):
    """Rows with x = 0 and z = 0 have h1 = 0, so r = eps^-1/2 = 1000, h2 = Y =
    0, s = 0 and dh1 = r gamma G: the largest row scale the chain can see."""
    M, K, d, N2, Kn = 300, 200, 264, 520, 136
    p = gen.rms_chain(M, K, d, N2, seed=15, bwd_K=Kn)
    x, z = p["x"].copy(), p["z"].copy()
    zero = np.array([0, 131, 255, 256, M - 1])   # first row, inside and across tile edges, last row
    x[zero] = 0
    z[zero] = 0
    W0, g, W1 = p["W0"], p["gamma"], p["W1"]
    h1, h2, psq = coda.coda_gemm_res_rmsprep(dev_bf16(x), dev_bf16(W0), dev_bf16(z), dev_bf16(g))
    ref = O.res_rmsprep(O.bf16(x), O.bf16(W0), O.bf16(z), O.bf16(g))
    assert_bf16(f64(h1), ref["h1"], "h1")
    assert np.all(f64(h1)[zero] == 0.0) and np.all(f64(psq)[zero] == 0.0)
    r = coda.coda_rms_reduce(psq, d, EPS)
    chain = O.gemm_rms_gemm_fwd(O.bf16(x), O.bf16(W0), O.bf16(z), O.bf16(g), O.bf16(W1), EPS)
    assert_stat(f64(r), chain["r"], "r")
    assert np.allclose(f64(r)[zero], 1000.0, rtol=1e-6)
    Y = coda.coda_gemm_rowscale(h2, dev_bf16(W1), r)
    assert_bf16(f64(Y), chain["Y"], "Y vs the float64 chain")
    assert np.all(f64(Y)[zero] == 0.0)

    dY, dYr, pdot = coda.coda_gemm_rowdot(dev_bf16(p["dO"]), dev_bf16(p["Wn"]), Y, r)
    rd = O.gemm_rowdot(O.bf16(p["dO"]), O.bf16(p["Wn"]), f64(Y), f64(r), d)
    assert_bf16(f64(dYr), rd["dYr"], "dYr = r dY (r = 1000 on the zero rows)")
    s = coda.coda_rowdot_reduce(pdot, d)
    assert_stat(f64(s), rd["s"], "s")
    assert np.all(f64(s)[zero] == 0.0)
    dh1, pdg = coda.coda_gemm_rmsnorm_bwd(dY, dev_bf16(W1), h1, dev_bf16(g), r, s)
    rb = O.gemm_rmsnorm_bwd(f64(dY), O.bf16(W1), f64(h1), O.bf16(g), f64(r), f64(s))
    assert_bf16(f64(dh1), rb["dh1"], "dh1")
    assert_bf16(f64(dh1)[zero], rb["dh1"][zero], "dh1 on the zero rows (r gamma G)")
    full = O.gemm_rms_gemm_bwd(O.bf16(x), O.bf16(W0), O.bf16(z), O.bf16(g), O.bf16(W1), EPS, f64(dY))
    assert_bf16(f64(dh1), full["dh1"], "dh1 vs the float64 chain")
    assert_stat(f64(coda.coda_colsum_reduce(pdg)), rb["dgamma"], "dgamma")


# ---------------------------------------------------------------- RoPE

def test_rope_last_positions(coda):
    """Rows at positions S-32 .. S-1 (S = 4096) and the wrap back to 0, on the
    angle-addition path (S % 32 == 0, head_dim 128): cos/sin of position
    p0 + l formed from table rows p0 and l."""
    M, K, N, hd, rc, S, theta = 4160, 64, 768, 128, 512, 4096, 10000.0
    c, s = coda.coda_rope_tables(S, hd, theta)
    p = gen.rope_problem(M, K, N, seed=16)
    pos = np.arange(M) % S
    out = coda.coda_gemm_rope(dev_bf16(p["X"]), dev_bf16(p["W"]), c, s, hd, rc)
    ref = O.gemm_rope(O.bf16(p["X"]), O.bf16(p["W"]), pos, hd, theta, rc)
    assert_bf16(f64(out), ref, "rope fwd")
    last = slice(S - 32, S)
    assert_bf16(f64(out)[last], ref[last], "rope fwd at positions S-32..S-1")
    assert_bf16(f64(out)[S:S + 32], ref[S:S + 32], "rope fwd after the wrap (positions 0..31)")
    g = coda.coda_gemm_rope_bwd(dev_bf16(p["A"]), dev_bf16(p["B"]), c, s, hd, rc)
    rg = O.gemm_rope_bwd(O.bf16(p["A"]), O.bf16(p["B"]), pos, hd, theta, rc)
    assert_bf16(f64(g), rg, "rope bwd")
    assert_bf16(f64(g)[last], rg[last], "rope bwd at positions S-32..S-1")


# ---------------------------------------------------------------- FP8 mainloop

def _dev_u8(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).cuda()


def test_ce_fp8_wide_logits(coda):
    """The FP8 (E4M3) mainloop feeds the same online log-sum-exp: logits of
    about +-60 formed as alpha * (H W^T) with alpha = 4 and E4M3 operands."""
    import torch
    M, K, V = 320, 64, 1000
    Hb, Wb, rl = _ce_edge_problem(M, K, V)
    # the bf16 construction re-encoded: H / 4 (40 and 60 become 10 and 15, exact in E4M3), W^T stored [V, K]
    H8 = gen.f32_to_e4m3_bits(O.bf16(Hb).astype(np.float32) / 4.0)
    W8 = gen.f32_to_e4m3_bits(np.ascontiguousarray(O.bf16(Wb).T.astype(np.float32)))
    a, b, alpha = O.e4m3(H8), O.e4m3(W8), 4.0
    L = alpha * O.matmul(a, b.T)
    assert L.max() > 55 and L.min() < -55
    am_ref = np.argmax(L, axis=1)
    choice = np.stack([np.zeros(M, np.int64), np.full(M, V - 1), np.full(M, 896), am_ref, rl.integers(0, V, M)],
                      axis=1)
    labels = choice[np.arange(M), np.arange(M) % 5].astype(np.int32)
    y = torch.from_numpy(labels).cuda()
    pmax, psum, parg, tgt = coda.coda_gemm_ce_lse_fp8(_dev_u8(H8), _dev_u8(W8), alpha, y)
    lse, loss_row, _, argmax = coda.coda_ce_reduce(pmax, psum, parg, tgt)
    ref = O.ce_fwd(L, labels)
    assert_stat(f64(lse), ref["lse"], "fp8 lse")
    assert_stat(f64(loss_row), ref["loss_row"], "fp8 loss rows")
    top2 = np.sort(L, axis=1)[:, -2:]
    sure = (top2[:, 1] - top2[:, 0]) > 1e-5 * np.sqrt(K) * np.max(np.abs(L), axis=1) + 1e-6
    assert sure.mean() > 0.9
    assert np.array_equal(argmax.cpu().numpy()[sure], ref["argmax"][sure])
    dl = coda.coda_gemm_ce_bwd_fp8(_dev_u8(H8), _dev_u8(W8), alpha, y, lse, 1.0 / M)
    assert_bf16(f64(dl), O.ce_bwd(L, labels, f64(lse), 1.0 / M), "fp8 dl")


def test_swiglu_fp8_saturated_gates(coda):
    """FP8 SwiGLU forward with gates |G| up to about 200 (E4M3 operands)."""
    M, K, F = 300, 64, 264
    Xb, Wb, _, _ = _saturated_swiglu(M, K, F, seed=17)
    X8 = gen.f32_to_e4m3_bits(O.bf16(Xb).astype(np.float32))
    W8 = gen.f32_to_e4m3_bits(np.ascontiguousarray(O.bf16(Wb).T.astype(np.float32) * 8.0))  # [2F, K]
    a, b, alpha = O.e4m3(X8), O.e4m3(W8), 0.125
    A, GU = coda.coda_gemm_swiglu_fp8(_dev_u8(X8), _dev_u8(W8), alpha, want_gu=True)
    ref = O.gemm_swiglu(a, alpha * b.T)
    G = ref["GU"][:, 0::2]
    assert np.sum(G > 88) > 100 and np.sum(G < -88) > 100
    assert_bf16(f64(GU), ref["GU"], "fp8 GU")
    assert_bf16(f64(A), ref["A"], "fp8 A = silu(G) U")
    assert np.all(f64(A)[f64(GU)[:, 0::2] < -100] == 0.0)
