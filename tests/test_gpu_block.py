"""Parity of the block-level chain (one period of two GEMM-residual-RMSNorm-GEMM
structures, RoPE path then SwiGLU path) with the float64 oracle.

Gates, as for the single operators:
  * each kernel against the oracle evaluated on exactly the tensors that
    kernel consumed (the GPU's own stored bf16 intermediates and fp32
    statistics): bf16 outputs at rel Frobenius <= 5e-3 and
    max |err| / (1 + |ref|) <= 3e-2, fp32 statistics at 1e-4;
  * the chain's results end to end against the pure float64 chain. A result
    at the end of the chain has passed through up to about nine bf16
    roundings of stored tensors (h1, h1g, QKV, h2, h2g, GU, dGUr, dh2, dYqr),
    each adding a relative RMS error of about 2^-9/sqrt(3) = 1.1e-3, so the
    end-to-end bound is rel Frobenius <= 1e-2 and max |err| / (rms(ref) +
    |ref|) <= 5e-2 (the rms term keeps weight gradients, which are sums over
    all rows and sit far from 1 in scale, on the same footing).
"""
import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, assert_stat, col_tile_sums, dev_bf16, f64

pytestmark = pytest.mark.gpu

EPS = 1e-6
THETA = 10000.0
CHAIN_FRO = 1e-2
CHAIN_MAX = 5e-2


def _dev_f32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def assert_chain(got, ref, name):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    d = got - ref
    fro = np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30)
    mx = float(np.max(np.abs(d) / (np.sqrt(np.mean(ref * ref)) + np.abs(ref))))
    assert fro <= CHAIN_FRO and mx <= CHAIN_MAX, f"{name}: chain rel Frobenius {fro:.3e}, scaled max {mx:.3e}"


@pytest.fixture(params=[0, 1], ids=["auto", "cta1"])
def cta_group(coda, request):
    coda.coda_set_cta_group(request.param)
    yield request.param
    coda.coda_set_cta_group(0)


# ------------------------------------------------- the composed kernels alone

@pytest.mark.parametrize("M,d,F,hd,S", [(200, 256, 384, 64, 128), (77, 96, 136, 32, 50)])
def test_composed_kernels(coda, cta_group, M, d, F, hd, S):
    import torch
    p = gen.block_problem(M, d, F, seed=5)
    R = np.random.default_rng(6)
    r = (0.5 + R.random(M)).astype(np.float32)
    pos = np.arange(M) % S
    rc = 2 * d
    X = gen.normal_bf16(R, (M, d))
    cos, sin = coda.coda_rope_tables(S, hd, THETA)
    rd = _dev_f32(r)

    q = coda.coda_gemm_rowscale_rope(dev_bf16(X), dev_bf16(p["Wqkv"]), rd, cos, sin, hd, rc)
    assert_bf16(f64(q), O.gemm_rowscale_rope(O.bf16(X), O.bf16(p["Wqkv"]), r, pos, hd, THETA, rc), "rowscale+RoPE")

    A, GU = coda.coda_gemm_rowscale_swiglu(dev_bf16(X), dev_bf16(p["Wgu"]), rd, want_gu=True)
    ref = O.gemm_rowscale_swiglu(O.bf16(X), O.bf16(p["Wgu"]), r)
    assert_bf16(f64(GU), ref["GU"], "rowscale+SwiGLU GU")
    assert_bf16(f64(A), ref["A"], "rowscale+SwiGLU A")
    A2, none = coda.coda_gemm_rowscale_swiglu(dev_bf16(X), dev_bf16(p["Wgu"]), rd)
    assert none is None and torch.equal(A2, A)

    dgur, pdot = coda.coda_gemm_swiglu_bwd_rowdot(dev_bf16(p["gh"]), dev_bf16(p["Wdn"]), GU, rd)
    rb = O.gemm_swiglu_bwd_rowdot(O.bf16(p["gh"]), O.bf16(p["Wdn"]), f64(GU), r, d)
    assert_bf16(f64(dgur), rb["dGUr"], "SwiGLU bwd dGUr")
    assert pdot.shape == (M, coda.coda_num_col_tiles(F))
    # block t of the partials covers dA columns [128 t, 128 t + 128), i.e. GU columns [256 t, 256 t + 256)
    assert_stat(f64(pdot), col_tile_sums(rb["dGU"] * f64(GU), 256), "row-statistic partials")
    s2 = coda.coda_rowdot_reduce(pdot, d)
    assert_stat(f64(s2), rb["s"], "s from the GPU partials")

    h = gen.normal_bf16(R, (M, d))
    dres = gen.normal_bf16(R, (M, d))
    dh, pdg = coda.coda_gemm_rmsnorm_bwd_res(dgur, dev_bf16(p["Wgu"]), dev_bf16(h), dev_bf16(p["gamma2"]), rd, s2,
                                             dev_bf16(dres))
    rr = O.gemm_rmsnorm_bwd_res(f64(dgur), O.bf16(p["Wgu"]), O.bf16(h), O.bf16(p["gamma2"]), r, f64(s2),
                                O.bf16(dres))
    assert_bf16(f64(dh), rr["dh"], "RMSNorm bwd + residual dh")
    assert_stat(f64(coda.coda_colsum_reduce(pdg)), rr["dgamma"], "dgamma")

    qkv = dev_bf16(gen.normal_bf16(R, (M, 3 * d)))
    dqr, s1 = coda.coda_rope_bwd_rowdot(dev_bf16(p["dQKV"]), qkv, rd, cos, sin, hd, rc, d)
    rg = O.rope_bwd_rowdot(O.bf16(p["dQKV"]), f64(qkv), r, pos, hd, THETA, rc, d)
    assert_bf16(f64(dqr), rg["dYqr"], "RoPE glue dYqr")
    assert_stat(f64(s1), rg["s"], "RoPE glue s")


# ------------------------------------------------------- one period, small

def _block_inputs(coda, M, d, F, hd, S, seed):
    p = gen.block_problem(M, d, F, seed=seed)
    t = {k: dev_bf16(v) for k, v in p.items()}
    t["dQKV"] = t["dQKV"].clone()
    cos, sin = coda.coda_rope_tables(S, hd, THETA)
    return p, t, cos, sin


def _oracle_args(p, pos, hd, rc):
    b = {k: O.bf16(v) for k, v in p.items()}
    return b, (b["P"], b["Wd"], b["x"], b["gamma1"], b["Wqkv"], b["O"], b["Wo"], b["gamma2"], b["Wgu"], pos, hd,
               THETA, rc, EPS)


@pytest.mark.parametrize("M,d,F,hd,S", [(200, 256, 384, 64, 128), (300, 128, 264, 32, 100)])
def test_block_fused_chain(coda, cta_group, M, d, F, hd, S):
    rc = 2 * d
    pos = np.arange(M) % S
    p, t, cos, sin = _block_inputs(coda, M, d, F, hd, S, seed=7)
    blk = coda.CodaBlock(t, hd, rc, cos, sin, EPS).fwd().bwd()
    b, args = _oracle_args(p, pos, hd, rc)

    # forward, kernel by kernel on the tensors each consumed
    a1 = O.res_rmsprep(b["P"], b["Wd"], b["x"], b["gamma1"])
    assert_bf16(f64(blk.h1), a1["h1"], "h1")
    assert_bf16(f64(blk.h1g), a1["h2"], "h1g")
    assert_stat(f64(blk.r1), O.rms_scale(a1["h1"], EPS), "r1")
    assert_bf16(f64(blk.qkv), O.gemm_rowscale_rope(f64(blk.h1g), b["Wqkv"], f64(blk.r1), pos, hd, THETA, rc), "QKV")
    a2 = O.res_rmsprep(b["O"], b["Wo"], f64(blk.h1), b["gamma2"])
    assert_bf16(f64(blk.h2), a2["h1"], "h2")
    assert_bf16(f64(blk.h2g), a2["h2"], "h2g")
    assert_stat(f64(blk.r2), O.rms_scale(a2["h1"], EPS), "r2")
    sw = O.gemm_rowscale_swiglu(f64(blk.h2g), b["Wgu"], f64(blk.r2))
    assert_bf16(f64(blk.gu), sw["GU"], "GU")
    assert_bf16(f64(blk.a), sw["A"], "A")

    # backward, kernel by kernel
    b1 = O.gemm_swiglu_bwd_rowdot(b["gh"], b["Wdn"], f64(blk.gu), f64(blk.r2), d)
    assert_bf16(f64(blk.dgur), b1["dGUr"], "dGUr")
    assert_stat(f64(blk.s2), b1["s"], "s2")
    b3 = O.gemm_rmsnorm_bwd_res(f64(blk.dgur), b["Wgu"], f64(blk.h2), b["gamma2"], f64(blk.r2), f64(blk.s2), b["gh"])
    assert_bf16(f64(blk.dh2), b3["dh"], "dh2")
    assert_stat(f64(blk.dgamma2), b3["dgamma"], "dgamma2")
    assert_bf16(f64(blk.dWgu), O.matmul(f64(blk.h2g).T, f64(blk.dgur)), "dWgu")
    assert_bf16(f64(blk.dO), O.matmul(f64(blk.dh2), b["Wo"].T), "dO")
    assert_bf16(f64(blk.dWo), O.matmul(b["O"].T, f64(blk.dh2)), "dWo")
    g = O.rope_bwd_rowdot(b["dQKV"], f64(blk.qkv), f64(blk.r1), pos, hd, THETA, rc, d)
    assert_bf16(f64(blk.dqr), g["dYqr"], "dYqr")
    assert_stat(f64(blk.s1), g["s"], "s1")
    b10 = O.gemm_rmsnorm_bwd_res(f64(blk.dqr), b["Wqkv"], f64(blk.h1), b["gamma1"], f64(blk.r1), f64(blk.s1),
                                 f64(blk.dh2))
    assert_bf16(f64(blk.dh1), b10["dh"], "dh1")
    assert_stat(f64(blk.dgamma1), b10["dgamma"], "dgamma1")
    assert_bf16(f64(blk.dWqkv), O.matmul(f64(blk.h1g).T, f64(blk.dqr)), "dWqkv")
    assert_bf16(f64(blk.dWd), O.matmul(b["P"].T, f64(blk.dh1)), "dWd")

    # end to end against the pure float64 chain
    ref = O.block_bwd(*args, b["dQKV"], b["gh"], b["Wdn"])
    rf = ref["fwd"]
    for name, got in [("QKV", blk.qkv), ("h2", blk.h2), ("A", blk.a)]:
        assert_chain(f64(got), rf[name], f"{name} vs the float64 chain")
    for name, got in [("dh2", blk.dh2), ("dO", blk.dO), ("dWo", blk.dWo), ("dWgu", blk.dWgu), ("dh1", blk.dh1),
                      ("dWqkv", blk.dWqkv), ("dWd", blk.dWd), ("dgamma1", blk.dgamma1), ("dgamma2", blk.dgamma2)]:
        assert_chain(f64(got), ref[name], f"{name} vs the float64 chain")


def test_block_unfused_chain(coda):
    M, d, F, hd, S = 200, 256, 384, 64, 128
    rc = 2 * d
    pos = np.arange(M) % S
    p, t, cos, sin = _block_inputs(coda, M, d, F, hd, S, seed=8)
    blk = coda.CodaBlock(t, hd, rc, cos, sin, EPS, unfused=True).fwd_unfused().bwd_unfused()
    b, args = _oracle_args(p, pos, hd, rc)
    ref = O.block_bwd(*args, b["dQKV"], b["gh"], b["Wdn"])
    rf = ref["fwd"]
    # the unfused path stores n1, n2 in the h1g, h2g fields and rotates dQKV in place
    assert_chain(f64(blk.h1g), rf["n1"], "n1")
    assert_chain(f64(blk.h2g), rf["n2"], "n2")
    assert_bf16(f64(t["dQKV"]), O.rope_bwd(b["dQKV"], pos, hd, THETA, rc), "dQKV rotated in place")
    for name, got in [("QKV", blk.qkv), ("h2", blk.h2), ("A", blk.a), ("GU", blk.gu)]:
        assert_chain(f64(got), rf[name], f"unfused {name}")
    for name, got in [("dh2", blk.dh2), ("dO", blk.dO), ("dWo", blk.dWo), ("dWgu", blk.dWgu), ("dh1", blk.dh1),
                      ("dWqkv", blk.dWqkv), ("dWd", blk.dWd), ("dgamma1", blk.dgamma1), ("dgamma2", blk.dgamma2)]:
        assert_chain(f64(got), ref[name], f"unfused {name}")


def test_block_repeatable_and_empty(coda):
    """A second fused run on the same descriptor gives the same bits; M = 0 is a no-op."""
    import torch
    M, d, F, hd, S = 96, 64, 96, 32, 32
    p, t, cos, sin = _block_inputs(coda, M, d, F, hd, S, seed=9)
    blk = coda.CodaBlock(t, hd, 2 * d, cos, sin, EPS).fwd().bwd()
    first = {k: getattr(blk, k).clone() for k in ("qkv", "a", "dh1", "dWd", "dgamma1")}
    blk.fwd().bwd()
    for k, v in first.items():
        assert torch.equal(getattr(blk, k), v), k
    e = {k: v[:0] if k in ("P", "x", "O", "dQKV", "gh") else v for k, v in t.items()}
    coda.CodaBlock(e, hd, 2 * d, cos, sin, EPS).fwd().bwd()
