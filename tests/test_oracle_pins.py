"""Pins for the float64 oracle: it must agree with things other than itself.

Each test checks an oracle function against one of
  * an identity the CODA pages state (commutation of r with the right
    multiply; the row-statistic identity of the RMSNorm backward),
  * a torch float64 library routine (rms_norm, silu, cross_entropy,
    logsumexp, autograd),
  * a closed form / invariant (rotation norms and group law, scale
    invariance of RMSNorm, W = 0 cross-entropy),
  * central finite differences, or
  * brute-force scalar loops on tiny shapes,
chosen so that a dropped term, a wrong sign or index, or a transposed
operand in the oracle fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import coda_inputs as gen
import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_values.json")


def rng(seed=1):
    return np.random.default_rng(seed)


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def t64(a, grad=False):
    return torch.tensor(np.asarray(a, np.float64), dtype=torch.float64, requires_grad=grad)


# ---------------------------------------------------------------------------
# GEMM-RMSNorm-GEMM forward
# ---------------------------------------------------------------------------

def _chain(M=6, K=5, d=7, N2=4, seed=3):
    r = rng(seed)
    return (r.standard_normal((M, K)), r.standard_normal((K, d)) / np.sqrt(K), r.standard_normal((M, d)),
            1 + 0.1 * r.standard_normal(d), r.standard_normal((d, N2)) / np.sqrt(d))


def test_rmsnorm_matches_torch_rms_norm():
    x, W0, z, g, W1 = _chain()
    h1 = x @ W0 + z
    n, r = O.rmsnorm(h1, g, 1e-6)
    ref = F.rms_norm(t64(h1), (h1.shape[1],), weight=t64(g), eps=1e-6).numpy()
    assert rel(n, ref) < 1e-13


def test_commutation_identity_and_fused_pieces():
    """RMSNorm(xW0+z, gamma) W1 = r ((xW0+z) (.) gamma) W1 (CODA note, Key design 1),
    and the three fused pieces (rmsprep -> reduce -> rowscale) rebuild Y."""
    x, W0, z, g, W1 = _chain(M=9, K=8, d=12, N2=5)
    eps = 1e-6
    f = O.gemm_rms_gemm_fwd(x, W0, z, g, W1, eps)
    h1 = x @ W0 + z
    r = 1.0 / np.sqrt(np.mean(h1 ** 2, axis=1) + eps)
    reparam = r[:, None] * ((h1 * g[None, :]) @ W1)
    assert rel(f["Y"], reparam) < 1e-13
    p = O.res_rmsprep(x, W0, z, g)
    # tile partials: split the 12 columns into tiles of 5 (ragged last tile)
    parts = np.stack([np.sum(p["h1"][:, c:c + 5] ** 2, axis=1) for c in range(0, 12, 5)], axis=1)
    r2 = O.rms_reduce(parts, 12, eps)
    assert rel(r2, f["r"]) < 1e-14
    assert rel(O.rowscale(p["h2"], W1, r2), f["Y"]) < 1e-13
    assert rel(p["h1"], f["h1"]) < 1e-15 and rel(p["h2"], f["h2"]) < 1e-15


def test_textbook_special_case():
    """gamma = 1, z = 0, W1 = I reduces the block to plain RMSNorm of x W0."""
    x, W0, _, _, _ = _chain(d=6)
    d = 6
    f = O.gemm_rms_gemm_fwd(x, W0, np.zeros((x.shape[0], d)), np.ones(d), np.eye(d), 1e-5)
    ref = F.rms_norm(t64(x @ W0), (d,), eps=1e-5).numpy()
    assert rel(f["Y"], ref) < 1e-13


def test_constant_row_closed_form():
    c, eps = -1.75, 1e-3
    r = O.rms_scale(np.full((1, 9), c), eps)
    assert abs(r[0] - 1.0 / math.sqrt(c * c + eps)) < 1e-15


def test_eps_placement_detects_outside_sqrt():
    """eps inside the sqrt: for a tiny row the two placements differ a lot."""
    h = np.full((1, 4), 1e-4)
    r = O.rms_scale(h, 1e-6)
    assert abs(r[0] - 1 / math.sqrt(1e-8 + 1e-6)) < 1e-9
    assert abs(r[0] - 1 / (1e-4 + 1e-6)) > 1.0


# ---------------------------------------------------------------------------
# GEMM-RMSNorm-GEMM backward
# ---------------------------------------------------------------------------

def test_chain_bwd_matches_torch_autograd():
    x, W0, z, g, W1 = _chain(M=7, K=6, d=10, N2=9, seed=11)
    dY = rng(12).standard_normal((7, 9))
    eps = 1e-6
    o = O.gemm_rms_gemm_bwd(x, W0, z, g, W1, eps, dY)
    tx, tW0, tz, tg, tW1 = (t64(a, True) for a in (x, W0, z, g, W1))
    Y = F.rms_norm(tx @ tW0 + tz, (10,), weight=tg, eps=eps) @ tW1
    (Y * t64(dY)).sum().backward()
    for name, tref in (("dx", tx), ("dW0", tW0), ("dz", tz), ("dgamma", tg), ("dW1", tW1)):
        assert rel(o[name], tref.grad.numpy()) < 1e-12, name


def test_chain_bwd_finite_differences():
    M, K, d, N2 = 3, 4, 5, 3
    x, W0, z, g, W1 = _chain(M, K, d, N2, seed=21)
    dY = rng(22).standard_normal((M, N2))
    eps = 1e-6
    o = O.gemm_rms_gemm_bwd(x, W0, z, g, W1, eps, dY)
    args = dict(x=x, W0=W0, z=z, gamma=g, W1=W1)

    def loss(a):
        return float(np.sum(dY * O.gemm_rms_gemm_fwd(a["x"], a["W0"], a["z"], a["gamma"], a["W1"], eps)["Y"]))

    grads = dict(x=o["dx"], W0=o["dW0"], z=o["dz"], gamma=o["dgamma"], W1=o["dW1"])
    h = 1e-6
    for name, arr in args.items():
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a_p = {k: v.copy() for k, v in args.items()}
            a_m = {k: v.copy() for k, v in args.items()}
            a_p[name][idx] += h
            a_m[name][idx] -= h
            num[idx] = (loss(a_p) - loss(a_m)) / (2 * h)
        assert rel(grads[name], num) < 1e-7, name


def test_s_identity_and_r2_form():
    """rowsum((dY W1^T) (.) h2) = rowsum(dY (.) h2 W1) (CODA note, Key design 3), and
    s on the final Y equals r times the pages' statistic on h3."""
    x, W0, z, g, W1 = _chain(M=8, K=6, d=9, N2=7, seed=5)
    dY = rng(6).standard_normal((8, 7))
    f = O.gemm_rms_gemm_fwd(x, W0, z, g, W1, 1e-6)
    lhs = np.sum((dY @ W1.T) * f["h2"], axis=1)
    rhs = np.sum(dY * f["h3"], axis=1)
    assert rel(lhs, rhs) < 1e-12
    s = O.rowdot_stat(dY, f["Y"], 9)
    assert rel(s, f["r"] * rhs / 9) < 1e-12


def test_rmsnorm_bwd_scale_invariance():
    """With eps = 0, RMSNorm is invariant to row scaling, so rowsum(h1 (.) dh1) = 0."""
    x, W0, z, g, W1 = _chain(M=5, K=4, d=8, N2=6, seed=8)
    dY = rng(9).standard_normal((5, 6))
    o = O.gemm_rms_gemm_bwd(x, W0, z, g, W1, 0.0, dY)
    h1 = x @ W0 + z
    dots = np.sum(h1 * o["dh1"], axis=1)
    assert np.max(np.abs(dots)) < 1e-12 * np.max(np.abs(o["dh1"])) * np.max(np.abs(h1)) * 8


def test_gemm_rowdot_and_rmsnorm_bwd_pieces():
    """The backward kernels' oracle pieces compose to the chain gradient."""
    x, W0, z, g, W1 = _chain(M=6, K=5, d=8, N2=7, seed=31)
    R = rng(32)
    dO = R.standard_normal((6, 4))
    Wn = R.standard_normal((4, 7))
    f = O.gemm_rms_gemm_fwd(x, W0, z, g, W1, 1e-6)
    rd = O.gemm_rowdot(dO, Wn, f["Y"], f["r"], 8)
    full = O.gemm_rms_gemm_bwd(x, W0, z, g, W1, 1e-6, dO @ Wn)
    assert rel(rd["s"], full["s"]) < 1e-13
    assert rel(rd["dYr"], full["dYr"]) < 1e-14
    b = O.gemm_rmsnorm_bwd(rd["dY"], W1, f["h1"], g, f["r"], rd["s"])
    assert rel(b["dh1"], full["dh1"]) < 1e-13
    assert rel(b["dgamma"], full["dgamma"]) < 1e-13


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------

def test_silu_matches_torch():
    g = np.linspace(-30, 30, 301)
    assert rel(O.silu(g), F.silu(t64(g)).numpy()) < 1e-15
    assert O.silu(np.array([0.0]))[0] == 0.0
    big = np.array([50.0])
    assert abs(O.silu(big)[0] - 50.0) < 1e-12


def test_swiglu_layout_and_autograd():
    R = rng(41)
    GU = R.standard_normal((5, 12)) * 3
    dA = R.standard_normal((5, 6))
    A = O.swiglu(GU)
    tGU = t64(GU, True)
    tA = F.silu(tGU[:, 0::2]) * tGU[:, 1::2]
    assert rel(A, tA.detach().numpy()) < 1e-15
    (tA * t64(dA)).sum().backward()
    assert rel(O.swiglu_bwd(dA, GU), tGU.grad.numpy()) < 1e-13
    # the gate is the even channel: zeroing the odd (up) channels zeroes the output
    GU2 = GU.copy()
    GU2[:, 1::2] = 0
    assert np.all(O.swiglu(GU2) == 0)
    GU3 = GU.copy()
    GU3[:, 0::2] = 0
    assert np.all(O.swiglu(GU3) == 0)


def test_swiglu_bwd_finite_differences():
    R = rng(43)
    GU = R.standard_normal((2, 6))
    dA = R.standard_normal((2, 3))
    an = O.swiglu_bwd(dA, GU)
    h = 1e-6
    num = np.zeros_like(GU)
    for idx in np.ndindex(GU.shape):
        p, m = GU.copy(), GU.copy()
        p[idx] += h
        m[idx] -= h
        num[idx] = (np.sum(dA * O.swiglu(p)) - np.sum(dA * O.swiglu(m))) / (2 * h)
    assert rel(an, num) < 1e-8


def test_gemm_swiglu_bwd_chain():
    R = rng(44)
    X = R.standard_normal((4, 6))
    Wgu = R.standard_normal((6, 10))
    Wd = R.standard_normal((5, 6))
    dY = R.standard_normal((4, 6))
    tX, tW, tWd = t64(X, True), t64(Wgu, True), t64(Wd, True)
    GU = tX @ tW
    out = (F.silu(GU[:, 0::2]) * GU[:, 1::2]) @ tWd
    (out * t64(dY)).sum().backward()
    o = O.gemm_swiglu_bwd(dY, Wd, X @ Wgu)
    assert rel(o["dGU"] @ Wgu.T, tX.grad.numpy()) < 1e-12
    assert rel(X.T @ o["dGU"], tW.grad.numpy()) < 1e-12


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def _rope_complex(P, pos, hd, theta, rope_cols):
    """Independent closed form: pair (2i, 2i+1) as a complex number times e^{i a}."""
    out = np.array(P, np.float64, copy=True)
    for h in range(rope_cols // hd):
        for i in range(hd // 2):
            c = h * hd + 2 * i
            a = np.asarray(pos, np.float64) * (theta ** (-2.0 * i / hd))
            zc = (P[:, c] + 1j * P[:, c + 1]) * np.exp(1j * a)
            out[:, c], out[:, c + 1] = zc.real, zc.imag
    return out


def test_rope_matches_complex_form_and_passthrough():
    R = rng(51)
    P = R.standard_normal((7, 24))
    pos = np.array([0, 1, 2, 5, 100, 4095, 17])
    o = O.rope(P, pos, 8, 10000.0, 16)
    assert rel(o, _rope_complex(P, pos, 8, 10000.0, 16)) < 1e-13
    assert np.array_equal(o[:, 16:], P[:, 16:])
    assert np.array_equal(o[0], P[0])  # position 0 is the identity


def test_rope_invariants():
    R = rng(52)
    P = R.standard_normal((5, 16))
    p = np.array([3, 9, 40, 1000, 4095])
    q = np.array([1, 7, 11, 2, 0])
    f = O.rope(P, p, 16, 10000.0, 16)
    norms = lambda A: A[:, 0::2] ** 2 + A[:, 1::2] ** 2  # noqa: E731
    assert rel(norms(f), norms(P)) < 1e-13
    assert rel(O.rope_bwd(f, p, 16, 10000.0, 16), P) < 1e-13         # bwd o fwd = id
    assert rel(O.rope(f, q, 16, 10000.0, 16), O.rope(P, p + q, 16, 10000.0, 16)) < 1e-12  # R(q)R(p) = R(p+q)
    Y = R.standard_normal((5, 16))                                      # adjoint
    assert abs(np.sum(f * Y) - np.sum(P * O.rope_bwd(Y, p, 16, 10000.0, 16))) < 1e-12


def test_rope_bwd_finite_differences():
    R = rng(53)
    P = R.standard_normal((3, 8))
    dO = R.standard_normal((3, 8))
    pos = np.array([2, 5, 11])
    an = O.rope_bwd(dO, pos, 4, 10000.0, 8)
    h = 1e-6
    num = np.zeros_like(P)
    for idx in np.ndindex(P.shape):
        a, b = P.copy(), P.copy()
        a[idx] += h
        b[idx] -= h
        num[idx] = (np.sum(dO * O.rope(a, pos, 4, 10000.0, 8)) - np.sum(dO * O.rope(b, pos, 4, 10000.0, 8))) / (2 * h)
    assert rel(an, num) < 1e-8


# ---------------------------------------------------------------------------
# Cross-entropy
# ---------------------------------------------------------------------------

def test_ce_matches_torch():
    R = rng(61)
    L = R.standard_normal((9, 40)) * 4
    y = R.integers(0, 40, 9)
    o = O.ce_fwd(L, y)
    tl = t64(L, True)
    ref = F.cross_entropy(tl, torch.tensor(y), reduction="none")
    assert rel(o["loss_row"], ref.detach().numpy()) < 1e-14
    assert rel(o["lse"], torch.logsumexp(t64(L), dim=1).numpy()) < 1e-15
    F.cross_entropy(tl, torch.tensor(y), reduction="mean").backward()
    assert rel(O.ce_bwd(L, y, o["lse"], 1.0 / 9), tl.grad.numpy()) < 1e-13
    assert abs(o["loss_mean"] - float(F.cross_entropy(t64(L), torch.tensor(y)))) < 1e-13


def test_ce_closed_forms_and_invariants():
    M, V = 6, 50
    y = np.arange(M) * 7 % V
    o = O.ce_fwd(np.zeros((M, V)), y)
    assert np.allclose(o["loss_row"], math.log(V), atol=0, rtol=1e-15)
    dl = O.ce_bwd(np.zeros((M, V)), y, o["lse"], 1.0 / M)
    exp = np.full((M, V), 1.0 / (M * V))
    exp[np.arange(M), y] -= 1.0 / M
    assert rel(dl, exp) < 1e-14
    R = rng(62)
    L = R.standard_normal((M, V)) * 3
    o1 = O.ce_fwd(L, y)
    o2 = O.ce_fwd(L + 11.5, y)
    assert rel(o2["lse"], o1["lse"] + 11.5) < 1e-14
    assert rel(o2["loss_row"], o1["loss_row"]) < 1e-12
    assert np.max(np.abs(np.sum(O.ce_bwd(L, y, o1["lse"], 0.3), axis=1))) < 1e-15


def test_ce_combine_tile_partials():
    """Per-tile (max, sum exp) states combine to the row LSE for any tiling."""
    R = rng(63)
    L = R.standard_normal((5, 37)) * 6
    for tile in (1, 4, 16, 37):
        pm = np.stack([L[:, c:c + tile].max(axis=1) for c in range(0, 37, tile)], axis=1)
        ps = np.stack([np.exp(L[:, c:c + tile] - pm[:, [k]]).sum(axis=1)
                       for k, c in enumerate(range(0, 37, tile))], axis=1)
        assert rel(O.ce_combine(pm, ps), torch.logsumexp(t64(L), 1).numpy()) < 1e-14


def test_ce_argmax_lowest_index_ties():
    L = np.array([[1.0, 3.0, 3.0, 0.0], [2.0, 2.0, 2.0, 2.0]])
    assert list(O.ce_fwd(L, [0, 0])["argmax"]) == [1, 0]


def test_gemm_ce_bwd_matches_autograd():
    R = rng(64)
    H = R.standard_normal((5, 6))
    W = R.standard_normal((6, 11))
    y = R.integers(0, 11, 5)
    tH, tW = t64(H, True), t64(W, True)
    F.cross_entropy(tH @ tW, torch.tensor(y)).backward()
    f = O.gemm_ce_fwd(H, W, y)
    b = O.gemm_ce_bwd(H, W, y, f["lse"], 1.0 / 5)
    assert rel(b["dH"], tH.grad.numpy()) < 1e-13
    assert rel(b["dW"], tW.grad.numpy()) < 1e-13


# ---------------------------------------------------------------------------
# Brute force: scalar loops from the definitions, tiny shapes
# ---------------------------------------------------------------------------

def _loop_mm(A, B):
    M, K = A.shape
    N = B.shape[1]
    C = np.zeros((M, N))
    for i, j in itertools.product(range(M), range(N)):
        acc = 0.0
        for k in range(K):
            acc += A[i, k] * B[k, j]
        C[i, j] = acc
    return C


def test_brute_force_all_ops():
    R = rng(71)
    M, K, d, N2 = 4, 5, 6, 3
    x, W0, z = R.standard_normal((M, K)), R.standard_normal((K, d)), R.standard_normal((M, d))
    g, W1 = R.standard_normal(d), R.standard_normal((d, N2))
    eps = 1e-3
    h1 = _loop_mm(x, W0) + z
    r = np.array([1 / math.sqrt(sum(h1[i, j] ** 2 for j in range(d)) / d + eps) for i in range(M)])
    h2 = np.array([[h1[i, j] * g[j] for j in range(d)] for i in range(M)])
    Y = np.array([[r[i] * sum(h2[i, k] * W1[k, j] for k in range(d)) for j in range(N2)] for i in range(M)])
    p = O.res_rmsprep(x, W0, z, g)
    assert rel(p["h1"], h1) < 1e-14 and rel(p["h2"], h2) < 1e-14
    assert rel(p["sumsq"], [sum(h1[i] ** 2) for i in range(M)]) < 1e-14
    assert rel(O.rowscale(h2, W1, r), Y) < 1e-14
    assert rel(O.gemm_rms_gemm_fwd(x, W0, z, g, W1, eps)["Y"], Y) < 1e-13

    dY = R.standard_normal((M, N2))
    s = np.array([sum(dY[i, j] * Y[i, j] for j in range(N2)) / d for i in range(M)])
    assert rel(O.rowdot_stat(dY, Y, d), s) < 1e-14
    G = _loop_mm(dY, W1.T)
    dh1 = np.array([[r[i] * g[j] * G[i, j] - r[i] ** 2 * s[i] * h1[i, j] for j in range(d)] for i in range(M)])
    dg = np.array([sum(r[i] * G[i, j] * h1[i, j] for i in range(M)) for j in range(d)])
    b = O.gemm_rmsnorm_bwd(dY, W1, h1, g, r, s)
    assert rel(b["dh1"], dh1) < 1e-13 and rel(b["dgamma"], dg) < 1e-13

    GU = R.standard_normal((M, 8))
    A = np.array([[GU[i, 2 * f] / (1 + math.exp(-GU[i, 2 * f])) * GU[i, 2 * f + 1] for f in range(4)]
                  for i in range(M)])
    assert rel(O.swiglu(GU), A) < 1e-14

    P = R.standard_normal((M, 8))
    pos = [0, 3, 7, 12]
    hd, th = 4, 500.0
    ref = P.copy()
    for i in range(M):
        for c in range(0, 8, 2):
            a = pos[i] * th ** (-2.0 * ((c % hd) // 2) / hd)
            ref[i, c] = P[i, c] * math.cos(a) - P[i, c + 1] * math.sin(a)
            ref[i, c + 1] = P[i, c] * math.sin(a) + P[i, c + 1] * math.cos(a)
    assert rel(O.rope(P, pos, hd, th, 8), ref) < 1e-14

    L = R.standard_normal((M, 9)) * 3
    y = [1, 8, 0, 4]
    lse = [math.log(sum(math.exp(v) for v in L[i])) for i in range(M)]
    o = O.ce_fwd(L, y)
    assert rel(o["lse"], lse) < 1e-14
    assert rel(o["loss_row"], [lse[i] - L[i, y[i]] for i in range(M)]) < 1e-14


# ---------------------------------------------------------------------------
# Hand-derived golden values
# ---------------------------------------------------------------------------

def _ev(v):
    if isinstance(v, str):
        return eval(v, {"math": math})  # noqa: S307 - trusted fixture in this repo
    if isinstance(v, list):
        return [_ev(u) for u in v]
    return v


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_golden_hand_values(case):
    inp = {k: (np.array(_ev(v)) if isinstance(v, list) else v) for k, v in case["inputs"].items()}
    exp = {k: np.array(_ev(v)) for k, v in case["expect"].items()}
    op = case["op"]
    if op == "rmsnorm":
        n, r = O.rmsnorm(inp["h1"], inp["gamma"], inp["eps"])
        got = dict(n=n, r=r)
    elif op == "rmsnorm_bwd":
        got = O.rmsnorm_bwd(inp["G"], inp["h1"], inp["gamma"], inp["r"], inp["s"])
    elif op == "swiglu":
        got = dict(A=O.swiglu(inp["GU"]))
    elif op == "swiglu_bwd":
        got = dict(dGU=O.swiglu_bwd(inp["dA"], inp["GU"]))
    elif op == "rope":
        got = dict(out=O.rope(inp["P"], inp["positions"], inp["head_dim"], inp["theta"], inp["rope_cols"]))
    elif op == "ce_fwd":
        got = O.ce_fwd(inp["logits"], inp["labels"])
    elif op == "ce_bwd":
        got = dict(dl=O.ce_bwd(inp["logits"], inp["labels"], inp["lse"], inp["grad_scale"]))
    elif op == "e4m3":
        got = dict(value=O.e4m3(np.asarray(inp["bits"], np.uint8)))
    else:
        raise AssertionError(op)
    for k, v in exp.items():
        if k == "argmax":
            assert list(got[k]) == list(v)
        else:
            assert np.max(np.abs(np.asarray(got[k], np.float64) - v)) < 1e-14, k


# ---------------------------------------------------------------------------
# The input generator (shared with the CUDA side) is deterministic and RNE
# ---------------------------------------------------------------------------

def test_inputs_bf16_rounding_and_determinism():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.00390625 + 2 ** -20], np.float32)
    got = O.bf16(gen.f32_to_bf16_bits(v))
    # 1 + 2^-8 is a tie -> even (1.0); 1 + 3*2^-8 is a tie -> even (1 + 2^-6)
    assert list(got[:4]) == [1.0, 1.0, 1.0 + 2 ** -6, -2.5]
    assert got[4] == 1.0078125
    a = gen.rms_chain(8, 16, 16, 8, bwd_K=4)
    b = gen.rms_chain(8, 16, 16, 8)
    for k in b:
        assert np.array_equal(a[k], b[k])
    x = O.bf16(gen.rms_chain(512, 64, 64, 8)["x"])
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02


def test_outlier_channel_inputs():
    """The outlier-channel stand-in: the same x, W0, gamma, W1 as rms_chain,
    and a z whose chosen channels are 20 times wider than the rest."""
    p = gen.rms_chain_outliers(2048, 32, 400, 16, seed=1, frac=0.01, scale=20.0)
    q = gen.rms_chain(2048, 32, 400, 16, seed=1)
    for k in ("x", "W0", "gamma", "W1"):
        assert np.array_equal(p[k], q[k])
    cols = p["outlier_cols"]
    assert len(cols) == 4 and len(set(cols.tolist())) == 4
    z = O.bf16(p["z"])
    rest = np.setdiff1d(np.arange(400), cols)
    assert abs(z[:, rest].std() - 1) < 0.02
    assert abs(z[:, cols].std() / 20 - 1) < 0.05
    again = gen.rms_chain_outliers(2048, 32, 400, 16, seed=1, frac=0.01, scale=20.0)
    assert np.array_equal(again["z"], p["z"])


# ---------------------------------------------------------------------------
# Block-level chain: one period of two GEMM-residual-RMSNorm-GEMM structures
# (RoPE path, then SwiGLU path). The plain definition is pinned to a torch
# float64 restatement (library rms_norm and silu, RoPE as a complex product)
# and to autograd and finite differences of the scalar
#   L = <dQKV, QKV> + <gh, A Wdn + h2>;
# the reparameterised, kernel-by-kernel composition is then pinned to it.
# ---------------------------------------------------------------------------

BLK = dict(M=6, d=16, F=12, hd=8, rope_cols=32, theta=10000.0, eps=1e-6)


def _block(seed=81, **kw):
    c = dict(BLK, **kw)
    R = rng(seed)
    M, d, F = c["M"], c["d"], c["F"]
    t = dict(
        P=R.standard_normal((M, F)), Wd=R.standard_normal((F, d)) / np.sqrt(F), x=R.standard_normal((M, d)),
        gamma1=1 + 0.1 * R.standard_normal(d), Wqkv=R.standard_normal((d, 3 * d)) / np.sqrt(d),
        O=R.standard_normal((M, d)), Wo=R.standard_normal((d, d)) / np.sqrt(d),
        gamma2=1 + 0.1 * R.standard_normal(d), Wgu=R.standard_normal((d, 2 * F)) / np.sqrt(d),
    )
    g = dict(dQKV=R.standard_normal((M, 3 * d)), gh=R.standard_normal((M, d)),
             Wdn=R.standard_normal((F, d)) / np.sqrt(F))
    pos = np.array([0, 1, 5, 17, 4095, 300])[:M]
    return c, t, g, pos


def _fwd_args(c, t, pos):
    return (t["P"], t["Wd"], t["x"], t["gamma1"], t["Wqkv"], t["O"], t["Wo"], t["gamma2"], t["Wgu"], pos,
            c["hd"], c["theta"], c["rope_cols"], c["eps"])


def _torch_block(c, T, pos):
    """Torch float64 restatement: rms_norm and silu from the library, the
    rotation as multiplication by exp(i angle) on complex pairs."""
    d = T["x"].shape[1]

    def rope_t(Y):
        hd, rc = c["hd"], c["rope_cols"]
        i = torch.arange(hd // 2, dtype=torch.float64)
        ang = torch.tensor(pos, dtype=torch.float64)[:, None] * c["theta"] ** (-2.0 * i / hd)[None, :]
        rot = torch.polar(torch.ones_like(ang), ang)                      # [M, hd/2]
        q = Y[:, :rc].reshape(Y.shape[0], rc // hd, hd // 2, 2)
        z = torch.view_as_complex(q.contiguous()) * rot[:, None, :]
        return torch.cat([torch.view_as_real(z).reshape(Y.shape[0], rc), Y[:, rc:]], dim=1)

    h1 = T["P"] @ T["Wd"] + T["x"]
    n1 = F.rms_norm(h1, (d,), T["gamma1"], c["eps"])
    QKV = rope_t(n1 @ T["Wqkv"])
    h2 = T["O"] @ T["Wo"] + h1
    n2 = F.rms_norm(h2, (d,), T["gamma2"], c["eps"])
    GU = n2 @ T["Wgu"]
    A = F.silu(GU[:, 0::2]) * GU[:, 1::2]
    return QKV, h2, A


def test_block_fwd_matches_torch():
    c, t, _, pos = _block()
    f = O.block_fwd(*_fwd_args(c, t, pos))
    QKV, h2, A = _torch_block(c, {k: t64(v) for k, v in t.items()}, pos)
    assert rel(f["QKV"], QKV.numpy()) < 1e-13
    assert rel(f["h2"], h2.numpy()) < 1e-13
    assert rel(f["A"], A.numpy()) < 1e-13
    assert np.array_equal(f["QKV"][:, c["rope_cols"]:], f["Yq"][:, c["rope_cols"]:])  # V passes through


def test_block_bwd_matches_autograd():
    c, t, g, pos = _block()
    b = O.block_bwd(*_fwd_args(c, t, pos), g["dQKV"], g["gh"], g["Wdn"])
    T = {k: t64(v, grad=True) for k, v in t.items()}
    QKV, h2, A = _torch_block(c, T, pos)
    L = torch.sum(t64(g["dQKV"]) * QKV) + torch.sum(t64(g["gh"]) * (A @ t64(g["Wdn"]) + h2))
    L.backward()
    for ours, theirs in [("dP", "P"), ("dx", "x"), ("dO", "O"), ("dWd", "Wd"), ("dgamma1", "gamma1"),
                         ("dWqkv", "Wqkv"), ("dWo", "Wo"), ("dgamma2", "gamma2"), ("dWgu", "Wgu")]:
        assert rel(b[ours], T[theirs].grad.numpy()) < 1e-12, ours


def test_block_bwd_finite_differences():
    c, t, g, pos = _block(seed=82, M=3, d=8, F=6, hd=8, rope_cols=16)

    def loss(tt):
        f = O.block_fwd(*_fwd_args(c, tt, pos))
        return np.sum(g["dQKV"] * f["QKV"]) + np.sum(g["gh"] * (O.matmul(f["A"], g["Wdn"]) + f["h2"]))

    b = O.block_bwd(*_fwd_args(c, t, pos), g["dQKV"], g["gh"], g["Wdn"])
    h = 1e-6
    for name, grad in [("gamma1", "dgamma1"), ("gamma2", "dgamma2"), ("x", "dx"), ("Wd", "dWd"), ("O", "dO")]:
        num = np.zeros_like(t[name])
        for idx in np.ndindex(t[name].shape):
            a = {k: v.copy() for k, v in t.items()}
            m = {k: v.copy() for k, v in t.items()}
            a[name][idx] += h
            m[name][idx] -= h
            num[idx] = (loss(a) - loss(m)) / (2 * h)
        assert rel(b[grad], num) < 1e-7, name


def test_block_fused_composition_equals_definition():
    c, t, g, pos = _block(seed=83)
    args = _fwd_args(c, t, pos)
    f = O.block_fwd(*args)
    ff = O.block_fwd_fused(*args)
    for k in ("h1", "h1g", "r1", "QKV", "h2", "h2g", "r2", "GU", "A"):
        assert rel(ff[k], f[k]) < 1e-13, k
    b = O.block_bwd(*args, g["dQKV"], g["gh"], g["Wdn"])
    bf = O.block_bwd_fused(ff, t["P"], t["Wqkv"], t["O"], t["Wo"], t["gamma1"], t["gamma2"], t["Wgu"], pos,
                           c["hd"], c["theta"], c["rope_cols"], g["dQKV"], g["gh"], g["Wdn"])
    for k in ("dh2", "dgamma2", "dWgu", "dO", "dWo", "dh1", "dgamma1", "dWqkv", "dWd"):
        assert rel(bf[k], b[k]) < 1e-12, k
    # the row statistics are the textbook (1/d) rowsum(dn (.) gamma (.) h) scaled by r
    d = c["d"]
    assert rel(bf["s2"], f["r2"] * np.sum(b["dn2"] * t["gamma2"] * f["h2"], axis=1) / d) < 1e-12
    assert rel(bf["s1"], f["r1"] * np.sum(b["dn1"] * t["gamma1"] * f["h1"], axis=1) / d) < 1e-12


def test_block_kernel_pieces():
    c, t, g, pos = _block(seed=84)
    R = rng(85)
    M, d = c["M"], c["d"]
    X = R.standard_normal((M, d))
    r = 0.5 + R.random(M)
    # rowscale commutes with the rotation and feeds the SwiGLU pair map unchanged
    q = O.gemm_rowscale_rope(X, t["Wqkv"], r, pos, c["hd"], c["theta"], c["rope_cols"])
    assert rel(q, r[:, None] * O.gemm_rope(X, t["Wqkv"], pos, c["hd"], c["theta"], c["rope_cols"])) < 1e-13
    s = O.gemm_rowscale_swiglu(X, t["Wgu"], r)
    assert rel(s["GU"], r[:, None] * (X @ t["Wgu"])) < 1e-13
    assert rel(s["A"], O.swiglu(s["GU"])) == 0.0
    # the RoPE glue's statistic is rotation invariant: it equals (1/d) rowsum(dQKV (.) QKV)
    QKV = R.standard_normal((M, 3 * d))
    gl = O.rope_bwd_rowdot(g["dQKV"], QKV, r, pos, c["hd"], c["theta"], c["rope_cols"], d)
    assert rel(gl["s"], np.sum(g["dQKV"] * QKV, axis=1) / d) < 1e-13
    assert rel(gl["dYqr"], r[:, None] * O.rope_bwd(g["dQKV"], pos, c["hd"], c["theta"], c["rope_cols"])) < 1e-14
    # the residual gradient is additive; with dres = 0 it is the plain RMSNorm-backward GEMM on dYr / r
    dYr = R.standard_normal((M, 2 * c["F"]))
    h = R.standard_normal((M, d))
    sv = R.standard_normal(M)
    dres = R.standard_normal((M, d))
    a = O.gemm_rmsnorm_bwd_res(dYr, t["Wgu"], h, t["gamma2"], r, sv, dres)
    z = O.gemm_rmsnorm_bwd_res(dYr, t["Wgu"], h, t["gamma2"], r, sv, np.zeros_like(dres))
    p = O.gemm_rmsnorm_bwd(dYr / r[:, None], t["Wgu"], h, t["gamma2"], r, sv)
    assert rel(a["dh"] - dres, z["dh"]) < 1e-13
    assert rel(z["dh"], p["dh1"]) < 1e-13 and rel(z["dgamma"], p["dgamma"]) < 1e-13
    # SwiGLU-backward GEMM with the row statistic: s over the 2F pre-activation columns, over d
    sb = O.gemm_swiglu_bwd_rowdot(g["gh"], g["Wdn"], s["GU"], r, d)
    assert rel(sb["dGU"], O.gemm_swiglu_bwd(g["gh"], g["Wdn"], s["GU"])["dGU"]) < 1e-14
    assert rel(sb["s"], np.sum(sb["dGU"] * s["GU"], axis=1) / d) < 1e-14


def test_block_inputs_generator():
    a = gen.block_problem(8, 16, 24, seed=3)
    b = gen.block_problem(8, 16, 24, seed=3, with_bwd=False)
    assert set(a) - set(b) == {"dQKV", "gh", "Wdn"}
    for k in b:
        assert np.array_equal(a[k], b[k])
    shapes = dict(P=(8, 24), Wd=(24, 16), x=(8, 16), gamma1=(16,), Wqkv=(16, 48), O=(8, 16), Wo=(16, 16),
                  gamma2=(16,), Wgu=(16, 48), dQKV=(8, 48), gh=(8, 16), Wdn=(24, 16))
    assert {k: v.shape for k, v in a.items()} == shapes
    w = O.bf16(gen.block_problem(64, 256, 512, with_bwd=False)["Wgu"])
    assert abs(w.std() * 16 - 1) < 0.02



# ---------------------------------------------------------------------------
# FP8 E4M3: the oracle's decoder and the input generator's encoder
# ---------------------------------------------------------------------------

def test_e4m3_decoder_matches_torch_float8():
    """All 256 bit patterns against torch's float8_e4m3fn (a library decoder)."""
    b = np.arange(256, dtype=np.uint8)
    mine = O.e4m3(b)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.isnan(mine).sum() == 2  # 0x7F and 0xFF
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))
    # monotone over the positive finite codes, largest 448
    pos = mine[:0x7F]
    assert np.all(np.diff(pos) > 0) and pos[-1] == 448.0


def test_e4m3_encoder_rne_and_saturation():
    R = rng(91)
    x = (R.standard_normal(200000) * np.exp(R.uniform(-8, 6, 200000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    ties = np.float32([1.0625, 1.1875, 3 * 2.0 ** -10, 5 * 2.0 ** -10, -9.0, 2.0 ** -6 - 2.0 ** -10, 0.0])
    x = np.concatenate([x, ties])
    enc = gen.f32_to_e4m3_bits(x)
    assert np.array_equal(enc, torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    # round trip of every finite code is exact
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    assert np.array_equal(gen.f32_to_e4m3_bits(O.e4m3(codes).astype(np.float32)) & 0x7F, codes & 0x7F)
    # saturation instead of NaN above 448
    assert list(gen.f32_to_e4m3_bits(np.float32([500.0, -1e6, 464.0]))) == [0x7E, 0xFE, 0x7E]


def test_fp8_problem_scales_and_determinism():
    a = gen.fp8_problem(64, 256, 48, seed=2, labels=True)
    b = gen.fp8_problem(64, 256, 48, seed=2)
    assert np.array_equal(a["A"], b["A"]) and np.array_equal(a["B"], b["B"])
    assert a["B"].shape == (48, 256) and a["sB"] == 1.0 / 16.0
    w = O.e4m3(gen.fp8_problem(8, 4096, 512)["B"]) / 64.0
    assert abs(w.std() * 64 - 1) < 0.02
