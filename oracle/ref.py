"""Plain float64 definitions of every operator on the CODA hot path.

See the package docstring for the citation short forms ("CODA note",
"pith page"). No blocking, fusion or reordering beyond what each definition
states; ``A @ B`` (a float64 BLAS matmul) is the only library primitive used.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16",
    "e4m3",
    "matmul",
    # GEMM-RMSNorm-GEMM forward
    "rms_scale",
    "rmsnorm",
    "gemm_rms_gemm_fwd",
    "res_rmsprep",
    "rms_reduce",
    "rowscale",
    # GEMM-RMSNorm-GEMM backward
    "rowdot_stat",
    "gemm_rowdot",
    "rmsnorm_bwd",
    "gemm_rmsnorm_bwd",
    "gemm_rms_gemm_bwd",
    # SwiGLU
    "silu",
    "sigmoid",
    "swiglu",
    "swiglu_bwd",
    "gemm_swiglu",
    "gemm_swiglu_bwd",
    # RoPE
    "rope_angles",
    "rope",
    "rope_bwd",
    "gemm_rope",
    "gemm_rope_bwd",
    # Cross-entropy
    "logsumexp_rows",
    "ce_fwd",
    "ce_combine",
    "ce_bwd",
    "gemm_ce_fwd",
    "gemm_ce_bwd",
    # Block-level chain
    "rmsnorm_bwd_textbook",
    "gemm_rowscale_rope",
    "gemm_rowscale_swiglu",
    "gemm_swiglu_bwd_rowdot",
    "gemm_rmsnorm_bwd_res",
    "rope_bwd_rowdot",
    "block_fwd",
    "block_bwd",
    "block_fwd_fused",
    "block_bwd_fused",
]


# ----------------------------------------------------------------------------
# Encoding and the contraction
# ----------------------------------------------------------------------------

def bf16(bits) -> np.ndarray:
    """Decode bfloat16 bit patterns (uint16) to float64: the 16 bits are the
    high half of an IEEE binary32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e4m3(bits) -> np.ndarray:
    """Decode FP8 E4M3 bit patterns to float64: sign bit 7, exponent bits 6..3
    with bias 7, mantissa bits 2..0. Exponent field 0 is subnormal,
    (-1)^s 2^-6 (m/8); otherwise (-1)^s 2^(e-7) (1 + m/8). There are no
    infinities; exponent 15 with mantissa 7 is NaN, so the largest finite
    magnitude is 2^8 * 1.75 = 448."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sgn = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (b & 0x7 == 7), np.nan, mag)
    return sgn * mag


def matmul(A, B) -> np.ndarray:
    """Dense float64 product ``A @ B`` (the GEMM mainloop's definition)."""
    return np.asarray(A, dtype=np.float64) @ np.asarray(B, dtype=np.float64)


# ----------------------------------------------------------------------------
# GEMM -> residual -> RMSNorm -> GEMM, forward
# CODA note, Key design 1: y = RMSNorm(x W0 + z, gamma) W1, with
# r = 1 / rms(x W0 + z) a per-row scalar; RMSNorm(h, gamma) = r * h (.) gamma.
# ----------------------------------------------------------------------------

def rms_scale(h1, eps: float) -> np.ndarray:
    """Per-row inverse RMS ``r_i = 1 / sqrt(mean_j h1[i,j]^2 + eps)``.

    eps sits inside the square root (pith page, Figure 5 caption:
    r = 1/sqrt(reduce(r_hat) + eps)); the mean is over the normalised width d.
    """
    h1 = np.asarray(h1, dtype=np.float64)
    return 1.0 / np.sqrt(np.mean(h1 * h1, axis=1) + eps)


def rmsnorm(h1, gamma, eps: float):
    """Textbook RMSNorm: ``n = r[:,None] * h1 * gamma[None,:]``; returns (n, r)."""
    r = rms_scale(h1, eps)
    return (r[:, None] * np.asarray(h1, np.float64)) * np.asarray(gamma, np.float64)[None, :], r


def gemm_rms_gemm_fwd(x, W0, z, gamma, W1, eps: float) -> dict:
    """Unfused definition of the GEMM-RMSNorm-GEMM block (CODA note, Key design 1).

    h0 = x W0; h1 = h0 + z (residual stream); n = RMSNorm(h1, gamma);
    Y = n W1. Also reports the reparameterised intermediates the fused kernels
    emit: h2 = h1 (.) gamma and h3 = h2 W1 (so that Y = r (.)row h3).
    """
    h0 = matmul(x, W0)
    h1 = h0 + np.asarray(z, np.float64)
    n, r = rmsnorm(h1, gamma, eps)
    Y = matmul(n, W1)
    h2 = h1 * np.asarray(gamma, np.float64)[None, :]
    h3 = matmul(h2, W1)
    return dict(h0=h0, h1=h1, h2=h2, n=n, r=r, h3=h3, Y=Y)


def res_rmsprep(x, W0, z, gamma) -> dict:
    """First GEMM of the reparameterised block and its epilogue
    (CODA note, Key design 1: h1 = h0 + z, h2 = h1 (.) gamma, and the per-row
    sum of squares of the *unscaled* h1 that feeds r).

    Returns h1, h2 and ``sumsq[i] = sum_j h1[i,j]^2`` over all columns; a
    tile-partial of it is the same sum restricted to that tile's columns.
    """
    h1 = matmul(x, W0) + np.asarray(z, np.float64)
    h2 = h1 * np.asarray(gamma, np.float64)[None, :]
    return dict(h1=h1, h2=h2, sumsq=np.sum(h1 * h1, axis=1))


def rms_reduce(partials, d: int, eps: float) -> np.ndarray:
    """Auxiliary reduction of tile partial sums of squares (pith page,
    Figure 4 and Figure 5 captions): ``r_i = 1/sqrt(sum_nb P[i,nb] / d + eps)``.

    The partials are per-(row, column tile) sums of h1^2; dividing the total by
    the normalised width d gives the row mean.
    """
    P = np.asarray(partials, dtype=np.float64)
    return 1.0 / np.sqrt(np.sum(P, axis=1) / d + eps)


def rowscale(h2, W1, r) -> np.ndarray:
    """Second GEMM with the delayed row scale (CODA note, Key design 1):
    ``Y[i,j] = r[i] * (h2 W1)[i,j]``."""
    return np.asarray(r, np.float64)[:, None] * matmul(h2, W1)


# ----------------------------------------------------------------------------
# GEMM-RMSNorm-GEMM, backward
# CODA note, Key design 3: the RMSNorm-backward row statistic
# s = (1/d) rowsum(dL/dh2 (.) h2) equals (1/d) rowsum(dL/dy (.) y) and can be
# formed in the epilogue of the GEMM that produces dL/dy.
# ----------------------------------------------------------------------------

def rowdot_stat(dY, Y, d: int) -> np.ndarray:
    """``s_i = (1/d) * sum_j dY[i,j] * Y[i,j]`` (CODA note, Key design 3)."""
    return np.sum(np.asarray(dY, np.float64) * np.asarray(Y, np.float64), axis=1) / d


def gemm_rowdot(dO, Wn, Y, r, d: int) -> dict:
    """The GEMM that produces the output gradient, with the row statistic in its
    epilogue: dY = dO Wn; s = (1/d) rowsum(dY (.) Y); dYr = r (.)row dY (the
    row-scaled gradient that the weight gradient of the second GEMM needs).
    """
    dY = matmul(dO, Wn)
    return dict(dY=dY, dYr=np.asarray(r, np.float64)[:, None] * dY, s=rowdot_stat(dY, Y, d))


def rmsnorm_bwd(G, h1, gamma, r, s) -> dict:
    """RMSNorm backward through n = r h1 (.) gamma given G = dL/dn.

    Differentiating r = (mean(h1^2) + eps)^(-1/2) gives
    dh1 = r gamma (.) G - r^3 h1 (1/d) rowsum(G (.) gamma (.) h1). With
    rowsum(G (.) h2) = rowsum(dY (.) Y) / r (CODA note, Key design 3) and
    s = (1/d) rowsum(dY (.) Y), this is ``dh1 = r gamma (.) G - r^2 s h1``.
    Also ``dgamma_j = sum_i r_i G[i,j] h1[i,j]``.
    """
    G = np.asarray(G, np.float64)
    h1 = np.asarray(h1, np.float64)
    gamma = np.asarray(gamma, np.float64)
    r = np.asarray(r, np.float64)
    s = np.asarray(s, np.float64)
    dh1 = r[:, None] * gamma[None, :] * G - (r * r * s)[:, None] * h1
    dgamma = np.sum(r[:, None] * G * h1, axis=0)
    return dict(dh1=dh1, dgamma=dgamma)


def gemm_rmsnorm_bwd(dY, W1, h1, gamma, r, s) -> dict:
    """Data-gradient GEMM of the second projection, G = dY W1^T, with the
    RMSNorm backward in its epilogue (the duality rule of CODA note,
    Key design 3: the backward tile rule attaches to the GEMM that produces
    the gradient)."""
    G = matmul(dY, np.asarray(W1, np.float64).T)
    out = rmsnorm_bwd(G, h1, gamma, r, s)
    out["G"] = G
    return out


def gemm_rms_gemm_bwd(x, W0, z, gamma, W1, eps: float, dY) -> dict:
    """Full backward of Y = RMSNorm(x W0 + z, gamma) W1 for upstream dY.

    Returns dx, dW0, dz, dgamma, dW1 and the intermediates (s, G, dh1, dYr).
    """
    f = gemm_rms_gemm_fwd(x, W0, z, gamma, W1, eps)
    d = f["h1"].shape[1]
    dY = np.asarray(dY, np.float64)
    s = rowdot_stat(dY, f["Y"], d)
    b = gemm_rmsnorm_bwd(dY, W1, f["h1"], gamma, f["r"], s)
    dYr = f["r"][:, None] * dY
    dW1 = matmul(f["h2"].T, dYr)
    dh1 = b["dh1"]
    return dict(
        s=s, G=b["G"], dh1=dh1, dz=dh1, dgamma=b["dgamma"], dYr=dYr, dW1=dW1,
        dx=matmul(dh1, np.asarray(W0, np.float64).T),
        dW0=matmul(np.asarray(x, np.float64).T, dh1),
    )


# ----------------------------------------------------------------------------
# SwiGLU pair map (CODA note, Key design 2; pith page, Figure 7 caption):
# even channel = gate G, odd channel = up U; output silu(G) (.) U.
# ----------------------------------------------------------------------------

def sigmoid(g) -> np.ndarray:
    g = np.asarray(g, np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-g))


def silu(g) -> np.ndarray:
    """``silu(g) = g * sigmoid(g)``."""
    g = np.asarray(g, np.float64)
    return g * sigmoid(g)


def swiglu(GU) -> np.ndarray:
    """``A[:, f] = silu(GU[:, 2f]) * GU[:, 2f+1]`` (adjacent gate/up pairs)."""
    GU = np.asarray(GU, np.float64)
    return silu(GU[:, 0::2]) * GU[:, 1::2]


def swiglu_bwd(dA, GU) -> np.ndarray:
    """Pair map backward: one incoming gradient dA gives both paired input
    gradients, packed back in the interleaved layout (pith page, Figure 7).

    dG = dA * U * sigma(G) * (1 + G (1 - sigma(G)));  dU = dA * silu(G).
    """
    GU = np.asarray(GU, np.float64)
    dA = np.asarray(dA, np.float64)
    G = GU[:, 0::2]
    U = GU[:, 1::2]
    sg = sigmoid(G)
    out = np.empty_like(GU)
    out[:, 0::2] = dA * U * sg * (1.0 + G * (1.0 - sg))
    out[:, 1::2] = dA * G * sg
    return out


def gemm_swiglu(X, Wgu) -> dict:
    """Up-projection GEMM with the SwiGLU pair map in its epilogue."""
    GU = matmul(X, Wgu)
    return dict(GU=GU, A=swiglu(GU))


def gemm_swiglu_bwd(dY, Wd, GU) -> dict:
    """Down-projection data-gradient GEMM dA = dY Wd^T (Wd stored [F, K]) with
    the SwiGLU backward in its epilogue, recomputing the gate from the saved
    pre-activation GU."""
    dA = matmul(dY, np.asarray(Wd, np.float64).T)
    return dict(dA=dA, dGU=swiglu_bwd(dA, GU))


# ----------------------------------------------------------------------------
# RoPE pair map (CODA note, Key design 2; pith page, Figure 7 caption): a 2-D
# rotation of adjacent channel pairs (2i, 2i+1) of each head, using
# pre-broadcast sin/cos vectors. Frequencies theta^(-2i/head_dim) (RoFormer).
# ----------------------------------------------------------------------------

def rope_angles(positions, head_dim: int, theta: float) -> np.ndarray:
    """``ang[p, i] = positions[p] * theta ** (-2 i / head_dim)``, i < head_dim/2."""
    pos = np.asarray(positions, np.float64)
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    return pos[:, None] * inv_freq[None, :]


def _rope_apply(P, positions, head_dim, theta, rope_cols, sign):
    P = np.array(P, dtype=np.float64, copy=True)
    ang = rope_angles(positions, head_dim, theta)            # [rows, hd/2]
    c, s = np.cos(ang), np.sin(ang)
    n_heads = rope_cols // head_dim
    for h in range(n_heads):
        base = h * head_dim
        e = P[:, base:base + head_dim:2].copy()
        o = P[:, base + 1:base + head_dim:2].copy()
        P[:, base:base + head_dim:2] = e * c - sign * o * s
        P[:, base + 1:base + head_dim:2] = sign * e * s + o * c
    return P


def rope(P, positions, head_dim: int, theta: float, rope_cols: int) -> np.ndarray:
    """Rotate pairs in columns [0, rope_cols) (the Q and K heads); columns at or
    beyond rope_cols (V) pass through.

    For pair i of a head at position p with angle a = p theta^(-2i/hd):
    o_e = a_e cos a - a_o sin a;  o_o = a_e sin a + a_o cos a.
    """
    return _rope_apply(P, positions, head_dim, theta, rope_cols, +1.0)


def rope_bwd(dO, positions, head_dim: int, theta: float, rope_cols: int) -> np.ndarray:
    """Transpose of the rotation (the backward of ``rope``):
    g_e = a_e cos + a_o sin;  g_o = -a_e sin + a_o cos."""
    return _rope_apply(dO, positions, head_dim, theta, rope_cols, -1.0)


def gemm_rope(X, W, positions, head_dim: int, theta: float, rope_cols: int) -> np.ndarray:
    """QKV projection with RoPE in the epilogue."""
    return rope(matmul(X, W), positions, head_dim, theta, rope_cols)


def gemm_rope_bwd(A, B, positions, head_dim: int, theta: float, rope_cols: int) -> np.ndarray:
    """A GEMM producing the gradient of the rotated output, with the transposed
    rotation in its epilogue (duality rule, CODA note, Key design 3)."""
    return rope_bwd(matmul(A, B), positions, head_dim, theta, rope_cols)


# ----------------------------------------------------------------------------
# Cross-entropy over the vocabulary (CODA note, Key design 4: a stateful
# transform keeps an online log-sum-exp across vocabulary tiles; partial
# statistics are combined by an auxiliary reduction).
# ----------------------------------------------------------------------------

def logsumexp_rows(L) -> np.ndarray:
    """``LSE_i = m_i + ln sum_j exp(L[i,j] - m_i)`` with ``m_i = max_j L[i,j]``."""
    L = np.asarray(L, np.float64)
    m = np.max(L, axis=1)
    return m + np.log(np.sum(np.exp(L - m[:, None]), axis=1))


def ce_fwd(logits, labels) -> dict:
    """Natural-log softmax cross-entropy, mean over rows:
    loss_i = LSE_i - logits[i, y_i]; loss = (1/M) sum_i loss_i.
    Also the row argmax (lowest index among equal maxima)."""
    L = np.asarray(logits, np.float64)
    y = np.asarray(labels, np.int64)
    lse = logsumexp_rows(L)
    tgt = L[np.arange(L.shape[0]), y]
    loss_row = lse - tgt
    return dict(lse=lse, tgt=tgt, loss_row=loss_row, loss_mean=float(np.mean(loss_row)) if len(y) else 0.0,
                argmax=np.argmax(L, axis=1) if L.shape[1] else np.zeros(0, np.int64))


def ce_combine(pmax, psum) -> np.ndarray:
    """Combine per-tile online-softmax states (m_t, sigma_t) of a row:
    ``LSE = Mx + ln sum_t sigma_t exp(m_t - Mx)`` with ``Mx = max_t m_t``."""
    pm = np.asarray(pmax, np.float64)
    ps = np.asarray(psum, np.float64)
    Mx = np.max(pm, axis=1)
    return Mx + np.log(np.sum(ps * np.exp(pm - Mx[:, None]), axis=1))


def ce_bwd(logits, labels, lse, grad_scale: float) -> np.ndarray:
    """``dl[i,j] = grad_scale * (exp(L[i,j] - LSE_i) - [j == y_i])``; for the mean
    loss with upstream gradient g, grad_scale = g / M."""
    L = np.asarray(logits, np.float64)
    P = np.exp(L - np.asarray(lse, np.float64)[:, None])
    P[np.arange(L.shape[0]), np.asarray(labels, np.int64)] -= 1.0
    return grad_scale * P


def gemm_ce_fwd(H, W, labels) -> dict:
    """LM-head GEMM with cross-entropy in the epilogue (logits never stored)."""
    out = ce_fwd(matmul(H, W), labels)
    return out


def gemm_ce_bwd(H, W, labels, lse, grad_scale: float) -> dict:
    """Backward of the LM-head cross-entropy: the logits are recomputed by the
    GEMM whose epilogue forms dl; dH = dl W^T and dW = H^T dl are plain GEMMs."""
    L = matmul(H, W)
    dl = ce_bwd(L, labels, lse, grad_scale)
    return dict(dl=dl, dH=matmul(dl, np.asarray(W, np.float64).T), dW=matmul(np.asarray(H, np.float64).T, dl))


# ----------------------------------------------------------------------------
# Block-level chain (CODA note, ablation on full Transformer blocks: two
# consecutive GEMM-Residual-RMSNorm-GEMM structures, one covering the RoPE
# path and one the SwiGLU path, with the light auxiliary reductions and glue).
#
# One period of a pre-norm layer stack, with the attention core left out (its
# output O is an input, and the gradient of the rotated QKV arrives as dQKV):
#   RoPE path:   h1 = P Wd + x;   n1 = RMSNorm(h1, gamma1);  QKV = RoPE(n1 Wqkv)
#   SwiGLU path: h2 = O Wo + h1;  n2 = RMSNorm(h2, gamma2);  GU = n2 Wgu;
#                A = SwiGLU(GU)
# The backward takes the gradient of the rotated QKV (dQKV) and of the next
# period's residual output h1' = A Wdn + h2 (gh), i.e. it differentiates
#   L = <dQKV, QKV> + <gh, A Wdn + h2>.
# ----------------------------------------------------------------------------

def rmsnorm_bwd_textbook(dn, u, gamma, r) -> dict:
    """Textbook RMSNorm backward through n = r u (.) gamma, r = (mean(u^2)+eps)^(-1/2):
    ``du = r gamma (.) dn - r^3 u (1/d) rowsum(dn (.) gamma (.) u)`` and
    ``dgamma_j = sum_i dn[i,j] r_i u[i,j]``."""
    dn = np.asarray(dn, np.float64)
    u = np.asarray(u, np.float64)
    gamma = np.asarray(gamma, np.float64)
    r = np.asarray(r, np.float64)
    d = u.shape[1]
    c = np.sum(dn * gamma[None, :] * u, axis=1) / d
    du = r[:, None] * gamma[None, :] * dn - (r ** 3 * c)[:, None] * u
    return dict(du=du, dgamma=np.sum(dn * r[:, None] * u, axis=0))


def gemm_rowscale_rope(X, W, r, positions, head_dim: int, theta: float, rope_cols: int) -> np.ndarray:
    """Second GEMM of the RoPE-path structure: the delayed row scale and the
    rotation in one epilogue, ``QKV = RoPE(r (.)row (X W))`` (CODA note, Key
    designs 1 and 2; r commutes with the right multiply and with the
    rotation, which is linear per row)."""
    return rope(rowscale(X, W, r), positions, head_dim, theta, rope_cols)


def gemm_rowscale_swiglu(X, Wgu, r) -> dict:
    """Second GEMM of the SwiGLU-path structure: ``GU = r (.)row (X Wgu)``,
    ``A = SwiGLU(GU)`` (the scale precedes the nonlinearity)."""
    GU = rowscale(X, Wgu, r)
    return dict(GU=GU, A=swiglu(GU))


def gemm_swiglu_bwd_rowdot(dY, Wd, GU, r, d: int) -> dict:
    """SwiGLU-backward GEMM of the chain, with the RMSNorm-backward row
    statistic in the same epilogue (CODA note, Key design 3: s is formed in
    the GEMM that produces the gradient of the rowscale GEMM's output GU):
    dA = dY Wd^T; dGU = swiglu_bwd(dA, GU); s = (1/d) rowsum(dGU (.) GU);
    dGUr = r (.)row dGU."""
    dA = matmul(dY, np.asarray(Wd, np.float64).T)
    dGU = swiglu_bwd(dA, GU)
    return dict(dA=dA, dGU=dGU, dGUr=np.asarray(r, np.float64)[:, None] * dGU, s=rowdot_stat(dGU, GU, d))


def gemm_rmsnorm_bwd_res(dYr, W1, h, gamma, r, s, dres) -> dict:
    """RMSNorm backward in the data-gradient GEMM, fed with the row-scaled
    gradient: ``Gr = dYr W1^T = r (.)row G``, so ``dh = gamma (.) Gr -
    r^2 s h + dres`` (the r^2 form of ``rmsnorm_bwd`` with G = Gr / r) where
    dres is the gradient reaching h through the residual connection, and
    ``dgamma_j = sum_i Gr[i,j] h[i,j]``."""
    Gr = matmul(dYr, np.asarray(W1, np.float64).T)
    r = np.asarray(r, np.float64)
    b = rmsnorm_bwd(Gr / r[:, None], h, gamma, r, s)
    return dict(Gr=Gr, dh=b["dh1"] + np.asarray(dres, np.float64), dgamma=b["dgamma"])


def rope_bwd_rowdot(dQKV, QKV, r, positions, head_dim: int, theta: float, rope_cols: int, d: int) -> dict:
    """Glue of the RoPE-path backward, on the gradient the attention backward
    delivers: dYq = RoPE^T(dQKV) (the gradient of the unrotated QKV
    projection Yq), the row statistic ``s = (1/d) rowsum(dYq (.) Yq)`` with
    Yq = RoPE^T(QKV) recovered from the stored rotated output, and
    ``dYqr = r (.)row dYq``."""
    dYq = rope_bwd(dQKV, positions, head_dim, theta, rope_cols)
    Yq = rope_bwd(QKV, positions, head_dim, theta, rope_cols)
    return dict(dYq=dYq, dYqr=np.asarray(r, np.float64)[:, None] * dYq, s=rowdot_stat(dYq, Yq, d))


def block_fwd(P, Wd, x, gamma1, Wqkv, O, Wo, gamma2, Wgu, positions, head_dim: int, theta: float,
              rope_cols: int, eps: float) -> dict:
    """Unfused definition of one period of the chain (see the section header).
    Also reports the reparameterised intermediates h1g = h1 (.) gamma1 and
    h2g = h2 (.) gamma2."""
    g1 = np.asarray(gamma1, np.float64)
    g2 = np.asarray(gamma2, np.float64)
    h1 = matmul(P, Wd) + np.asarray(x, np.float64)
    n1, r1 = rmsnorm(h1, g1, eps)
    Yq = matmul(n1, Wqkv)
    QKV = rope(Yq, positions, head_dim, theta, rope_cols)
    h2 = matmul(O, Wo) + h1
    n2, r2 = rmsnorm(h2, g2, eps)
    GU = matmul(n2, Wgu)
    return dict(h1=h1, n1=n1, r1=r1, Yq=Yq, QKV=QKV, h2=h2, n2=n2, r2=r2, GU=GU, A=swiglu(GU),
                h1g=h1 * g1[None, :], h2g=h2 * g2[None, :])


def block_bwd(P, Wd, x, gamma1, Wqkv, O, Wo, gamma2, Wgu, positions, head_dim: int, theta: float,
              rope_cols: int, eps: float, dQKV, gh, Wdn) -> dict:
    """Backward of one period by the plain chain rule (textbook RMSNorm
    backward, no row statistic). dP = dh1 Wd^T is the gradient sent to the
    previous period; in a chain its GEMM is the previous period's
    SwiGLU-backward GEMM."""
    f = block_fwd(P, Wd, x, gamma1, Wqkv, O, Wo, gamma2, Wgu, positions, head_dim, theta, rope_cols, eps)
    gh = np.asarray(gh, np.float64)
    dA = matmul(gh, np.asarray(Wdn, np.float64).T)
    dGU = swiglu_bwd(dA, f["GU"])
    dn2 = matmul(dGU, np.asarray(Wgu, np.float64).T)
    b2 = rmsnorm_bwd_textbook(dn2, f["h2"], gamma2, f["r2"])
    dh2 = b2["du"] + gh
    dYq = rope_bwd(dQKV, positions, head_dim, theta, rope_cols)
    dn1 = matmul(dYq, np.asarray(Wqkv, np.float64).T)
    b1 = rmsnorm_bwd_textbook(dn1, f["h1"], gamma1, f["r1"])
    dh1 = b1["du"] + dh2
    return dict(
        fwd=f, dA=dA, dGU=dGU, dn2=dn2, dh2=dh2, dgamma2=b2["dgamma"], dWgu=matmul(f["n2"].T, dGU),
        dO=matmul(dh2, np.asarray(Wo, np.float64).T), dWo=matmul(np.asarray(O, np.float64).T, dh2),
        dYq=dYq, dn1=dn1, dh1=dh1, dx=dh1, dgamma1=b1["dgamma"], dWqkv=matmul(f["n1"].T, dYq),
        dWd=matmul(np.asarray(P, np.float64).T, dh1), dP=matmul(dh1, np.asarray(Wd, np.float64).T),
    )


def block_fwd_fused(P, Wd, x, gamma1, Wqkv, O, Wo, gamma2, Wgu, positions, head_dim: int, theta: float,
                    rope_cols: int, eps: float) -> dict:
    """The reparameterised forward, step by step as the fused kernels run it:
    residual + RMS-prep GEMM, aux reduction of the sums of squares, rowscale
    GEMM with the pair map, for each of the two structures."""
    d = np.asarray(x).shape[1]
    a = res_rmsprep(P, Wd, x, gamma1)
    r1 = rms_reduce(a["sumsq"][:, None], d, eps)
    QKV = gemm_rowscale_rope(a["h2"], Wqkv, r1, positions, head_dim, theta, rope_cols)
    b = res_rmsprep(O, Wo, a["h1"], gamma2)
    r2 = rms_reduce(b["sumsq"][:, None], d, eps)
    s = gemm_rowscale_swiglu(b["h2"], Wgu, r2)
    return dict(h1=a["h1"], h1g=a["h2"], r1=r1, QKV=QKV, h2=b["h1"], h2g=b["h2"], r2=r2, GU=s["GU"], A=s["A"])


def block_bwd_fused(fused_fwd: dict, P, Wqkv, O, Wo, gamma1, gamma2, Wgu, positions, head_dim: int,
                    theta: float, rope_cols: int, dQKV, gh, Wdn) -> dict:
    """The reparameterised backward, step by step as the fused kernels run
    it, from the fused forward's saved tensors: SwiGLU-backward GEMM with the
    row statistic; RMSNorm-backward GEMM with the residual gradient; the
    RoPE-path glue (transposed rotation, row statistic, row scale); the
    second RMSNorm-backward GEMM; the weight-gradient GEMMs on the row-scaled
    gradients."""
    f = fused_fwd
    d = f["h1"].shape[1]
    b1 = gemm_swiglu_bwd_rowdot(gh, Wdn, f["GU"], f["r2"], d)
    b3 = gemm_rmsnorm_bwd_res(b1["dGUr"], Wgu, f["h2"], gamma2, f["r2"], b1["s"], gh)
    dh2 = b3["dh"]
    g = rope_bwd_rowdot(dQKV, f["QKV"], f["r1"], positions, head_dim, theta, rope_cols, d)
    b10 = gemm_rmsnorm_bwd_res(g["dYqr"], Wqkv, f["h1"], gamma1, f["r1"], g["s"], dh2)
    dh1 = b10["dh"]
    return dict(
        dGUr=b1["dGUr"], s2=b1["s"], dh2=dh2, dgamma2=b3["dgamma"], dWgu=matmul(f["h2g"].T, b1["dGUr"]),
        dO=matmul(dh2, np.asarray(Wo, np.float64).T), dWo=matmul(np.asarray(O, np.float64).T, dh2),
        dYqr=g["dYqr"], s1=g["s"], dh1=dh1, dgamma1=b10["dgamma"], dWqkv=matmul(f["h1g"].T, g["dYqr"]),
        dWd=matmul(np.asarray(P, np.float64).T, dh1),
    )
