"""GB300 (sm_103a) CODA GEMM-epilogue library: Python binding.

Thin marshalling over the C ABI in include/coda.h (libcoda.so, loaded with
ctypes). Every computation runs in libcoda's CUDA kernels; this module only
checks tensor dtypes/devices/shapes, allocates outputs with torch, passes
pointers and the current CUDA stream, and turns error codes into exceptions.
Function names are the C names.

bf16 tensors are ``torch.bfloat16``; statistics ``torch.float32``; labels
``torch.int32``. All tensors live on the current CUDA device.
"""
from __future__ import annotations

import torch

from . import _lib

__all__ = [
    "CodaError", "lib", "coda_init", "coda_device_status", "coda_set_wait_timeout_ns", "coda_set_cta_group", "coda_set_stream_k", "coda_test_inject_missing_load",
    "coda_num_col_tiles", "coda_num_row_tiles", "coda_gemm", "coda_gemm_res_rmsprep", "coda_rms_reduce",
    "coda_gemm_rowscale", "coda_gemm_swiglu", "coda_gemm_swiglu_bwd", "coda_rope_tables", "coda_gemm_rope",
    "coda_gemm_rope_bwd", "coda_gemm_ce_lse", "coda_ce_reduce", "coda_gemm_ce_bwd", "coda_gemm_rowdot",
    "coda_rowdot_reduce", "coda_gemm_rmsnorm_bwd", "coda_colsum_reduce", "coda_unfused_add",
    "coda_unfused_rmsnorm", "coda_unfused_rowscale", "coda_unfused_swiglu", "coda_unfused_swiglu_bwd",
    "coda_unfused_rope", "coda_unfused_rope_bwd", "coda_unfused_ce_fwd", "coda_unfused_ce_bwd",
    "coda_unfused_rowdot", "coda_unfused_rmsnorm_bwd", "coda_gemm_rowscale_rope", "coda_gemm_rowscale_swiglu",
    "coda_gemm_swiglu_bwd_rowdot", "coda_gemm_rmsnorm_bwd_res", "coda_rope_bwd_rowdot",
    "coda_block_workspace_bytes", "CodaBlock", "coda_gemm_fp8", "coda_gemm_rope_fp8", "coda_gemm_swiglu_fp8",
    "coda_gemm_ce_lse_fp8", "coda_gemm_ce_bwd_fp8",
]


class CodaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libcoda error {code}: {msg}")
        self.code = code


def lib():
    return _lib.load()


def _check(rc: int):
    if rc != 0:
        raise CodaError(rc, lib().coda_last_error().decode(errors="replace"))


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _on_device(t, name):
    """The kernels run on the current CUDA device and read every pointer there."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (got {type(t).__name__}"
                        f"{' on ' + str(t.device) if isinstance(t, torch.Tensor) else ''})")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, not on the current device cuda:{torch.cuda.current_device()}")
    return t


def _typed(t, name, dtype, ndim=None, shape=None):
    """Dtype, device, contiguity and (optionally) rank and exact shape of a tensor
    the kernels read or write: a mismatch here would become an out-of-bounds
    access on the device, so it is rejected before the call."""
    _on_device(t, name)
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims (got {tuple(t.shape)})")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)} (got {tuple(t.shape)})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _bf16(t, name, ndim=None, shape=None):
    return _typed(t, name, torch.bfloat16, ndim, shape)


def _f32(t, name, shape=None):
    return _typed(t, name, torch.float32, None, shape)


def _i32(t, name, shape=None):
    return _typed(t, name, torch.int32, None, shape)


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


def _out(t, shape, dtype, like, name="out"):
    """A caller-provided output buffer, checked like an input; else a new one."""
    return _empty(shape, dtype, like) if t is None else _typed(t, name, dtype, None, shape)


def _mismatch(args) -> str:
    """Message for inconsistent operand shapes, listing every tensor argument."""
    shapes = ", ".join(f"{k} {tuple(v.shape)}" for k, v in args.items() if isinstance(v, torch.Tensor))
    return f"shape mismatch: {shapes}"


def _tables(cos, sin, head_dim):
    _f32(cos, "cos", None), _f32(sin, "sin", None)
    if cos.dim() != 2 or cos.shape != sin.shape or cos.shape[1] != head_dim // 2:
        raise ValueError(f"cos and sin must both be [S, head_dim/2 = {head_dim // 2}] "
                         f"(got {tuple(cos.shape)} and {tuple(sin.shape)})")


# ----------------------------------------------------------------- runtime

def coda_init(device: int = 0):
    _check(lib().coda_init(device))


def coda_device_status(clear: bool = True) -> int:
    rc = lib().coda_device_status(1 if clear else 0)
    if rc < 0:
        _check(rc)
    return rc


def coda_set_wait_timeout_ns(ns: int):
    _check(lib().coda_set_wait_timeout_ns(int(ns)))


def coda_set_cta_group(g: int):
    """0 = automatic, 1 = single-SM 128 x 256 tiles, 2 = SM-pair 256 x 256 tiles."""
    _check(lib().coda_set_cta_group(int(g)))


def coda_set_stream_k(mode: int):
    """Stream-K split of the fused GEMMs: 0 = off, 1 = automatic (default), 2 = wherever it applies."""
    _check(lib().coda_set_stream_k(int(mode)))


def coda_test_inject_missing_load():
    """Test hook: the next fused-GEMM launch skips its first stage fill (see coda.h)."""
    _check(lib().coda_test_inject_missing_load())


def coda_num_col_tiles(N: int) -> int:
    return lib().coda_num_col_tiles(N)


def coda_num_row_tiles(M: int) -> int:
    return lib().coda_num_row_tiles(M)


# ----------------------------------------------------------------- GEMMs

def coda_gemm(A, B, transA: bool = False, transB: bool = False, out=None, stream=None):
    """C = op(A) op(B). A is [M,K] (or [K,M] with transA), B is [K,N] (or [N,K])."""
    for t, nm in ((A, "A"), (B, "B")):
        _on_device(t, nm)
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{nm} must be bfloat16 (got {t.dtype})")
    if A.dim() != 2 or B.dim() != 2 or A.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("A and B must be 2-D with unit column stride")
    M, K = (A.shape[1], A.shape[0]) if transA else (A.shape[0], A.shape[1])
    Kb, N = (B.shape[1], B.shape[0]) if transB else (B.shape[0], B.shape[1])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    if out is None:
        out = _empty((M, N), torch.bfloat16, A)
    _on_device(out, "out")
    if out.dtype != torch.bfloat16 or out.dim() != 2 or tuple(out.shape) != (M, N) or out.stride(1) != 1:
        raise ValueError(f"out must be a bfloat16 [{M}, {N}] tensor with unit column stride")
    _check(lib().coda_gemm(M, N, K, _ptr(A), A.stride(0), int(transA), _ptr(B), B.stride(0), int(transB),
                           _ptr(out), out.stride(0), _stream(stream)))
    return out


def coda_gemm_res_rmsprep(x, W0, z, gamma, h1=None, h2=None, psq=None, stream=None):
    """h1 = x W0 + z, h2 = h1 * gamma, psq = per-column-tile sums of h1^2."""
    _bf16(x, "x", 2), _bf16(W0, "W0", 2), _bf16(z, "z", 2), _bf16(gamma, "gamma", 1)
    M, K = x.shape
    N = W0.shape[1]
    if W0.shape[0] != K or z.shape != (M, N) or gamma.shape[0] != N:
        raise ValueError(_mismatch(locals()))
    h1 = _out(h1, (M, N), torch.bfloat16, x, "h1")
    h2 = _out(h2, (M, N), torch.bfloat16, x, "h2")
    psq = _out(psq, (M, coda_num_col_tiles(N)), torch.float32, x, "psq")
    _check(lib().coda_gemm_res_rmsprep(M, N, K, _ptr(x), _ptr(W0), _ptr(z), _ptr(gamma), _ptr(h1), _ptr(h2),
                                       _ptr(psq), _stream(stream)))
    return h1, h2, psq


def coda_rms_reduce(psq, d: int, eps: float, r=None, stream=None):
    _f32(psq, "psq")
    if psq.dim() != 2:
        raise ValueError("psq must be [M, nb]")
    M, nb = psq.shape
    r = _out(r, (M,), torch.float32, psq, "r")
    _check(lib().coda_rms_reduce(M, nb, d, _ptr(psq), float(eps), _ptr(r), _stream(stream)))
    return r


def coda_gemm_rowscale(h2, W1, r, out=None, stream=None):
    _bf16(h2, "h2", 2), _bf16(W1, "W1", 2), _f32(r, "r")
    M, K = h2.shape
    N = W1.shape[1]
    if W1.shape[0] != K or r.shape[0] != M:
        raise ValueError(_mismatch(locals()))
    out = _out(out, (M, N), torch.bfloat16, h2)
    _check(lib().coda_gemm_rowscale(M, N, K, _ptr(h2), _ptr(W1), _ptr(r), _ptr(out), _stream(stream)))
    return out


def coda_gemm_swiglu(X, Wgu, want_gu: bool = False, out=None, gu=None, stream=None):
    """A = silu(G) * U with gate/up interleaved in the columns of X Wgu."""
    _bf16(X, "X", 2), _bf16(Wgu, "Wgu", 2)
    M, K = X.shape
    F2 = Wgu.shape[1]
    if Wgu.shape[0] != K or F2 % 2:
        raise ValueError(_mismatch(locals()))
    F = F2 // 2
    out = _out(out, (M, F), torch.bfloat16, X)
    gu = _out(gu, (M, F2), torch.bfloat16, X, "gu") if (want_gu or gu is not None) else None
    _check(lib().coda_gemm_swiglu(M, F, K, _ptr(X), _ptr(Wgu), _ptr(out), _ptr(gu), _stream(stream)))
    return out, gu


def coda_gemm_swiglu_bwd(dY, Wd, gu, out=None, stream=None):
    """dGU (interleaved dG, dU) from dA = dY Wd^T; Wd stored [F, K]."""
    _bf16(dY, "dY", 2), _bf16(Wd, "Wd", 2)
    M, K = dY.shape
    F = Wd.shape[0]
    if Wd.shape[1] != K:
        raise ValueError(f"Wd must be [F, K = {K}] (got {tuple(Wd.shape)})")
    _bf16(gu, "gu", 2, (M, 2 * F))
    out = _out(out, (M, 2 * F), torch.bfloat16, dY)
    _check(lib().coda_gemm_swiglu_bwd(M, F, K, _ptr(dY), _ptr(Wd), _ptr(gu), _ptr(out), _stream(stream)))
    return out


def coda_rope_tables(S: int, head_dim: int, theta: float, device=None, stream=None):
    device = torch.device("cuda") if device is None else device
    c = torch.empty((S, head_dim // 2), dtype=torch.float32, device=device)
    s = torch.empty_like(c)
    _check(lib().coda_rope_tables(S, head_dim, float(theta), _ptr(c), _ptr(s), _stream(stream)))
    return c, s


def _rope(fname, X, W, cos, sin, head_dim, rope_cols, out, stream):
    _bf16(X, "X", 2), _bf16(W, "W", 2), _tables(cos, sin, head_dim)
    M, K = X.shape
    N = W.shape[1]
    if W.shape[0] != K:
        raise ValueError(_mismatch(locals()))
    out = _out(out, (M, N), torch.bfloat16, X)
    _check(getattr(lib(), fname)(M, N, K, _ptr(X), _ptr(W), _ptr(cos), _ptr(sin), cos.shape[0], head_dim,
                                 rope_cols, _ptr(out), _stream(stream)))
    return out


def coda_gemm_rope(X, W, cos, sin, head_dim: int, rope_cols: int, out=None, stream=None):
    return _rope("coda_gemm_rope", X, W, cos, sin, head_dim, rope_cols, out, stream)


def coda_gemm_rope_bwd(A, B, cos, sin, head_dim: int, rope_cols: int, out=None, stream=None):
    return _rope("coda_gemm_rope_bwd", A, B, cos, sin, head_dim, rope_cols, out, stream)


def coda_gemm_ce_lse(H, W, labels, with_argmax: bool = True, stream=None):
    """Per-(row, column tile) (max, sum exp, argmax) of the logits H W and the
    target logit per row. Returns (pmax, psum, parg or None, tgt)."""
    _bf16(H, "H", 2), _bf16(W, "W", 2), _i32(labels, "labels")
    M, K = H.shape
    V = W.shape[1]
    if W.shape[0] != K or labels.shape[0] != M:
        raise ValueError(_mismatch(locals()))
    nb = coda_num_col_tiles(V)
    pmax = _empty((M, nb), torch.float32, H)
    psum = _empty((M, nb), torch.float32, H)
    parg = _empty((M, nb), torch.int32, H) if with_argmax else None
    tgt = _empty((M,), torch.float32, H)
    _check(lib().coda_gemm_ce_lse(M, V, K, _ptr(H), _ptr(W), _ptr(labels), _ptr(pmax), _ptr(psum), _ptr(parg),
                                  _ptr(tgt), _stream(stream)))
    return pmax, psum, parg, tgt


def coda_ce_reduce(pmax, psum, parg, tgt, stream=None):
    """Returns (lse, loss_row, loss_mean[1], argmax or None)."""
    _f32(pmax, "pmax")
    if pmax.dim() != 2:
        raise ValueError("pmax must be [M, nb]")
    M, nb = pmax.shape
    _f32(psum, "psum", (M, nb)), _f32(tgt, "tgt", (M,))
    if parg is not None:
        _i32(parg, "parg", (M, nb))
    lse = _empty((M,), torch.float32, pmax)
    loss_row = _empty((M,), torch.float32, pmax)
    loss_mean = _empty((1,), torch.float32, pmax)
    argmax = _empty((M,), torch.int32, pmax) if parg is not None else None
    _check(lib().coda_ce_reduce(M, nb, _ptr(pmax), _ptr(psum), _ptr(parg), _ptr(tgt), _ptr(lse), _ptr(loss_row),
                                _ptr(loss_mean), _ptr(argmax), _stream(stream)))
    return lse, loss_row, loss_mean, argmax


def coda_gemm_ce_bwd(H, W, labels, lse, grad_scale: float, out=None, stream=None):
    _bf16(H, "H", 2), _bf16(W, "W", 2)
    M, K = H.shape
    V = W.shape[1]
    if W.shape[0] != K:
        raise ValueError(_mismatch(locals()))
    _i32(labels, "labels", (M,)), _f32(lse, "lse", (M,))
    out = _out(out, (M, V), torch.bfloat16, H)
    _check(lib().coda_gemm_ce_bwd(M, V, K, _ptr(H), _ptr(W), _ptr(labels), _ptr(lse), float(grad_scale),
                                  _ptr(out), _stream(stream)))
    return out


def coda_gemm_rowdot(dO, Wn, Y, r=None, want_dyr: bool = True, stream=None):
    """dY = dO Wn, dYr = r * dY (optional), pdot tile partials of rowsum(dY * Y)."""
    _bf16(dO, "dO", 2), _bf16(Wn, "Wn", 2)
    M, K = dO.shape
    N = Wn.shape[1]
    if Wn.shape[0] != K:
        raise ValueError(_mismatch(locals()))
    _bf16(Y, "Y", 2, (M, N))
    if want_dyr:
        if r is None:
            raise ValueError("r is required for the dYr side output")
        _f32(r, "r", (M,))
    dY = _empty((M, N), torch.bfloat16, dO)
    dYr = _empty((M, N), torch.bfloat16, dO) if want_dyr else None
    pdot = _empty((M, coda_num_col_tiles(N)), torch.float32, dO)
    _check(lib().coda_gemm_rowdot(M, N, K, _ptr(dO), _ptr(Wn), _ptr(Y), _ptr(r), _ptr(dY), _ptr(dYr), _ptr(pdot),
                                  _stream(stream)))
    return dY, dYr, pdot


def coda_rowdot_reduce(pdot, d: int, stream=None):
    _f32(pdot, "pdot")
    if pdot.dim() != 2:
        raise ValueError("pdot must be [M, nb]")
    M, nb = pdot.shape
    s = _empty((M,), torch.float32, pdot)
    _check(lib().coda_rowdot_reduce(M, nb, d, _ptr(pdot), _ptr(s), _stream(stream)))
    return s


def coda_gemm_rmsnorm_bwd(dY, W1, h1, gamma, r, s, stream=None):
    """dh1 = r gamma G - r^2 s h1 with G = dY W1^T (W1 stored [d, K]); pdg column partials."""
    _bf16(dY, "dY", 2), _bf16(W1, "W1", 2)
    M, K = dY.shape
    d = W1.shape[0]
    if W1.shape[1] != K:
        raise ValueError(_mismatch(locals()))
    _bf16(h1, "h1", 2, (M, d)), _bf16(gamma, "gamma", 1, (d,)), _f32(r, "r", (M,)), _f32(s, "s", (M,))
    dh1 = _empty((M, d), torch.bfloat16, dY)
    pdg = _empty((coda_num_row_tiles(M), d), torch.float32, dY)
    _check(lib().coda_gemm_rmsnorm_bwd(M, d, K, _ptr(dY), _ptr(W1), _ptr(h1), _ptr(gamma), _ptr(r), _ptr(s),
                                       _ptr(dh1), _ptr(pdg), _stream(stream)))
    return dh1, pdg


def coda_colsum_reduce(pdg, stream=None):
    _f32(pdg, "pdg")
    if pdg.dim() != 2:
        raise ValueError("pdg must be [rows, d]")
    rows, d = pdg.shape
    out = _empty((d,), torch.float32, pdg)
    _check(lib().coda_colsum_reduce(rows, d, _ptr(pdg), _ptr(out), _stream(stream)))
    return out


# ----------------------------------------------------------------- unfused path

def coda_unfused_add(a, b, out=None, stream=None):
    _bf16(a, "a", 2)
    M, N = a.shape
    _bf16(b, "b", 2, (M, N))
    out = _out(out, (M, N), torch.bfloat16, a)
    _check(lib().coda_unfused_add(M, N, _ptr(a), _ptr(b), _ptr(out), _stream(stream)))
    return out


def coda_unfused_rmsnorm(h, gamma, eps: float, stream=None):
    _bf16(h, "h", 2)
    M, d = h.shape
    _bf16(gamma, "gamma", 1, (d,))
    n = torch.empty_like(h)
    r = _empty((M,), torch.float32, h)
    _check(lib().coda_unfused_rmsnorm(M, d, _ptr(h), _ptr(gamma), float(eps), _ptr(n), _ptr(r), _stream(stream)))
    return n, r


def coda_unfused_rowscale(x, r, stream=None):
    _bf16(x, "x", 2)
    M, N = x.shape
    _f32(r, "r", (M,))
    out = torch.empty_like(x)
    _check(lib().coda_unfused_rowscale(M, N, _ptr(x), _ptr(r), _ptr(out), _stream(stream)))
    return out


def coda_unfused_swiglu(gu, stream=None):
    _bf16(gu, "gu", 2)
    M, F2 = gu.shape
    if F2 % 2:
        raise ValueError("gu must have an even number of columns (gate/up pairs)")
    out = _empty((M, F2 // 2), torch.bfloat16, gu)
    _check(lib().coda_unfused_swiglu(M, F2 // 2, _ptr(gu), _ptr(out), _stream(stream)))
    return out


def coda_unfused_swiglu_bwd(dA, gu, stream=None):
    _bf16(dA, "dA", 2)
    M, F = dA.shape
    _bf16(gu, "gu", 2, (M, 2 * F))
    out = _empty((M, 2 * F), torch.bfloat16, dA)
    _check(lib().coda_unfused_swiglu_bwd(M, F, _ptr(dA), _ptr(gu), _ptr(out), _stream(stream)))
    return out


def coda_unfused_rope(x, cos, sin, head_dim: int, rope_cols: int, stream=None):
    """In place on x [M, N]."""
    _bf16(x, "x", 2), _tables(cos, sin, head_dim)
    M, N = x.shape
    _check(lib().coda_unfused_rope(M, N, _ptr(cos), _ptr(sin), cos.shape[0], head_dim, rope_cols, _ptr(x),
                                   _stream(stream)))
    return x


def coda_unfused_rope_bwd(x, cos, sin, head_dim: int, rope_cols: int, stream=None):
    _bf16(x, "x", 2), _tables(cos, sin, head_dim)
    M, N = x.shape
    _check(lib().coda_unfused_rope_bwd(M, N, _ptr(cos), _ptr(sin), cos.shape[0], head_dim, rope_cols, _ptr(x),
                                       _stream(stream)))
    return x


def coda_unfused_ce_fwd(logits, labels, stream=None):
    _bf16(logits, "logits", 2)
    M, V = logits.shape
    _i32(labels, "labels", (M,))
    lse = _empty((M,), torch.float32, logits)
    loss_row = _empty((M,), torch.float32, logits)
    loss_mean = _empty((1,), torch.float32, logits)
    argmax = _empty((M,), torch.int32, logits)
    _check(lib().coda_unfused_ce_fwd(M, V, _ptr(logits), _ptr(labels), _ptr(lse), _ptr(loss_row), _ptr(loss_mean),
                                     _ptr(argmax), _stream(stream)))
    return lse, loss_row, loss_mean, argmax


def coda_unfused_ce_bwd(logits, labels, lse, grad_scale: float, stream=None):
    _bf16(logits, "logits", 2)
    M, V = logits.shape
    _i32(labels, "labels", (M,)), _f32(lse, "lse", (M,))
    out = torch.empty_like(logits)
    _check(lib().coda_unfused_ce_bwd(M, V, _ptr(logits), _ptr(labels), _ptr(lse), float(grad_scale), _ptr(out),
                                     _stream(stream)))
    return out


def coda_unfused_rowdot(dY, Y, d: int, stream=None):
    _bf16(dY, "dY", 2)
    M, N = dY.shape
    _bf16(Y, "Y", 2, (M, N))
    s = _empty((M,), torch.float32, dY)
    _check(lib().coda_unfused_rowdot(M, N, d, _ptr(dY), _ptr(Y), _ptr(s), _stream(stream)))
    return s


def coda_unfused_rmsnorm_bwd(G, h, gamma, r, stream=None):
    _bf16(G, "G", 2)
    M, d = G.shape
    _bf16(h, "h", 2, (M, d)), _bf16(gamma, "gamma", 1, (d,)), _f32(r, "r", (M,))
    dh = torch.empty_like(G)
    pdg = _empty((coda_num_row_tiles(M), d), torch.float32, G)
    _check(lib().coda_unfused_rmsnorm_bwd(M, d, _ptr(G), _ptr(h), _ptr(gamma), _ptr(r), _ptr(dh), _ptr(pdg),
                                          _stream(stream)))
    return dh, pdg


# ----------------------------------------------------------------- block-level chain

def coda_gemm_rowscale_rope(X, W, r, cos, sin, head_dim: int, rope_cols: int, out=None, stream=None):
    """out = RoPE(r * (X W)) (row scale and rotation in one epilogue)."""
    _bf16(X, "X", 2), _bf16(W, "W", 2), _tables(cos, sin, head_dim)
    M, K = X.shape
    N = W.shape[1]
    if W.shape[0] != K:
        raise ValueError(_mismatch(locals()))
    _f32(r, "r", (M,))
    out = _out(out, (M, N), torch.bfloat16, X)
    _check(lib().coda_gemm_rowscale_rope(M, N, K, _ptr(X), _ptr(W), _ptr(r), _ptr(cos), _ptr(sin), cos.shape[0],
                                         head_dim, rope_cols, _ptr(out), _stream(stream)))
    return out


def coda_gemm_rowscale_swiglu(X, Wgu, r, want_gu: bool = False, out=None, gu=None, stream=None):
    """GU = r * (X Wgu), A = silu(G) * U; returns (A, GU or None)."""
    _bf16(X, "X", 2), _bf16(Wgu, "Wgu", 2)
    M, K = X.shape
    F2 = Wgu.shape[1]
    if Wgu.shape[0] != K or F2 % 2:
        raise ValueError(_mismatch(locals()))
    _f32(r, "r", (M,))
    F = F2 // 2
    out = _out(out, (M, F), torch.bfloat16, X)
    gu = _out(gu, (M, F2), torch.bfloat16, X, "gu") if (want_gu or gu is not None) else None
    _check(lib().coda_gemm_rowscale_swiglu(M, F, K, _ptr(X), _ptr(Wgu), _ptr(r), _ptr(out), _ptr(gu),
                                           _stream(stream)))
    return out, gu


def coda_gemm_swiglu_bwd_rowdot(dY, Wd, gu, r, stream=None):
    """dGUr = r * SwiGLU'(dY Wd^T; gu) and the row-statistic partials of dGU * gu.
    Returns (dgur [M,2F], pdot [M, ceil(F/128)])."""
    _bf16(dY, "dY", 2), _bf16(Wd, "Wd", 2)
    M, K = dY.shape
    F = Wd.shape[0]
    if Wd.shape[1] != K:
        raise ValueError(_mismatch(locals()))
    _bf16(gu, "gu", 2, (M, 2 * F)), _f32(r, "r", (M,))
    dgur = _empty((M, 2 * F), torch.bfloat16, dY)
    pdot = _empty((M, coda_num_col_tiles(F)), torch.float32, dY)
    _check(lib().coda_gemm_swiglu_bwd_rowdot(M, F, K, _ptr(dY), _ptr(Wd), _ptr(gu), _ptr(r), _ptr(dgur), _ptr(pdot),
                                             _stream(stream)))
    return dgur, pdot


def coda_gemm_rmsnorm_bwd_res(dYr, W1, h, gamma, r, s, dres, stream=None):
    """dh = gamma * (dYr W1^T) - r^2 s h + dres (W1 stored [d, K]); returns (dh, pdg)."""
    _bf16(dYr, "dYr", 2), _bf16(W1, "W1", 2)
    M, K = dYr.shape
    d = W1.shape[0]
    if W1.shape[1] != K:
        raise ValueError(_mismatch(locals()))
    _bf16(h, "h", 2, (M, d)), _bf16(gamma, "gamma", 1, (d,)), _bf16(dres, "dres", 2, (M, d))
    _f32(r, "r", (M,)), _f32(s, "s", (M,))
    dh = _empty((M, d), torch.bfloat16, dYr)
    pdg = _empty((coda_num_row_tiles(M), d), torch.float32, dYr)
    _check(lib().coda_gemm_rmsnorm_bwd_res(M, d, K, _ptr(dYr), _ptr(W1), _ptr(h), _ptr(gamma), _ptr(r), _ptr(s),
                                           _ptr(dres), _ptr(dh), _ptr(pdg), _stream(stream)))
    return dh, pdg


def coda_rope_bwd_rowdot(dqkv, qkv, r, cos, sin, head_dim: int, rope_cols: int, d: int, stream=None):
    """dqr = r * RoPE^T(dqkv), s = (1/d) rowsum(dqkv * qkv); returns (dqr, s)."""
    _bf16(dqkv, "dqkv", 2), _tables(cos, sin, head_dim)
    M, N = dqkv.shape
    _bf16(qkv, "qkv", 2, (M, N)), _f32(r, "r", (M,))
    dqr = torch.empty_like(dqkv)
    s = _empty((M,), torch.float32, dqkv)
    _check(lib().coda_rope_bwd_rowdot(M, N, _ptr(dqkv), _ptr(qkv), _ptr(r), _ptr(cos), _ptr(sin), cos.shape[0],
                                      head_dim, rope_cols, d, _ptr(dqr), _ptr(s), _stream(stream)))
    return dqr, s


def coda_block_workspace_bytes(M: int, d: int, F: int, unfused: bool = False) -> int:
    return int(lib().coda_block_workspace_bytes(M, d, F, int(unfused)))


class CodaBlock:
    """One period of the block-level chain (coda_block_t): the caller's inputs
    and weights, and every saved tensor, output and scratch buffer, allocated
    here with torch. ``fwd()``/``bwd()`` run the fused sequence,
    ``fwd_unfused()``/``bwd_unfused()`` the unfused one (which rotates
    ``dqkv`` in place). Field meanings are those of include/coda.h.

    ``t``: dict of CUDA bf16 tensors P, x, O, Wd, gamma1, Wqkv, Wo, gamma2, Wgu
    and, for the backward, dQKV, gh, Wdn.
    """

    _IN = ("P", "x", "O", "Wd", "gamma1", "Wqkv", "Wo", "gamma2", "Wgu")

    def __init__(self, t: dict, head_dim: int, rope_cols: int, cos, sin, eps: float = 1e-6, unfused: bool = False):
        _bf16(t["P"], "P", 2), _bf16(t["x"], "x", 2)
        M, F = t["P"].shape
        d = t["x"].shape[1]
        shapes = {"P": (M, F), "x": (M, d), "O": (M, d), "Wd": (F, d), "gamma1": (d,), "Wqkv": (d, 3 * d),
                  "Wo": (d, d), "gamma2": (d,), "Wgu": (d, 2 * F), "dQKV": (M, 3 * d), "gh": (M, d), "Wdn": (F, d)}
        for k in self._IN:
            _bf16(t[k], k, None, shapes[k])
        _tables(cos, sin, head_dim)
        dev = t["x"]
        bf, f32 = torch.bfloat16, torch.float32
        self.M, self.d, self.F = M, d, F
        self.t = t
        self.cos, self.sin = cos, sin
        e = lambda *shape, dt=bf: _empty(shape, dt, dev)  # noqa: E731
        self.h1, self.h1g, self.h2, self.h2g = e(M, d), e(M, d), e(M, d), e(M, d)
        self.gu, self.r1, self.r2 = e(M, 2 * F), e(M, dt=f32), e(M, dt=f32)
        self.qkv, self.a = e(M, 3 * d), e(M, F)
        self.dh1, self.dh2, self.dO = e(M, d), e(M, d), e(M, d)
        self.dWd, self.dWqkv, self.dWo, self.dWgu = e(F, d), e(d, 3 * d), e(d, d), e(d, 2 * F)
        self.dgamma1, self.dgamma2 = e(d, dt=f32), e(d, dt=f32)
        self.dgur, self.dqr = e(M, 2 * F), e(M, 3 * d)
        self.s1, self.s2 = e(M, dt=f32), e(M, dt=f32)
        nbytes = max(coda_block_workspace_bytes(M, d, F, unfused), coda_block_workspace_bytes(M, d, F, False))
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev.device)
        ws = (self.workspace.data_ptr() + 255) & ~255
        b = _lib.CodaBlock()
        b.M, b.d, b.F, b.head_dim, b.rope_cols, b.S, b.eps = M, d, F, head_dim, rope_cols, cos.shape[0], float(eps)
        b.cos_tab, b.sin_tab = _ptr(cos), _ptr(sin)
        for k in self._IN:
            setattr(b, k, _ptr(t[k]))
        for k in ("h1", "h1g", "h2", "h2g", "gu", "r1", "r2", "qkv", "a", "dh1", "dh2", "dO", "dWd", "dWqkv", "dWo",
                  "dWgu", "dgamma1", "dgamma2", "dgur", "dqr", "s1", "s2"):
            setattr(b, k, _ptr(getattr(self, k)))
        for k, f in (("dQKV", "dqkv"), ("gh", "gh"), ("Wdn", "Wdn")):
            if k in t:
                _bf16(t[k], k, None, shapes[k])
                setattr(b, f, _ptr(t[k]))
        b.workspace = ws
        self._b = b

    def _run(self, fname, stream):
        _check(getattr(lib(), fname)(self._b, _stream(stream)))
        return self

    def fwd(self, stream=None):
        return self._run("coda_block_fwd", stream)

    def fwd_noalloc(self, stream=None):
        """The fused forward with the library's static scratch instead of the
        workspace (coda_block_fwd_noalloc); calls must not overlap on the GPU."""
        return self._run("coda_block_fwd_noalloc", stream)

    def bwd(self, stream=None):
        return self._run("coda_block_bwd", stream)

    def fwd_unfused(self, stream=None):
        return self._run("coda_block_fwd_unfused", stream)

    def bwd_unfused(self, stream=None):
        return self._run("coda_block_bwd_unfused", stream)


# ----------------------------------------------------------------- FP8 (E4M3) mainloop

def _e4m3(t, name):
    """E4M3 operands travel as uint8 tensors (or torch.float8_e4m3fn, viewed as bytes)."""
    if t.dtype != torch.uint8:
        if str(t.dtype) != "torch.float8_e4m3fn":
            raise TypeError(f"{name} must be a CUDA uint8 or float8_e4m3fn tensor (got {t.dtype})")
        t = t.view(torch.uint8)
    _on_device(t, name)
    if not t.is_contiguous() or t.dim() != 2:
        raise ValueError(f"{name} must be a contiguous 2-D CUDA tensor")
    return t


def coda_gemm_fp8(A, B, alpha: float, out=None, stream=None):
    """C = alpha A B^T with A [M,K], B [N,K] E4M3; C bf16 [M,N]."""
    A, B = _e4m3(A, "A"), _e4m3(B, "B")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError(_mismatch(locals()))
    out = _out(out, (M, N), torch.bfloat16, A)
    _check(lib().coda_gemm_fp8(M, N, K, _ptr(A), _ptr(B), float(alpha), _ptr(out), _stream(stream)))
    return out


def coda_gemm_rope_fp8(X, W, alpha: float, cos, sin, head_dim: int, rope_cols: int, out=None, stream=None):
    X, W = _e4m3(X, "X"), _e4m3(W, "W")
    _tables(cos, sin, head_dim)
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError(_mismatch(locals()))
    out = _out(out, (M, N), torch.bfloat16, X)
    _check(lib().coda_gemm_rope_fp8(M, N, K, _ptr(X), _ptr(W), float(alpha), _ptr(cos), _ptr(sin), cos.shape[0],
                                    head_dim, rope_cols, _ptr(out), _stream(stream)))
    return out


def coda_gemm_swiglu_fp8(X, Wgu, alpha: float, want_gu: bool = False, out=None, gu=None, stream=None):
    """A = silu(G) * U on GU = alpha X Wgu^T, Wgu [2F, K] (rows gate/up interleaved); returns (A, GU or None)."""
    X, Wgu = _e4m3(X, "X"), _e4m3(Wgu, "Wgu")
    M, K = X.shape
    F2 = Wgu.shape[0]
    if Wgu.shape[1] != K or F2 % 2:
        raise ValueError(_mismatch(locals()))
    F = F2 // 2
    out = _out(out, (M, F), torch.bfloat16, X)
    gu = _out(gu, (M, F2), torch.bfloat16, X, "gu") if (want_gu or gu is not None) else None
    _check(lib().coda_gemm_swiglu_fp8(M, F, K, _ptr(X), _ptr(Wgu), float(alpha), _ptr(out), _ptr(gu),
                                      _stream(stream)))
    return out, gu


def coda_gemm_ce_lse_fp8(H, W, alpha: float, labels, with_argmax: bool = True, stream=None):
    H, W = _e4m3(H, "H"), _e4m3(W, "W")
    _i32(labels, "labels")
    M, K = H.shape
    V = W.shape[0]
    if W.shape[1] != K or labels.shape[0] != M:
        raise ValueError(_mismatch(locals()))
    nb = coda_num_col_tiles(V)
    pmax = _empty((M, nb), torch.float32, H)
    psum = _empty((M, nb), torch.float32, H)
    parg = _empty((M, nb), torch.int32, H) if with_argmax else None
    tgt = _empty((M,), torch.float32, H)
    _check(lib().coda_gemm_ce_lse_fp8(M, V, K, _ptr(H), _ptr(W), float(alpha), _ptr(labels), _ptr(pmax), _ptr(psum),
                                      _ptr(parg), _ptr(tgt), _stream(stream)))
    return pmax, psum, parg, tgt


def coda_gemm_ce_bwd_fp8(H, W, alpha: float, labels, lse, grad_scale: float, out=None, stream=None):
    H, W = _e4m3(H, "H"), _e4m3(W, "W")
    M, K = H.shape
    V = W.shape[0]
    if W.shape[1] != K:
        raise ValueError(_mismatch(locals()))
    _i32(labels, "labels", (M,)), _f32(lse, "lse", (M,))
    out = _out(out, (M, V), torch.bfloat16, H)
    _check(lib().coda_gemm_ce_bwd_fp8(M, V, K, _ptr(H), _ptr(W), float(alpha), _ptr(labels), _ptr(lse),
                                      float(grad_scale), _ptr(out), _stream(stream)))
    return out
