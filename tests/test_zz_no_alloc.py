"""The block-chain forward without a caller workspace (coda_block_fwd_noalloc),
for callers that cannot allocate device memory: a plugin given only its input
and output buffers, a serving loop that may not call cudaMalloc after start-up
(the call can synchronise the device and take unbounded time), a process whose
pool already holds the device's memory. Its sum-of-squares partials live in
the library's static device array. Two calls in a row on one stream must both
give the workspace variant's bits and match the float64 oracle; a size past
the array's limit is refused before any launch."""
import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_stat, dev_bf16, f64

pytestmark = pytest.mark.gpu

EPS = 1e-6
THETA = 10000.0


def test_block_fwd_noalloc_twice(coda):
    import torch
    M, d, F, hd, S = 200, 256, 384, 64, 128
    rc = 2 * d
    p = gen.block_problem(M, d, F, seed=21, with_bwd=False)
    t = {k: dev_bf16(v) for k, v in p.items()}
    cos, sin = coda.coda_rope_tables(S, hd, THETA)
    ref_blk = coda.CodaBlock(t, hd, rc, cos, sin, EPS).fwd()
    blk = coda.CodaBlock(t, hd, rc, cos, sin, EPS)
    outs = []
    for _ in range(2):
        for k in ("h1", "h1g", "h2", "h2g", "gu", "qkv", "a", "r1", "r2"):
            getattr(blk, k).fill_(float("nan"))
        blk.fwd_noalloc()
        torch.cuda.synchronize()
        outs.append({k: getattr(blk, k).clone() for k in ("h1", "h2", "gu", "qkv", "a", "r1", "r2")})
    for k in outs[0]:
        assert torch.equal(outs[0][k], outs[1][k]), f"{k}: the two calls differ"
        assert torch.equal(outs[0][k], getattr(ref_blk, k)), f"{k}: differs from the workspace variant"
    b = {k: O.bf16(v) for k, v in p.items()}
    pos = np.arange(M) % S
    f = O.block_fwd(b["P"], b["Wd"], b["x"], b["gamma1"], b["Wqkv"], b["O"], b["Wo"], b["gamma2"], b["Wgu"], pos,
                    hd, THETA, rc, EPS)
    assert_stat(f64(blk.r1), O.rms_scale(O.res_rmsprep(b["P"], b["Wd"], b["x"], b["gamma1"])["h1"], EPS), "r1")
    for name in ("QKV", "A"):
        got = f64(blk.qkv if name == "QKV" else blk.a)
        err = np.linalg.norm(got - f[name]) / np.linalg.norm(f[name])
        assert err <= 1e-2, f"{name}: rel Frobenius {err:.3e} against the float64 chain"
    assert coda.coda_device_status(clear=True) == 0


def test_block_fwd_noalloc_limit(coda):
    from gemm_epilogue_transformer_gb300 import _lib
    b = _lib.CodaBlock()
    b.M, b.d, b.F = 1 << 20, 1024, 1024   # 2^20 rows x 8 blocks x 4 B = 32 MiB of partials
    assert coda.lib().coda_block_fwd_noalloc(b, None) == -2  # CODA_ERR_UNSUPPORTED, nothing launched
    assert b"static scratch" in coda.lib().coda_last_error()


def test_block_fwd_noalloc_never_splits(coda):
    """The no-allocation forward never takes the stream-K split, whose per-stream
    workspace would be allocated: with the split forced on, it gives the bits of
    the workspace variant run without the split, at a size where the split
    applies (1536 rows: the 3456-wide QKV GEMM has 84 SM-pair tiles and the
    4608-wide gate/up GEMM 108, on 76 pairs, with K = 1152)."""
    import torch
    M, d, F, hd, S = 1536, 1152, 2304, 128, 512
    p = gen.block_problem(M, d, F, seed=23, with_bwd=False)
    t = {k: dev_bf16(v) for k, v in p.items()}
    cos, sin = coda.coda_rope_tables(S, hd, THETA)
    names = ("h1", "h2", "gu", "qkv", "a", "r1", "r2")
    try:
        coda.coda_set_stream_k(0)
        ref = coda.CodaBlock(t, hd, 2 * d, cos, sin, EPS).fwd()
        coda.coda_set_stream_k(2)
        split = coda.CodaBlock(t, hd, 2 * d, cos, sin, EPS).fwd()
        blk = coda.CodaBlock(t, hd, 2 * d, cos, sin, EPS)
        blk.fwd_noalloc()
        torch.cuda.synchronize()
    finally:
        coda.coda_set_stream_k(1)
    assert not torch.equal(split.gu, ref.gu), "the workspace variant did not use the split"
    for k in names:
        assert torch.equal(getattr(blk, k), getattr(ref, k)), f"{k}: the no-allocation forward used the split"
    assert coda.coda_device_status(clear=True) == 0

