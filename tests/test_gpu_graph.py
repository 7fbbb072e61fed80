"""The fused launch sequences replay from a CUDA graph: the block chain's 19
launches (forward and backward) and the tiny GEMM-RMSNorm-GEMM chain are
captured once and replayed, and every output matches the directly launched
sequence bit for bit."""
import numpy as np
import pytest

import coda_inputs as gen
from _util import dev_bf16

pytestmark = pytest.mark.gpu


def _capture(fn):
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                      # first launches (kernel attributes, occupancy) happen outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    return g


def test_block_chain_graph_replay(coda):
    import torch
    M, d, F, hd, S = 256, 256, 384, 64, 128
    p = gen.block_problem(M, d, F, seed=31)
    t = {k: dev_bf16(v) for k, v in p.items()}
    cos, sin = coda.coda_rope_tables(S, hd, 10000.0)
    blk = coda.CodaBlock(t, hd, 2 * d, cos, sin)
    names = ("h1", "h2", "gu", "qkv", "a", "r1", "r2", "dgur", "dqr", "dh1", "dh2", "dO", "dWd", "dWqkv", "dWo",
             "dWgu", "dgamma1", "dgamma2", "s1", "s2")
    blk.fwd().bwd()
    torch.cuda.synchronize()
    ref = {k: getattr(blk, k).clone() for k in names}
    g = _capture(lambda: blk.fwd().bwd())
    for k in names:
        getattr(blk, k).fill_(float("nan"))
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for k in names:
            assert torch.equal(getattr(blk, k), ref[k]), k
    assert coda.coda_device_status(clear=True) == 0


def test_tiny_rms_chain_graph_replay(coda):
    import torch
    p = gen.rms_chain(256, 512, 512, 512, seed=0, bwd_K=512)
    x, W0, z, g_, W1, dO, Wn = (dev_bf16(p[k]) for k in ("x", "W0", "z", "gamma", "W1", "dO", "Wn"))
    out = {}

    def step():
        h1, h2, psq = coda.coda_gemm_res_rmsprep(x, W0, z, g_, h1=out.get("h1"), h2=out.get("h2"), psq=out.get("psq"))
        out.update(h1=h1, h2=h2, psq=psq)
        out["r"] = coda.coda_rms_reduce(psq, 512, 1e-6, r=out.get("r"))
        out["Y"] = coda.coda_gemm_rowscale(h2, W1, out["r"], out=out.get("Y"))

    step()
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in out.items()}
    g = _capture(step)
    for v in out.values():
        v.zero_()
    g.replay()
    torch.cuda.synchronize()
    for k, v in out.items():
        assert torch.equal(v, ref[k]), k


def test_capture_runs_without_the_split(coda):
    """A launch captured into a CUDA graph never uses the stream-K split (its
    arrival-word epoch would be baked into every replay): with the split forced
    on, the replayed GEMM gives the data-parallel schedule's bits, not those of
    the direct launch that used the split."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(17)
    A = (torch.randn(1800, 1096, device="cuda", generator=g)).bfloat16()
    B = (torch.randn(1096, 3400, device="cuda", generator=g) * 1096 ** -0.5).bfloat16()
    C = torch.empty(1800, 3400, dtype=torch.bfloat16, device="cuda")
    try:
        coda.coda_set_stream_k(0)
        dp = coda.coda_gemm(A, B).clone()
        coda.coda_set_stream_k(2)
        sk = coda.coda_gemm(A, B).clone()
        torch.cuda.synchronize()
        assert not torch.equal(dp, sk), "the direct launch did not use the split"
        graph = _capture(lambda: coda.coda_gemm(A, B, out=C))
        C.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(C, dp), "the captured launch used the split"
    finally:
        coda.coda_set_stream_k(1)
    assert coda.coda_device_status(clear=True) == 0

