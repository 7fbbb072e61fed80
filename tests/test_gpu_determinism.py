"""Determinism of the fused kernels: repeated launches of each tile variant
(single-SM and SM-pair) give the same bits.

Every launch of a variant computes the same tiles with the same K order and
the same epilogue program; only the assignment of tiles to persistent CTAs
and the timing differ. Any difference between two launches would be a race in
the barrier protocol (a stage overwritten before its MMAs finished, an
accumulator read before it was complete, a split tile's partial read before
it was written). Shapes span several waves of persistent clusters, ragged
edges, the half-tile tail items and the stream-K split."""
import pytest

pytestmark = pytest.mark.gpu

REPS = 4


def _flat(out):
    if isinstance(out, (tuple, list)):
        return [t for o in out for t in _flat(o)]
    return [] if out is None else [out]


def _cases(coda):
    import torch
    g = torch.Generator(device="cuda").manual_seed(123)

    def bf(*s, std=1.0):
        return (torch.randn(*s, device="cuda", generator=g) * std).bfloat16()

    M, N, K = 4096, 4096, 512
    A, B = bf(M, K), bf(K, N, std=K ** -0.5)
    At, Bt = bf(K, M), bf(N, K, std=K ** -0.5)
    c, s = coda.coda_rope_tables(2048, 128, 1e4)
    X, Wr = bf(2000, 768), bf(768, 3072, std=768 ** -0.5)
    Wgu = bf(768, 2 * 1800, std=768 ** -0.5)
    dY, Wd, GU = bf(2000, 768), bf(1800, 768, std=768 ** -0.5), bf(2000, 2 * 1800)
    x, z, W0 = bf(1500, 1024), bf(1500, 2048), bf(1024, 2048, std=1024 ** -0.5)
    gam = (1 + 0.1 * torch.randn(2048, device="cuda", generator=g)).bfloat16()
    r = torch.rand(1500, device="cuda", generator=g) + 0.5
    sv = torch.rand(1500, device="cuda", generator=g)
    W1 = bf(1024, 2048, std=2048 ** -0.5)          # [d, K]: G = z W1^T is [1500, 1024]
    gam1 = (1 + 0.1 * torch.randn(1024, device="cuda", generator=g)).bfloat16()
    H, Wv = bf(1200, 512), bf(512, 5000, std=512 ** -0.5)
    y = torch.randint(0, 5000, (1200,), device="cuda", dtype=torch.int32, generator=g)
    Ak, Bk = bf(1800, 1096), bf(1096, 3400, std=1096 ** -0.5)
    GUk = bf(1800, 2 * 3400)
    Wdk = bf(3400, 1096, std=1096 ** -0.5)

    def streamk(fn):
        # the stream-K split forced on: split tiles meet through the workspace
        def run():
            coda.coda_set_stream_k(2)
            try:
                return fn()
            finally:
                coda.coda_set_stream_k(1)
        return run
    A8 = torch.randint(0, 256, (2048, 1024), device="cuda", dtype=torch.uint8, generator=g) & 0x77
    B8 = torch.randint(0, 256, (3072, 1024), device="cuda", dtype=torch.uint8, generator=g) & 0x77
    return {
        "gemm": lambda: coda.coda_gemm(A, B),
        "gemm_tA_tB": lambda: coda.coda_gemm(At, Bt, transA=True, transB=True),
        "rope": lambda: coda.coda_gemm_rope(X, Wr, c, s, 128, 2048),
        "swiglu_gu": lambda: coda.coda_gemm_swiglu(X, Wgu, want_gu=True),
        "swiglu_bwd": lambda: coda.coda_gemm_swiglu_bwd(dY, Wd, GU),
        "res_rmsprep": lambda: coda.coda_gemm_res_rmsprep(x, W0, z, gam),
        "rowdot": lambda: coda.coda_gemm_rowdot(x, W0, z, r),
        "rmsnorm_bwd": lambda: coda.coda_gemm_rmsnorm_bwd(z, W1, x, gam1, r, sv),
        "ce_lse": lambda: coda.coda_gemm_ce_lse(H, Wv, y),
        "fp8": lambda: coda.coda_gemm_fp8(A8, B8, 0.03),
        "gemm_streamk": streamk(lambda: coda.coda_gemm(Ak, Bk)),
        "swiglu_bwd_streamk": streamk(lambda: coda.coda_gemm_swiglu_bwd(Ak, Wdk, GUk)),
    }


def test_repeatable(coda):
    import torch
    cases = _cases(coda)
    first = {}
    try:
        for rep in range(REPS):
            for cg in (2, 1):
                coda.coda_set_cta_group(cg)
                # every case once per pass, so each launch follows a different kernel
                for name, fn in cases.items():
                    outs = [t.clone() for t in _flat(fn())]
                    ref = first.setdefault((name, cg), outs)
                    for i, (o, e) in enumerate(zip(outs, ref)):
                        assert torch.equal(o, e), f"{name} output {i}: cta group {cg}, pass {rep} differs"
    finally:
        coda.coda_set_cta_group(0)
    assert coda.coda_device_status(clear=True) == 0
