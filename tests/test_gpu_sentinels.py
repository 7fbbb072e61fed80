"""Unwritten-tile and out-of-bounds sentinels for every fused operator.

Each output buffer is pre-filled with NaN (int32 outputs with -7) and padded
with extra rows (and, for the plain GEMM, extra columns through a leading
dimension larger than N). After one launch on ragged shapes, every element of
the output must have been written (no sentinel left, so no tile or partial
statistic was skipped) and every padding element must still hold the sentinel
(no write past the output's extent). Parity tests alone can miss an unwritten
tile when a reused allocation still holds a correct earlier result."""
import pytest

pytestmark = pytest.mark.gpu

PAD = 32  # padding rows after each output
INT_SENTINEL = -7


@pytest.fixture(params=[1, 2], ids=["cta1", "cta2"])
def cta_group(coda, request):
    coda.coda_set_cta_group(request.param)
    yield request.param
    coda.coda_set_cta_group(0)


def _bf(g, *shape, std=1.0):
    import torch
    return (torch.randn(*shape, device="cuda", generator=g) * std).bfloat16()


class Outs:
    """Sentinel-filled outputs, each the first rows of a padded buffer."""

    def __init__(self):
        self.items = []

    def new(self, rows, cols, dtype):
        import torch
        full = torch.empty((rows + PAD, cols), dtype=dtype, device="cuda")
        if dtype == torch.int32:
            full.fill_(INT_SENTINEL)
        else:
            full.fill_(float("nan"))
        self.items.append((full, rows))
        return full[:rows]

    def check(self, name):
        import torch
        torch.cuda.synchronize()
        for i, (full, rows) in enumerate(self.items):
            body, pad = full[:rows], full[rows:]
            if full.dtype == torch.int32:
                assert not bool((body == INT_SENTINEL).any()), f"{name}: output {i} has unwritten entries"
                assert bool((pad == INT_SENTINEL).all()), f"{name}: output {i} written past its rows"
            else:
                assert not bool(torch.isnan(body.float()).any()), f"{name}: output {i} has unwritten entries"
                assert bool(torch.isnan(pad.float()).all()), f"{name}: output {i} written past its rows"


def _ptr(t):
    return None if t is None else t.data_ptr()


def test_every_output_written_once_and_only_inside(coda, cta_group):
    import torch
    L = coda.lib()
    st = torch.cuda.current_stream().cuda_stream
    g = torch.Generator(device="cuda").manual_seed(17)
    M, K, N = 300, 208, 520          # ragged rows, a partial last column tile, K not a multiple of 64
    nb = coda.coda_num_col_tiles(N)
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32

    # plain GEMM, with padding columns through ldc = N + 8
    A, B = _bf(g, M, K), _bf(g, K, N, std=K ** -0.5)
    full = torch.full((M + PAD, N + 8), float("nan"), dtype=bf, device="cuda")
    assert L.coda_gemm(M, N, K, _ptr(A), K, 0, _ptr(B), N, 0, _ptr(full), N + 8, st) == 0
    torch.cuda.synchronize()
    assert not bool(torch.isnan(full[:M, :N].float()).any()), "gemm: unwritten entries"
    assert bool(torch.isnan(full[:M, N:].float()).all()) and bool(torch.isnan(full[M:].float()).all()), \
        "gemm: written outside C"

    # residual + RMS prep, r, rowscale
    o = Outs()
    z, gam = _bf(g, M, N), (1 + 0.1 * torch.randn(N, device="cuda", generator=g)).bfloat16()
    h1, h2, psq = o.new(M, N, bf), o.new(M, N, bf), o.new(M, nb, f32)
    assert L.coda_gemm_res_rmsprep(M, N, K, _ptr(A), _ptr(B), _ptr(z), _ptr(gam), _ptr(h1), _ptr(h2), _ptr(psq),
                                   st) == 0
    o.check("res_rmsprep")
    r = coda.coda_rms_reduce(psq, N, 1e-6)
    W1 = _bf(g, N, 264, std=N ** -0.5)
    o = Outs()
    Y = o.new(M, 264, bf)
    assert L.coda_gemm_rowscale(M, 264, N, _ptr(h2), _ptr(W1), _ptr(r), _ptr(Y), st) == 0
    o.check("rowscale")

    # SwiGLU forward with GU, and backward
    F = 264
    Wgu = _bf(g, K, 2 * F, std=K ** -0.5)
    o = Outs()
    Aout, GU = o.new(M, F, bf), o.new(M, 2 * F, bf)
    assert L.coda_gemm_swiglu(M, F, K, _ptr(A), _ptr(Wgu), _ptr(Aout), _ptr(GU), st) == 0
    o.check("swiglu")
    dY, Wd = _bf(g, M, K), _bf(g, F, K, std=K ** -0.5)
    o = Outs()
    dGU = o.new(M, 2 * F, bf)
    assert L.coda_gemm_swiglu_bwd(M, F, K, _ptr(dY), _ptr(Wd), _ptr(GU), _ptr(dGU), st) == 0
    o.check("swiglu_bwd")

    # RoPE forward and backward (S a multiple of 32: shared-table path; and not)
    for S in (256, 100):
        c, s = coda.coda_rope_tables(S, 64, 1e4)
        for fn in ("coda_gemm_rope", "coda_gemm_rope_bwd"):
            o = Outs()
            out = o.new(M, 512, bf)
            Wr = _bf(g, K, 512, std=K ** -0.5)
            assert getattr(L, fn)(M, 512, K, _ptr(A), _ptr(Wr), _ptr(c), _ptr(s), S, 64, 256, _ptr(out), st) == 0
            o.check(f"{fn} S={S}")

    # rowdot (dY, dYr, partials) and the RMSNorm backward (dh1, column partials)
    o = Outs()
    dYo, dYr, pdot = o.new(M, N, bf), o.new(M, N, bf), o.new(M, nb, f32)
    assert L.coda_gemm_rowdot(M, N, K, _ptr(A), _ptr(B), _ptr(h2), _ptr(r), _ptr(dYo), _ptr(dYr), _ptr(pdot),
                              st) == 0
    o.check("rowdot")
    s_ = coda.coda_rowdot_reduce(pdot, N)
    W1b = _bf(g, N, N, std=N ** -0.5)  # [d, K] with K = d
    o = Outs()
    rt = coda.coda_num_row_tiles(M)
    dh1, pdg = o.new(M, N, bf), o.new(rt, N, f32)
    assert L.coda_gemm_rmsnorm_bwd(M, N, N, _ptr(dYo), _ptr(W1b), _ptr(h1), _ptr(gam), _ptr(r), _ptr(s_),
                                   _ptr(dh1), _ptr(pdg), st) == 0
    o.check("rmsnorm_bwd")

    # cross-entropy forward partials and dlogits
    V = 1000
    Wv = _bf(g, K, V, std=K ** -0.5)
    y = torch.randint(0, V, (M,), device="cuda", dtype=i32, generator=g)
    nbv = coda.coda_num_col_tiles(V)
    o = Outs()
    pmax, psum, parg, tgt = o.new(M, nbv, f32), o.new(M, nbv, f32), o.new(M, nbv, i32), o.new(M, 1, f32)
    assert L.coda_gemm_ce_lse(M, V, K, _ptr(A), _ptr(Wv), _ptr(y), _ptr(pmax), _ptr(psum), _ptr(parg), _ptr(tgt),
                              st) == 0
    o.check("ce_lse")
    lse = coda.coda_ce_reduce(pmax, psum, parg, tgt[:, 0].contiguous())[0]
    o = Outs()
    dl = o.new(M, V, bf)
    assert L.coda_gemm_ce_bwd(M, V, K, _ptr(A), _ptr(Wv), _ptr(y), _ptr(lse), 1.0 / M, _ptr(dl), st) == 0
    o.check("ce_bwd")
    assert coda.coda_device_status(clear=True) == 0


def test_chain_and_fp8_outputs_written_once_and_only_inside(coda, cta_group):
    """The same sentinel check for the block chain's composed kernels and glue,
    and for the FP8 mainloop variants."""
    import torch
    L = coda.lib()
    st = torch.cuda.current_stream().cuda_stream
    g = torch.Generator(device="cuda").manual_seed(23)
    M, K, d, F = 300, 208, 256, 264
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    r = torch.rand(M, device="cuda", generator=g) + 0.5
    X = _bf(g, M, K)

    c, s = coda.coda_rope_tables(128, 64, 1e4)
    W = _bf(g, K, 3 * d, std=K ** -0.5)
    o = Outs()
    qkv = o.new(M, 3 * d, bf)
    assert L.coda_gemm_rowscale_rope(M, 3 * d, K, _ptr(X), _ptr(W), _ptr(r), _ptr(c), _ptr(s), 128, 64, 2 * d,
                                     _ptr(qkv), st) == 0
    o.check("rowscale_rope")
    dqkv = _bf(g, M, 3 * d)
    o = Outs()
    dqr, s1 = o.new(M, 3 * d, bf), o.new(M, 1, f32)
    assert L.coda_rope_bwd_rowdot(M, 3 * d, _ptr(dqkv), _ptr(qkv), _ptr(r), _ptr(c), _ptr(s), 128, 64, 2 * d, d,
                                  _ptr(dqr), _ptr(s1), st) == 0
    o.check("rope_bwd_rowdot")

    Wgu = _bf(g, K, 2 * F, std=K ** -0.5)
    o = Outs()
    A, GU = o.new(M, F, bf), o.new(M, 2 * F, bf)
    assert L.coda_gemm_rowscale_swiglu(M, F, K, _ptr(X), _ptr(Wgu), _ptr(r), _ptr(A), _ptr(GU), st) == 0
    o.check("rowscale_swiglu")
    gh, Wdn = _bf(g, M, d), _bf(g, F, d, std=d ** -0.5)
    for Kb in (d, 4096):  # both input-ring instantiations (K <= 3072 and above)
        ghk, Wdk = (gh, Wdn) if Kb == d else (_bf(g, M, Kb), _bf(g, F, Kb, std=Kb ** -0.5))
        o = Outs()
        dgur, pdot = o.new(M, 2 * F, bf), o.new(M, coda.coda_num_col_tiles(F), f32)
        assert L.coda_gemm_swiglu_bwd_rowdot(M, F, Kb, _ptr(ghk), _ptr(Wdk), _ptr(GU), _ptr(r), _ptr(dgur),
                                             _ptr(pdot), st) == 0
        o.check(f"swiglu_bwd_rowdot K={Kb}")
        W1 = _bf(g, d, 2 * F, std=(2 * F) ** -0.5) if Kb == d else _bf(g, d, Kb, std=Kb ** -0.5)
        dYr = dgur if Kb == d else _bf(g, M, Kb)
        h, dres = _bf(g, M, d), _bf(g, M, d)
        gam = (1 + 0.1 * torch.randn(d, device="cuda", generator=g)).bfloat16()
        sv = torch.rand(M, device="cuda", generator=g)
        Kr = 2 * F if Kb == d else Kb
        o = Outs()
        dh, pdg = o.new(M, d, bf), o.new(coda.coda_num_row_tiles(M), d, f32)
        assert L.coda_gemm_rmsnorm_bwd_res(M, d, Kr, _ptr(dYr), _ptr(W1), _ptr(h), _ptr(gam), _ptr(r), _ptr(sv),
                                           _ptr(dres), _ptr(dh), _ptr(pdg), st) == 0
        o.check(f"rmsnorm_bwd_res K={Kr}")

    # FP8 (E4M3) mainloop: operands [M,K] and [N,K]; bytes masked away from NaN codes
    def e4m3(*shape):
        return torch.randint(0, 256, shape, device="cuda", dtype=torch.uint8, generator=g) & 0x77
    A8, B8 = e4m3(M, K), e4m3(520, K)
    o = Outs()
    C8 = o.new(M, 520, bf)
    assert L.coda_gemm_fp8(M, 520, K, _ptr(A8), _ptr(B8), 0.01, _ptr(C8), st) == 0
    o.check("gemm_fp8")
    o = Outs()
    R8 = o.new(M, 512, bf)
    assert L.coda_gemm_rope_fp8(M, 512, K, _ptr(A8), _ptr(B8[:512]), 0.01, _ptr(c), _ptr(s), 128, 64, 256,
                                _ptr(R8), st) == 0
    o.check("rope_fp8")
    o = Outs()
    A8o, GU8 = o.new(M, F, bf), o.new(M, 2 * F, bf)
    Wgu8 = e4m3(2 * F, K)
    assert L.coda_gemm_swiglu_fp8(M, F, K, _ptr(A8), _ptr(Wgu8), 0.01, _ptr(A8o), _ptr(GU8), st) == 0
    o.check("swiglu_fp8")
    V = 1000
    Wv8 = e4m3(V, K)
    y = torch.randint(0, V, (M,), device="cuda", dtype=i32, generator=g)
    nbv = coda.coda_num_col_tiles(V)
    o = Outs()
    pmax, psum, parg, tgt = o.new(M, nbv, f32), o.new(M, nbv, f32), o.new(M, nbv, i32), o.new(M, 1, f32)
    assert L.coda_gemm_ce_lse_fp8(M, V, K, _ptr(A8), _ptr(Wv8), 0.01, _ptr(y), _ptr(pmax), _ptr(psum), _ptr(parg),
                                  _ptr(tgt), st) == 0
    o.check("ce_lse_fp8")
    lse = coda.coda_ce_reduce(pmax, psum, parg, tgt[:, 0].contiguous())[0]
    o = Outs()
    dl = o.new(M, V, bf)
    assert L.coda_gemm_ce_bwd_fp8(M, V, K, _ptr(A8), _ptr(Wv8), 0.01, _ptr(y), _ptr(lse), 1.0 / M, _ptr(dl), st) == 0
    o.check("ce_bwd_fp8")
    assert coda.coda_device_status(clear=True) == 0
