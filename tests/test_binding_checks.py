"""Argument checks of the Python binding: a tensor on the wrong device, of the
wrong dtype or shape, or a caller-provided output of the wrong shape, is
rejected before anything is launched (on the device it would be an
out-of-bounds access). The CPU cases need no GPU and no library."""
import pytest

torch = pytest.importorskip("torch")

import gemm_epilogue_transformer_gb300 as G  # noqa: E402


def _cpu_calls():
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)  # noqa: E731
    f32 = lambda *s: torch.zeros(*s, dtype=torch.float32)  # noqa: E731
    i32 = lambda *s: torch.zeros(*s, dtype=torch.int32)  # noqa: E731
    c, s = f32(64, 64), f32(64, 64)
    return {
        "coda_gemm": lambda: G.coda_gemm(bf(64, 64), bf(64, 64)),
        "coda_gemm_res_rmsprep": lambda: G.coda_gemm_res_rmsprep(bf(64, 64), bf(64, 64), bf(64, 64), bf(64)),
        "coda_rms_reduce": lambda: G.coda_rms_reduce(f32(64, 1), 64, 1e-6),
        "coda_gemm_rowscale": lambda: G.coda_gemm_rowscale(bf(64, 64), bf(64, 64), f32(64)),
        "coda_gemm_swiglu": lambda: G.coda_gemm_swiglu(bf(64, 64), bf(64, 128)),
        "coda_gemm_swiglu_bwd": lambda: G.coda_gemm_swiglu_bwd(bf(64, 64), bf(64, 64), bf(64, 128)),
        "coda_gemm_rope": lambda: G.coda_gemm_rope(bf(64, 64), bf(64, 128), c, s, 128, 128),
        "coda_gemm_rope_bwd": lambda: G.coda_gemm_rope_bwd(bf(64, 64), bf(64, 128), c, s, 128, 128),
        "coda_gemm_ce_lse": lambda: G.coda_gemm_ce_lse(bf(64, 64), bf(64, 256), i32(64)),
        "coda_ce_reduce": lambda: G.coda_ce_reduce(f32(64, 1), f32(64, 1), None, f32(64)),
        "coda_gemm_ce_bwd": lambda: G.coda_gemm_ce_bwd(bf(64, 64), bf(64, 256), i32(64), f32(64), 1.0),
        "coda_gemm_rowdot": lambda: G.coda_gemm_rowdot(bf(64, 64), bf(64, 64), bf(64, 64), f32(64)),
        "coda_rowdot_reduce": lambda: G.coda_rowdot_reduce(f32(64, 1), 64),
        "coda_gemm_rmsnorm_bwd": lambda: G.coda_gemm_rmsnorm_bwd(bf(64, 64), bf(64, 64), bf(64, 64), bf(64),
                                                                 f32(64), f32(64)),
        "coda_colsum_reduce": lambda: G.coda_colsum_reduce(f32(2, 64)),
        "coda_unfused_add": lambda: G.coda_unfused_add(bf(64, 64), bf(64, 64)),
        "coda_unfused_rmsnorm": lambda: G.coda_unfused_rmsnorm(bf(64, 64), bf(64), 1e-6),
        "coda_unfused_rowscale": lambda: G.coda_unfused_rowscale(bf(64, 64), f32(64)),
        "coda_unfused_swiglu": lambda: G.coda_unfused_swiglu(bf(64, 128)),
        "coda_unfused_swiglu_bwd": lambda: G.coda_unfused_swiglu_bwd(bf(64, 64), bf(64, 128)),
        "coda_unfused_rope": lambda: G.coda_unfused_rope(bf(64, 128), c, s, 128, 128),
        "coda_unfused_rope_bwd": lambda: G.coda_unfused_rope_bwd(bf(64, 128), c, s, 128, 128),
        "coda_unfused_ce_fwd": lambda: G.coda_unfused_ce_fwd(bf(64, 256), i32(64)),
        "coda_unfused_ce_bwd": lambda: G.coda_unfused_ce_bwd(bf(64, 256), i32(64), f32(64), 1.0),
        "coda_unfused_rowdot": lambda: G.coda_unfused_rowdot(bf(64, 64), bf(64, 64), 64),
        "coda_unfused_rmsnorm_bwd": lambda: G.coda_unfused_rmsnorm_bwd(bf(64, 64), bf(64, 64), bf(64), f32(64)),
        "coda_gemm_rowscale_rope": lambda: G.coda_gemm_rowscale_rope(bf(64, 64), bf(64, 128), f32(64), c, s, 128,
                                                                     128),
        "coda_gemm_rowscale_swiglu": lambda: G.coda_gemm_rowscale_swiglu(bf(64, 64), bf(64, 128), f32(64)),
        "coda_gemm_swiglu_bwd_rowdot": lambda: G.coda_gemm_swiglu_bwd_rowdot(bf(64, 64), bf(64, 64), bf(64, 128),
                                                                             f32(64)),
        "coda_gemm_rmsnorm_bwd_res": lambda: G.coda_gemm_rmsnorm_bwd_res(bf(64, 64), bf(64, 64), bf(64, 64), bf(64),
                                                                         f32(64), f32(64), bf(64, 64)),
        "coda_rope_bwd_rowdot": lambda: G.coda_rope_bwd_rowdot(bf(64, 128), bf(64, 128), f32(64), c, s, 128, 128,
                                                               64),
        "coda_gemm_fp8": lambda: G.coda_gemm_fp8(torch.zeros(64, 64, dtype=torch.uint8),
                                                 torch.zeros(64, 64, dtype=torch.uint8), 1.0),
    }


@pytest.mark.parametrize("name", sorted(_cpu_calls()))
def test_host_tensors_rejected(name):
    with pytest.raises(TypeError, match="CUDA tensor"):
        _cpu_calls()[name]()


@pytest.mark.gpu
def test_mismatched_shapes_rejected(coda):
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    f32 = lambda *s: torch.zeros(*s, dtype=torch.float32, device="cuda")  # noqa: E731
    c, s = coda.coda_rope_tables(64, 128, 1e4)
    X, W = bf(64, 64), bf(64, 256)
    with pytest.raises(ValueError, match="out"):
        coda.coda_gemm(X, W, out=bf(64, 128))                      # output too small
    with pytest.raises(ValueError, match="out"):
        coda.coda_gemm_rope(X, W, c, s, 128, 256, out=bf(32, 256))
    with pytest.raises(TypeError, match="out"):
        coda.coda_gemm_rope(X, W, c, s, 128, 256, out=f32(64, 256))
    with pytest.raises(ValueError, match="cos and sin"):
        coda.coda_gemm_rope(X, W, c[:, :32].contiguous(), s, 128, 256)
    with pytest.raises(ValueError, match="b must have shape"):
        coda.coda_unfused_add(bf(64, 64), bf(32, 64))              # second operand too small
    with pytest.raises(ValueError, match="gu must have shape"):
        coda.coda_gemm_swiglu_bwd(bf(64, 64), bf(32, 64), bf(64, 32))
    with pytest.raises(ValueError, match="r must have shape"):
        coda.coda_gemm_rowscale_rope(X, W, f32(32), c, s, 128, 256)
    with pytest.raises(ValueError, match="contiguous"):
        coda.coda_unfused_rowdot(bf(64, 128), bf(128, 64).t(), 64)
    assert coda.coda_device_status(clear=True) == 0
