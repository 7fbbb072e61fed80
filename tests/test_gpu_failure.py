"""Failure detection on the GPU without a fault: a fill that nothing issues
(a test hook in the producer) makes the MMA issuer's bounded wait run out.
The kernel must report CODA_DEVST_TIMEOUT through the device status word,
return promptly, and leave the context usable for a correct next launch."""
import time

import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, dev_bf16, f64

pytestmark = pytest.mark.gpu

CODA_DEVST_TIMEOUT = 1


@pytest.mark.parametrize("cg", [1, 2], ids=["cta1", "cta2"])
def test_missing_load_times_out_and_context_survives(coda, cg):
    rng = [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(9).spawn(2)]
    M, N, K = 512, 512, 512
    A = gen.normal_bf16(rng[0], (M, K))
    B = gen.normal_bf16(rng[1], (K, N), std=1.0 / np.sqrt(K))
    dA, dB = dev_bf16(A), dev_bf16(B)
    try:
        coda.coda_set_cta_group(cg)
        coda.coda_set_wait_timeout_ns(2_000_000)  # 2 ms
        assert coda.coda_device_status(clear=True) == 0
        coda.coda_test_inject_missing_load()
        t0 = time.perf_counter()
        coda.coda_gemm(dA, dB)
        st = coda.coda_device_status(clear=True)  # synchronises
        elapsed = time.perf_counter() - t0
        assert st & CODA_DEVST_TIMEOUT, f"status {st}"
        assert elapsed < 5.0, f"the aborted launch took {elapsed:.2f} s"
    finally:
        coda.coda_set_wait_timeout_ns(2_000_000_000)
        coda.coda_set_cta_group(0)
    # the hook is one-shot and the context is intact: the same GEMM is correct
    C = coda.coda_gemm(dA, dB)
    assert coda.coda_device_status(clear=True) == 0
    assert_bf16(f64(C), O.matmul(O.bf16(A), O.bf16(B)), "GEMM after the aborted launch")


def _rope_case(coda):
    p = gen.rope_problem(512, 256, 768, seed=4)
    c, s = coda.coda_rope_tables(4096, 128, 10000.0)
    X, W = dev_bf16(p["X"]), dev_bf16(p["W"])
    run = lambda: coda.coda_gemm_rope(X, W, c, s, 128, 512)  # noqa: E731
    ref = O.gemm_rope(O.bf16(p["X"]), O.bf16(p["W"]), np.arange(512), 128, 10000.0, 512)
    return run, ref


def _swiglu_bwd_case(coda):
    p = gen.swiglu_problem(512, 256, 384, seed=5)
    GU = gen.normal_bf16(np.random.default_rng(5), (512, 768))
    dY, Wd, gu = dev_bf16(p["dY"]), dev_bf16(p["Wd"]), dev_bf16(GU)
    run = lambda: coda.coda_gemm_swiglu_bwd(dY, Wd, gu)  # noqa: E731
    ref = O.gemm_swiglu_bwd(O.bf16(p["dY"]), O.bf16(p["Wd"]), O.bf16(GU))["dGU"]
    return run, ref


def _fp8_case(coda):
    import torch
    p = gen.fp8_problem(512, 256, 512, seed=6)
    A = torch.from_numpy(p["A"]).cuda()
    B = torch.from_numpy(p["B"]).cuda()
    alpha = p["sA"] * p["sB"]
    run = lambda: coda.coda_gemm_fp8(A, B, alpha)  # noqa: E731
    ref = O.matmul(O.e4m3(p["A"]), O.e4m3(p["B"]).T) * alpha
    return run, ref


def _streamk_case(coda):
    """More tiles than one wave with the stream-K split forced on: the abort
    hits a launch whose split tiles would meet through the workspace, and the
    next launch (a new epoch for the arrival words) is correct."""
    p = gen.swiglu_problem(1800, 1096, 1700, seed=7)
    X, W = dev_bf16(p["X"]), dev_bf16(p["Wgu"])

    def run():
        coda.coda_set_stream_k(2)
        try:
            return coda.coda_gemm(X, W)
        finally:
            coda.coda_set_stream_k(1)
    ref = O.matmul(O.bf16(p["X"]), O.bf16(p["Wgu"]))
    return run, ref


@pytest.mark.parametrize("case", [_rope_case, _swiglu_bwd_case, _fp8_case, _streamk_case],
                         ids=["rope_shared_tables", "swiglu_bwd_inputs", "fp8_mainloop", "stream_k_split"])
@pytest.mark.parametrize("cg", [1, 2], ids=["cta1", "cta2"])
def test_abort_with_epilogue_inputs_in_flight(coda, cg, case):
    """The same missing fill in a kernel whose epilogue warps filled a shared
    table first (RoPE), in one whose epilogue warps already have TMA input
    boxes in flight (SwiGLU pre-activations), in the FP8 mainloop and with the
    stream-K split: the abort path drains what is in flight, and the context
    stays usable."""
    run, ref = case(coda)
    try:
        coda.coda_set_cta_group(cg)
        coda.coda_set_wait_timeout_ns(2_000_000)
        assert coda.coda_device_status(clear=True) == 0
        coda.coda_test_inject_missing_load()
        t0 = time.perf_counter()
        run()
        st = coda.coda_device_status(clear=True)
        assert st & CODA_DEVST_TIMEOUT, f"status {st}"
        assert time.perf_counter() - t0 < 5.0
    finally:
        coda.coda_set_wait_timeout_ns(2_000_000_000)
        coda.coda_set_cta_group(0)
    out = run()
    assert coda.coda_device_status(clear=True) == 0
    assert_bf16(f64(out), ref, "result after the aborted launch")
