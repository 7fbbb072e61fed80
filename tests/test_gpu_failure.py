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
