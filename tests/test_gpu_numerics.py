"""Numerics of the delayed row scale, as a synthetic report.

The pages state that the fused GEMM-RMSNorm-GEMM (delayed r, CODA note, Key
design 1) has a lower relative error than the standard path when both are
compared with a high-precision reference (CODA note, experiments; pith page,
Figure 6, measured on Llama-3 8B layers whose values the figure image holds).
The trained layers are not available, so synthetic problems stand in: the
GEMM-RMSNorm-GEMM configurations of the workloads (N(0,1) activations), and a
residual stream with outlier channels. The float64 oracle is the reference.

Both paths must meet the parity tolerance. Which one is closer is reported
(printed as one JSON line per case) and not gated, since the pages' own
numbers are not extractable."""
import json

import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, dev_bf16, f64

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _rel_fro(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def _rows(M, n, seed):
    if n >= M:
        return np.arange(M)
    r = np.random.default_rng(seed).choice(M, size=n - 2, replace=False)
    return np.unique(np.concatenate([[0, M - 1], r]))


@pytest.mark.parametrize("case", ["tiny_256x512", "chain_8192", "d4096_outlier_channels"])
def test_delayed_row_scale_numerics(coda, case):
    if case == "tiny_256x512":
        p, sample = gen.rms_chain(256, 512, 512, 512, seed=0), 256
    elif case == "chain_8192":
        p, sample = gen.rms_chain(8192, 8192, 8192, 8192, seed=0), 128
    else:
        p, sample = gen.rms_chain_outliers(4096, 4096, 4096, 4096, seed=0), 128
    x, W0, z, g, W1 = (dev_bf16(p[k]) for k in ("x", "W0", "z", "gamma", "W1"))
    M, d = z.shape
    # fused: residual + gamma + partial sums in GEMM1, r from the partials, r applied after GEMM2
    h1, h2, psq = coda.coda_gemm_res_rmsprep(x, W0, z, g)
    r = coda.coda_rms_reduce(psq, d, EPS)
    Y_fused = coda.coda_gemm_rowscale(h2, W1, r)
    # unfused: GEMM, add, RMSNorm (normalised n rounded to bf16), GEMM
    t = coda.coda_gemm(x, W0)
    h1u = coda.coda_unfused_add(t, z)
    n, _ = coda.coda_unfused_rmsnorm(h1u, g, EPS)
    Y_unfused = coda.coda_gemm(n, W1)
    rows = _rows(M, sample, seed=5)
    ref = O.gemm_rms_gemm_fwd(O.bf16(p["x"][rows]), O.bf16(p["W0"]), O.bf16(p["z"][rows]), O.bf16(p["gamma"]),
                              O.bf16(p["W1"]), EPS)["Y"]
    yf, yu = f64(Y_fused[rows]), f64(Y_unfused[rows])
    assert_bf16(yf, ref, f"{case}: fused Y")
    assert_bf16(yu, ref, f"{case}: unfused Y")
    ef, eu = _rel_fro(yf, ref), _rel_fro(yu, ref)
    print(json.dumps({"numerics": case, "rows": int(len(rows)), "rel_fro_fused": ef, "rel_fro_unfused": eu,
                      "unfused_over_fused": eu / ef}))
    assert coda.coda_device_status(clear=True) == 0
