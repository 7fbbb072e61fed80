"""Parity of the unfused comparison kernels (separate HBM-bound element-wise
and normalisation kernels) with the float64 oracle on the inputs they read."""
import numpy as np
import pytest

import coda_inputs as gen
import oracle as O
from _util import assert_bf16, assert_stat, dev_bf16, f64

pytestmark = pytest.mark.gpu


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


@pytest.mark.parametrize("M,N", [(300, 520), (1, 8), (257, 4096)])
def test_add_rowscale(coda, M, N):
    a = gen.normal_bf16(_rng(1), (M, N))
    b = gen.normal_bf16(_rng(2), (M, N))
    out = coda.coda_unfused_add(dev_bf16(a), dev_bf16(b))
    assert_bf16(f64(out), O.bf16(a) + O.bf16(b), "add")
    import torch
    r = torch.from_numpy(np.abs(_rng(3).standard_normal(M)).astype(np.float32) + 0.1).cuda()
    s = coda.coda_unfused_rowscale(dev_bf16(a), r)
    assert_bf16(f64(s), f64(r)[:, None] * O.bf16(a), "rowscale")


@pytest.mark.parametrize("M,d", [(300, 520), (64, 8192), (3, 8), (33, 16384), (40, 20480)])
def test_rmsnorm_fwd_bwd(coda, M, d):
    h = gen.normal_bf16(_rng(4), (M, d))
    g = gen.normal_bf16(_rng(5), (d,), std=0.1, mean=1.0)
    n, r = coda.coda_unfused_rmsnorm(dev_bf16(h), dev_bf16(g), 1e-6)
    ref_n, ref_r = O.rmsnorm(O.bf16(h), O.bf16(g), 1e-6)
    assert_stat(f64(r), ref_r, "r")
    assert_bf16(f64(n), ref_n, "n")
    G = gen.normal_bf16(_rng(6), (M, d))
    dh, pdg = coda.coda_unfused_rmsnorm_bwd(dev_bf16(G), dev_bf16(h), dev_bf16(g), r)
    # textbook form: the statistic is formed from G, gamma and h inside the kernel
    c = np.sum(O.bf16(G) * O.bf16(g)[None, :] * O.bf16(h), axis=1) / d
    s_equiv = f64(r) * c  # the (1/d) rowsum(dY (.) Y) statistic this corresponds to
    ref = O.rmsnorm_bwd(O.bf16(G), O.bf16(h), O.bf16(g), f64(r), s_equiv)
    assert_bf16(f64(dh), ref["dh1"], "dh")
    dg = coda.coda_colsum_reduce(pdg)
    assert_stat(f64(dg), ref["dgamma"], "dgamma")
    rowdot = coda.coda_unfused_rowdot(dev_bf16(G), dev_bf16(h), d)
    assert_stat(f64(rowdot), O.rowdot_stat(O.bf16(G), O.bf16(h), d), "rowdot")


@pytest.mark.parametrize("M,F", [(300, 264), (2, 8)])
def test_swiglu(coda, M, F):
    gu = gen.normal_bf16(_rng(7), (M, 2 * F), std=3.0)
    dA = gen.normal_bf16(_rng(8), (M, F))
    a = coda.coda_unfused_swiglu(dev_bf16(gu))
    assert_bf16(f64(a), O.swiglu(O.bf16(gu)), "swiglu")
    dgu = coda.coda_unfused_swiglu_bwd(dev_bf16(dA), dev_bf16(gu))
    assert_bf16(f64(dgu), O.swiglu_bwd(O.bf16(dA), O.bf16(gu)), "swiglu bwd")


@pytest.mark.parametrize("M,N,hd,rope_cols,S", [(300, 768, 128, 512, 256), (5, 64, 8, 64, 3)])
def test_rope(coda, M, N, hd, rope_cols, S):
    x = gen.normal_bf16(_rng(9), (M, N))
    if hd % 32 == 0:
        c, s = coda.coda_rope_tables(S, hd, 10000.0)
    else:
        import torch
        ang = O.rope_angles(np.arange(S), hd, 10000.0)
        c = torch.from_numpy(np.cos(ang).astype(np.float32)).cuda()
        s = torch.from_numpy(np.sin(ang).astype(np.float32)).cuda()
    pos = np.arange(M) % S
    t = dev_bf16(x)
    coda.coda_unfused_rope(t, c, s, hd, rope_cols)
    assert_bf16(f64(t), O.rope(O.bf16(x), pos, hd, 10000.0, rope_cols), "rope")
    t = dev_bf16(x)
    coda.coda_unfused_rope_bwd(t, c, s, hd, rope_cols)
    assert_bf16(f64(t), O.rope_bwd(O.bf16(x), pos, hd, 10000.0, rope_cols), "rope bwd")


@pytest.mark.parametrize("M,V", [(300, 1000), (4, 32768), (2, 8), (13, 4104)])
def test_ce(coda, M, V):
    import torch
    L = gen.normal_bf16(_rng(10), (M, V), std=3.0)
    y = _rng(11).integers(0, V, M, dtype=np.int32)
    lse, loss_row, loss_mean, am = coda.coda_unfused_ce_fwd(dev_bf16(L), torch.from_numpy(y).cuda())
    ref = O.ce_fwd(O.bf16(L), y)
    assert_stat(f64(lse), ref["lse"], "lse")
    assert_stat(f64(loss_row), ref["loss_row"], "loss_row")
    assert abs(float(loss_mean.item()) - ref["loss_mean"]) <= 1e-4 * abs(ref["loss_mean"])
    # bf16 logits can tie exactly: the lowest index must win
    assert np.array_equal(am.cpu().numpy(), ref["argmax"])
    dl = coda.coda_unfused_ce_bwd(dev_bf16(L), torch.from_numpy(y).cuda(), lse, 1.0 / M)
    assert_bf16(f64(dl), O.ce_bwd(O.bf16(L), y, f64(lse), 1.0 / M), "dl")


@pytest.mark.parametrize("M,d", [(40, 520), (33, 8192)])
def test_rmsnorm_bwd_partials_4byte_aligned(coda, M, d):
    """The dgamma partials may start on any 4-byte boundary (the entry point
    checks 4-byte alignment only): results bitwise equal to an aligned call."""
    import torch
    h = dev_bf16(gen.normal_bf16(_rng(12), (M, d)))
    g = dev_bf16(gen.normal_bf16(_rng(13), (d,), std=0.1, mean=1.0))
    G = dev_bf16(gen.normal_bf16(_rng(14), (M, d)))
    _, r = coda.coda_unfused_rmsnorm(h, g, 1e-6)
    dh_ref, pdg_ref = coda.coda_unfused_rmsnorm_bwd(G, h, g, r)
    rows = coda.coda_num_row_tiles(M)
    buf = torch.full((rows * d + 1,), float("nan"), dtype=torch.float32, device=G.device)
    pdg = buf[1:].view(rows, d)  # 4 bytes past a 256-byte boundary
    assert pdg.data_ptr() % 16 == 4
    dh = torch.empty_like(G)
    rc = coda.lib().coda_unfused_rmsnorm_bwd(M, d, G.data_ptr(), h.data_ptr(), g.data_ptr(), r.data_ptr(),
                                            dh.data_ptr(), pdg.data_ptr(), None)
    assert rc == 0, coda.lib().coda_last_error()
    torch.cuda.synchronize()
    assert torch.equal(dh, dh_ref)
    assert torch.equal(pdg, pdg_ref)
