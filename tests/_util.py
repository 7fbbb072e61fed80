"""Shared helpers for the parity tests: moving seeded bf16 bits onto the GPU,
reading results back as float64, and the tolerance checks.

Tolerances (written in each assertion through these helpers):
  * bf16 outputs (fp32 accumulation): relative Frobenius error <= 5e-3 and
    max_i |err_i| / (1 + |ref_i|) <= 3e-2;
  * fp32 statistics (r, s, LSE, loss, partials): |err_i| <= 1e-4 * max(|ref_i|,
    rms(ref)) (the rms floor keeps cancelling sums that land near zero from
    turning into a meaningless elementwise relative error);
  * indices: exact.
"""
from __future__ import annotations

import numpy as np

import oracle as O

BF16_FRO = 5e-3
BF16_MAX = 3e-2
STAT_REL = 1e-4


def dev_bf16(bits, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def host_bits(t) -> np.ndarray:
    import torch
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t) -> np.ndarray:
    """bf16 tensor -> float64 via the oracle's own decoder; other dtypes upcast."""
    import torch
    if t.dtype == torch.bfloat16:
        return O.bf16(host_bits(t))
    return t.detach().cpu().numpy().astype(np.float64)


def bf16_errors(got: np.ndarray, ref: np.ndarray):
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    d = got - ref
    fro = np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30)
    mx = float(np.max(np.abs(d) / (1.0 + np.abs(ref)))) if d.size else 0.0
    return float(fro), mx


def assert_bf16(got, ref, name=""):
    got = np.asarray(got, np.float64)
    assert got.shape == np.shape(ref), f"{name}: shape {got.shape} vs {np.shape(ref)}"
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    fro, mx = bf16_errors(got, ref)
    assert fro <= BF16_FRO and mx <= BF16_MAX, f"{name}: rel Frobenius {fro:.3e} (<= {BF16_FRO}), max {mx:.3e} (<= {BF16_MAX})"
    return fro, mx


def assert_stat(got, ref, name="", tol=STAT_REL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    if ref.size == 0:
        return 0.0
    floor = max(float(np.sqrt(np.mean(ref * ref))), 1e-30)
    err = float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))
    assert err <= tol, f"{name}: relative error {err:.3e} > {tol}"
    return err


def col_tile_sums(x: np.ndarray, tile: int = 128) -> np.ndarray:
    """Per-(row, 128-column block) sums: the reference for the epilogue partials."""
    n = x.shape[1]
    return np.stack([x[:, c:c + tile].sum(axis=1) for c in range(0, n, tile)], axis=1) if n else np.zeros((x.shape[0], 0))
