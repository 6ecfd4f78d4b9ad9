"""Tolerances and comparison helpers for the GPU-vs-oracle parity tests.

Tolerances: bf16 inputs -> O max |err| <= 1e-2 and mean |err| <= 1e-3, lse
within 1e-3 absolute; fp32 path -> 1e-5 on O and lse. Rows that see no key
must come back as O = 0 and lse = -inf exactly.
"""

import numpy as np
import torch

BF16_O_MAX = 1e-2
BF16_O_MEAN = 1e-3
LSE_ABS = 1e-3
F32_TOL = 1e-5


def _np64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, *, o_max=BF16_O_MAX, o_mean=BF16_O_MEAN, lse_abs=LSE_ABS, what=""):
    """Element-wise check of O and lse against the oracle's."""
    o = _np64(o_gpu)
    l = _np64(lse_gpu)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    lse_ref = np.asarray(lse_ref, dtype=np.float64)
    assert o.shape == o_ref.shape, (what, o.shape, o_ref.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    assert err.max() <= o_max, f"{what}: O max |err| {err.max():.3e} > {o_max}"
    assert err.mean() <= o_mean, f"{what}: O mean |err| {err.mean():.3e} > {o_mean}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(l)), f"{what}: -inf rows differ"
    assert np.all(l[~fin] == -np.inf), f"{what}: rows without keys must have lse = -inf"
    if fin.any():
        le = np.abs(l[fin] - lse_ref[fin])
        assert le.max() <= lse_abs, f"{what}: lse max |err| {le.max():.3e} > {lse_abs}"
    return float(err.max()), float(err.mean())


def compare_f32(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    return compare(o_gpu, lse_gpu, o_ref, lse_ref, o_max=F32_TOL, o_mean=F32_TOL, lse_abs=F32_TOL, what=what)
