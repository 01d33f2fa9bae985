"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances (stated for the bf16 outputs against the float64 oracle): max-abs
2e-2 and mean-abs 2e-3 on O, 1e-3 absolute on the natural-log LSE.
"""
import numpy as np

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_o(got, want, what=""):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - want)
    assert err.max() <= O_MAX_ABS, f"{what}: max abs err {err.max():.4g} at {np.unravel_index(err.argmax(), err.shape)}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: mean abs err {err.mean():.4g}"
    return float(err.max()), float(err.mean())


def check_lse(got, want, what=""):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape
    err = np.abs(got - want)
    assert err.max() <= LSE_ABS, f"{what}: lse max abs err {err.max():.4g}"
    return float(err.max())
