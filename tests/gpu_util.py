"""Helpers for the GPU parity tests: device transfer and the fp32 tolerance check.

Tolerance (stated against the oracle's fp64 result rounded to fp32):
    |y_gpu - y_ref| <= 1e-5 * sum_b |s_a s_w (acc - z_w rs)| + 1e-6
The integer stages (codes, scales, row sums, per-block accumulators) must match bit
for bit.
"""
import numpy as np
import torch

REL_TOL = 1e-5
ABS_TOL = 1e-6


def dev():
    return torch.device("cuda:0")


def to_dev(a):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def inputs_to_dev(d):
    return {k: (to_dev(v) if isinstance(v, np.ndarray) else v) for k, v in d.items()}


def check_y(y_gpu, y_ref, bound, what=""):
    """Assert every output is within tolerance; returns (max abs err, max err / allowed)."""
    y = y_gpu.detach().cpu().numpy().astype(np.float64) if isinstance(y_gpu, torch.Tensor) else y_gpu
    ref = y_ref.astype(np.float32).astype(np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs"
    err = np.abs(y - ref)
    allowed = REL_TOL * bound + ABS_TOL
    bad = err > allowed
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outputs outside tolerance; "
                             f"first {idx.tolist()} err {err[bad][:5]} allowed {allowed[bad][:5]}")
    return float(err.max()), float((err / allowed).max())
