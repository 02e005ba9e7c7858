"""Shared helpers of the parity tests (comparison rules, not method arithmetic)."""
import numpy as np

# Tolerances of the final outputs against the oracle's fp64 result:
# |y - r| <= tol * max(|r|, rms of r's row), tol = 1e-3 for fp32 outputs and
# 1e-2 for bf16 outputs (the relative bounds of the hot path's accuracy
# contract; the rms floor keeps outputs that cancel to ~0 from dividing by ~0).
TOL_F32 = 1e-3
TOL_BF16 = 1e-2


def rel_err(y, ref):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt((ref ** 2).mean(axis=-1, keepdims=True))
    floor = np.maximum(np.abs(ref), rms)
    floor = np.where(floor == 0, 1.0, floor)
    return np.abs(y - ref) / floor


def assert_close(y, ref, tol, what=""):
    e = rel_err(y, ref)
    assert np.all(np.isfinite(np.asarray(y, dtype=np.float64))), f"{what}: non-finite output"
    assert e.max() <= tol, f"{what}: max rel err {e.max():.3e} > {tol} (p99 {np.percentile(e, 99):.3e})"
    return e
