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


# End-to-end MoE output (gate_up -> bf16 h -> q8_1 -> down): the intermediate
# is re-quantized, and an fp32 product (any fp32 accumulation, ~1e-6 relative)
# puts about 0.1% of the bf16 h values on the other side of a rounding tie
# from the fp64 reference; each such flip moves one q8_1 step of h (up to
# 2^-7 of the block maximum) and with it the down product.  So the end-to-end
# check is norm-wise per token at the bf16 bound, with an elementwise guard;
# every stage is also checked elementwise on its own (test_gpu_moe.py).
TOL_MOE_E2E_NORM = 1e-2
TOL_MOE_E2E_ELEM = 5e-2


def assert_close_moe_e2e(y, ref, what=""):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    num = np.linalg.norm(y - ref, axis=-1)
    den = np.maximum(np.linalg.norm(ref, axis=-1), 1e-30)
    rel = np.where(np.linalg.norm(ref, axis=-1) == 0, np.linalg.norm(y, axis=-1), num / den)
    assert rel.max() <= TOL_MOE_E2E_NORM, f"{what}: per-token norm-wise rel err {rel.max():.3e}"
    assert_close(y, ref, TOL_MOE_E2E_ELEM, what)
