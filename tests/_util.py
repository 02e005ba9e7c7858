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


# End-to-end MoE output (gate_up -> bf16 h -> q8_1 -> down) against the full
# oracle chain.  The intermediate h is rounded to bf16 and re-quantized to
# q8_1, so a g or u that differs from the fp64 value in its last bits can put
# h on the other side of a rounding boundary; the q8_1 code then moves by one
# step d = amax/127 of its block, and the down product by w * W[c][i] * d.
# Measured on the full-size block (E = 256, top-8, H = 2048, I = 512):
#   tensor-core path (hi + lo fp16 operands, fp32 accumulation): 0.67% of the
#     bf16 h and 0.04% of the q8_1 codes differ from the oracle's;
#   route-batched MMVQ path (exact int32 block sums): 0.015% / 0.0005%.
# One differing code adds at most about 2.5e-3 of the output row's rms
# (route weight <= 1, |W| <= 4 sigma, d <= 4 sigma_h / 127), and bf16 output
# rounding up to 2^-9 of |y|.  With 1.6 differing codes per output element on
# average on the tensor-core path (8 routes x 512 inputs x 0.0004), seven
# aligned worst-case ones have probability below 1e-6, hence 2e-2 there
# (largest measured: 1.01e-2 over 131072 elements); the MMVQ path, with 80x
# fewer, keeps the bf16 bound 1e-2 (largest measured: 3.9e-3).  The check is
# also norm-wise per token at the bf16 bound, and each stage is checked
# elementwise on its own (test_gpu_moe.py).
TOL_MOE_E2E_NORM = 1e-2
TOL_MOE_E2E_ELEM = 2e-2          # tensor-core grouped GEMMs
TOL_MOE_E2E_ELEM_VEC = 1e-2      # route-batched MMVQ (exact block sums)


def assert_close_moe_e2e(y, ref, what="", elem_tol=TOL_MOE_E2E_ELEM):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    num = np.linalg.norm(y - ref, axis=-1)
    den = np.maximum(np.linalg.norm(ref, axis=-1), 1e-30)
    rel = np.where(np.linalg.norm(ref, axis=-1) == 0, np.linalg.norm(y, axis=-1), num / den)
    assert rel.max() <= TOL_MOE_E2E_NORM, f"{what}: per-token norm-wise rel err {rel.max():.3e}"
    if elem_tol is not None:   # None: the norm-wise bound only (the opt-in single-operand gate_up)
        assert_close(y, ref, elem_tol, what)
