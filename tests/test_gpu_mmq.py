"""GPU parity of the tensor-core MMQ path (m above the MMVQ threshold).

MMQ feeds tcgen05 fp16 operands that hold the dequantized weight and q8_1
values (the exact fp32 value of the blockwise formula), accumulating over K in
fp32.  16-bit outputs use one fp16 operand per side and are held to the 1e-2
bf16 bound; fp32 outputs use hi + lo operands on both sides (three MMAs per K
step) and are held to the 1e-3 bound.
"""
import numpy as np
import pytest
import torch

import oracle
from _util import TOL_BF16, TOL_F32, assert_close
from gguf_block_quantized_quantize_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def g():
    from gguf_block_quantized_quantize_gb300 import build

    build.build()
    import gguf_block_quantized_quantize_gb300 as g

    g.load_library()
    return g


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _weights(wt, n, k, seed, safe=False):
    if safe:
        return synth.safe_blocks(wt, n, k, seed)
    return oracle.quantize_weights(wt, synth.normal((n, k), 0.02, seed))


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
@pytest.mark.parametrize("m", [9, 16, 17, 32, 64, 100, 128, 256, 300])
def test_mmq_bf16_shapes(g, wt, m):
    n, k = 300, 1056 if wt in (oracle.Q8_0, oracle.Q4_0, oracle.MXFP4) else 1024   # ragged n; k % 64 == 32 where it can
    w = _weights(wt, n, k, seed=m, safe=(m % 2 == 1))
    x = synth.activations(m, k, seed=m + 1, dtype=torch.bfloat16)
    ref = oracle.mul_mat(wt, w, k, oracle.quantize_q8_1(x.float().numpy()))
    y = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV))
    assert y.dtype == torch.bfloat16
    assert_close(y.float().cpu().numpy(), ref, TOL_BF16, f"mmq type {wt} m {m}")


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
@pytest.mark.parametrize("m", [12, 40, 200])
def test_mmq_fp32_output(g, wt, m):
    n, k = 257, 2048
    w = _weights(wt, n, k, seed=3)
    x = synth.activations(m, k, seed=4, dtype=torch.float32)
    ref = oracle.mul_mat(wt, w, k, oracle.quantize_q8_1(x.numpy()))
    y = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV))
    assert_close(y.cpu().numpy(), ref, TOL_F32, f"mmq fp32 type {wt}")


def test_mmq_prequantized_and_column_slices(g):
    k, m = 2048, 96
    x = synth.activations(m, k, seed=7, dtype=torch.bfloat16)
    xq = g.gguf_quantize_q8_1(x.to(DEV))
    xq_ref = oracle.quantize_q8_1(x.float().numpy())
    out = torch.zeros(m, 512 + 256, dtype=torch.bfloat16, device=DEV)
    w1, w2 = _weights(oracle.Q4_K, 512, k, 8), _weights(oracle.Q6_K, 256, k, 9)
    g.gguf_mul_mat(_u8(w1), oracle.Q4_K, 512, k, xq, xt=oracle.Q8_1, m=m, out=out[:, :512])
    g.gguf_mul_mat(_u8(w2), oracle.Q6_K, 256, k, xq, xt=oracle.Q8_1, m=m, out=out[:, 512:])
    ref = np.concatenate([oracle.mul_mat(oracle.Q4_K, w1, k, xq_ref), oracle.mul_mat(oracle.Q6_K, w2, k, xq_ref)], 1)
    assert_close(out.float().cpu().numpy(), ref, TOL_BF16, "mmq segments")


def test_mmq_threshold_option(g):
    """m = 8 runs MMVQ by default; with mmvq_max_m = 4 it runs MMQ; both agree."""
    n, k, m = 256, 512, 8
    w = _weights(oracle.Q4_K, n, k, 10)
    x = synth.activations(m, k, seed=11, dtype=torch.bfloat16).to(DEV)
    a = g.gguf_mul_mat(_u8(w), oracle.Q4_K, n, k, x).float()
    g.gguf_set_option("mmvq_max_m", 4)
    try:
        b = g.gguf_mul_mat(_u8(w), oracle.Q4_K, n, k, x).float()
    finally:
        g.gguf_set_option("mmvq_max_m", 8)
    ref = oracle.mul_mat(oracle.Q4_K, w, k, oracle.quantize_q8_1(x.float().cpu().numpy()))
    assert_close(a.cpu().numpy(), ref, TOL_BF16, "mmvq")
    assert_close(b.cpu().numpy(), ref, TOL_BF16, "mmq")


def test_mmq_prefill_q4_k_full_size_sampled(g):
    # prefill MMQ: Q4_K weight 8192 x 2048, bf16 activations M = 8192, bf16 out
    n, k, m = 8192, 2048, 8192
    w = _weights(oracle.Q4_K, n, k, seed=20)
    x = synth.activations(m, k, seed=21, dtype=torch.bfloat16)
    y = g.gguf_mul_mat(_u8(w), oracle.Q4_K, n, k, x.to(DEV))
    rng = np.random.default_rng(22)
    rows = np.sort(rng.choice(n, 48, replace=False))
    toks = np.sort(rng.choice(m, 24, replace=False))
    rows[0], rows[-1], toks[0], toks[-1] = 0, n - 1, 0, m - 1
    ref = oracle.mul_mat(oracle.Q4_K, w[rows], k, oracle.quantize_q8_1(x[toks].float().numpy()))
    got = y[torch.from_numpy(toks).to(DEV)][:, torch.from_numpy(rows).to(DEV)].float().cpu().numpy()
    # row rms for the tolerance floor comes from a full oracle row of the sampled tokens
    assert_close(got, ref, TOL_BF16, "Q4_K 8192x2048 @ 8192")


def test_mmq_lm_head_q6_k_full_size_sampled(g):
    # prefill MMQ: Q6_K weight 248320 x 2048, M = 2048 tokens, bf16 out
    n, k, m = 248320, 2048, 2048
    w = synth.safe_blocks(oracle.Q6_K, n, k, seed=30)
    x = synth.activations(m, k, seed=31, dtype=torch.bfloat16)
    y = g.gguf_mul_mat(_u8(w), oracle.Q6_K, n, k, x.to(DEV))
    rng = np.random.default_rng(32)
    rows = np.sort(rng.choice(n, 40, replace=False))
    toks = np.sort(rng.choice(m, 16, replace=False))
    rows[0], rows[-1], toks[-1] = 0, n - 1, m - 1
    ref = oracle.mul_mat(oracle.Q6_K, w[rows], k, oracle.quantize_q8_1(x[toks].float().numpy()))
    got = y[torch.from_numpy(toks).to(DEV)][:, torch.from_numpy(rows).to(DEV)].float().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert_close(got, ref, TOL_BF16, "Q6_K 248320x2048 @ 2048")


def test_device_error_word_is_clear_after_mmq(g):
    """A normal tensor-core call leaves the error word of the bounded waits at 0."""
    g.gguf_device_errors(clear=True)
    n, k, m = 1000, 2048, 300
    w = _u8(_weights(oracle.Q4_K, n, k, seed=9, safe=True))
    for dt in (torch.bfloat16, torch.float32):
        g.gguf_mul_mat(w, oracle.Q4_K, n, k, synth.activations(m, k, seed=10, dtype=dt).to(DEV))
    assert g.gguf_device_errors(clear=False) == 0
    flag = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    g.gguf_device_errors_async(flag, clear=True)
    assert int(flag.item()) == 0


@pytest.fixture
def stage_option(g):
    saved = g.gguf_get_option("mmq_stage")
    yield
    g.gguf_set_option("mmq_stage", saved)


# shapes whose packed rows the GEMM stages in shared memory by bulk tensor
# copies: 256-value chunks (row bytes a multiple of 16) or whole short rows
@pytest.mark.parametrize("wt,n,k", [(oracle.Q4_K, 300, 1024), (oracle.Q5_K, 257, 2048), (oracle.Q6_K, 300, 2048),
                                    (oracle.Q6_K, 200, 512), (oracle.Q8_0, 333, 1024), (oracle.Q4_0, 129, 1024),
                                    (oracle.MXFP4, 300, 1024)])
@pytest.mark.parametrize("m,dtype", [(12, torch.bfloat16), (100, torch.bfloat16), (300, torch.bfloat16),
                                     (40, torch.float32), (200, torch.float32)])
def test_mmq_staged_weights_against_oracle(g, stage_option, wt, n, k, m, dtype):
    w = _weights(wt, n, k, seed=m + n, safe=(m % 2 == 0))
    x = synth.activations(m, k, seed=m + 7, dtype=dtype)
    ref = oracle.mul_mat(wt, w, k, oracle.quantize_q8_1(x.float().numpy()))
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    ys = []
    for stage in (1, 0):
        g.gguf_set_option("mmq_stage", stage)
        y = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV)).float().cpu().numpy()
        assert_close(y, ref, tol, f"mmq staged={stage} type {wt} n {n} k {k} m {m}")
        ys.append(y)
    # both ways feed the MMA the same operand values; only the order of the
    # fp32 accumulation may differ between the split-K partial sums
    assert_close(ys[0], ys[1], 1e-5 if dtype == torch.float32 else TOL_BF16, "staged vs global loads")


@pytest.fixture
def lib_engine(g):
    """Option mmq_engine = 1 for the test: prefill products with 16-bit
    outputs run as dequantize + library GEMM."""
    g.gguf_set_option("mmq_engine", 1)
    yield
    g.gguf_set_option("mmq_engine", 0)


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
@pytest.mark.parametrize("m,out", [(64, torch.bfloat16), (300, torch.bfloat16), (129, torch.float16)])
def test_mmq_library_engine_against_oracle_and_fused(g, lib_engine, wt, m, out):
    # the dequantize + library GEMM engine against the oracle at the 16-bit
    # bound, and against the fused tensor-core MMQ on the same inputs (the
    # engines differ by accumulation order and, for Q4_K / Q5_K, the min term's
    # use of d_a * sum(q) in place of the stored s_a)
    n, k = 520, 1024
    w = _weights(wt, n, k, seed=m + wt, safe=True)
    x = synth.activations(m, k, seed=m, dtype=out)
    ref = oracle.mul_mat(wt, w, k, oracle.quantize_q8_1(x.float().numpy()))
    y1 = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV)).float().cpu().numpy()
    g.gguf_set_option("mmq_engine", 0)
    y0 = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV)).float().cpu().numpy()
    assert_close(y1, ref, TOL_BF16, f"library engine type {wt} m {m}")
    assert_close(y1, y0, TOL_BF16, f"library engine vs fused MMQ type {wt} m {m}")


def test_mmq_library_engine_keeps_fp32_on_fused_path(g, lib_engine):
    # fp32 outputs need the hi + lo operands of the fused MMQ: the option leaves
    # them on it (the 1e-3 bound holds; split-K sums may differ in order only)
    n, k, m = 300, 1024, 40
    w = _weights(oracle.Q4_K, n, k, seed=7)
    x = synth.activations(m, k, seed=8, dtype=torch.float32)
    ref = oracle.mul_mat(oracle.Q4_K, w, k, oracle.quantize_q8_1(x.numpy()))
    a = g.gguf_mul_mat(_u8(w), oracle.Q4_K, n, k, x.to(DEV)).cpu().numpy()
    g.gguf_set_option("mmq_engine", 0)
    b = g.gguf_mul_mat(_u8(w), oracle.Q4_K, n, k, x.to(DEV)).cpu().numpy()
    assert_close(a, ref, TOL_F32, "fp32 output with mmq_engine = 1")
    assert_close(a, b, 1e-5, "fp32 output with and without the option")
