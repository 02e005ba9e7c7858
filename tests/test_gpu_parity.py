"""GPU parity of the CUDA path against the oracle (through the C ABI).

Bit-exact: q8_1 quantization, dequantize / get_rows, per-block int32 dots.
Within tolerance (fp32 1e-3, bf16 1e-2 of max(|r|, row rms)): mul_mat.
Shapes span several CTAs and ragged tails; the full-size decode shapes are
checked on a sampled subset of output rows that the oracle computes.
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
    assert torch.cuda.is_available()
    return g


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _bits(t):
    """uint16 bit patterns of a bf16 / f16 CUDA tensor."""
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- quantize

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("m,k", [(1, 32), (37, 4096), (8, 14336), (300, 2048)])
def test_quantize_q8_1_bit_exact(g, dtype, m, k):
    x = synth.activations(m, k, seed=m + k, dtype=dtype)
    x[0, :32] = 0                       # all-zero block
    if k >= 64:
        x[0, 32:64] = torch.linspace(-3.5, 3.5, 32).to(dtype)   # ties after scaling
    ref = oracle.quantize_q8_1(x.float().numpy())
    got = g.gguf_quantize_q8_1(x.to(DEV)).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


def test_quantize_q8_1_strided_rows(g):
    base = synth.activations(16, 1024 + 64, seed=5, dtype=torch.bfloat16)
    x = base[:, 32:32 + 1024]           # row stride 1088, misaligned start
    ref = oracle.quantize_q8_1(x.float().contiguous().numpy())
    got = g.gguf_quantize_q8_1(base.to(DEV)[:, 32:32 + 1024]).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


def test_quantize_q8_1_hand_values(g):
    x = torch.zeros(1, 64)
    x[0, 0], x[0, 1], x[0, 2], x[0, 7] = 127.0, 2.5, -2.5, 126.5
    x[0, 32 + 5], x[0, 32 + 6] = -254.0, 1.0
    got = g.gguf_quantize_q8_1(x.to(DEV)).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.quantize_q8_1(x.numpy()))
    d, s, q = oracle.q8_1_fields(got)
    assert d[0, 0] == 0x3C00 and q[0, 0, 1] == 3 and q[0, 0, 2] == -3 and q[0, 0, 7] == 127
    assert d[0, 1] == 0x4000 and q[0, 1, 5] == -127 and q[0, 1, 6] == 1


# ---------------------------------------------------------------- dequantize / get_rows

def _weights(wt, n, k, seed, safe=False):
    if safe:
        return synth.safe_blocks(wt, n, k, seed)
    return oracle.quantize_weights(wt, synth.normal((n, k), 0.02, seed) * synth.lognormal_row_scale(n, seed + 1))


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
@pytest.mark.parametrize("safe", [False, True])
@pytest.mark.parametrize("ot", [oracle.F32, oracle.BF16, oracle.F16])
def test_dequantize_bit_exact(g, wt, safe, ot):
    n, k = 37, 800 if wt in (oracle.Q8_0, oracle.Q4_0, oracle.MXFP4) else 768
    w = _weights(wt, n, k, seed=7, safe=safe)
    ref = oracle.dequantize(wt, w, k, ot)
    out = g.gguf_dequantize(_u8(w), wt, n, k, out_dtype={0: torch.float32, 30: torch.bfloat16, 1: torch.float16}[ot])
    got = out.cpu().numpy() if ot == oracle.F32 else _bits(out)
    np.testing.assert_array_equal(got.view(np.uint32) if ot == oracle.F32 else got,
                                  ref.view(np.uint32) if ot == oracle.F32 else ref)


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
def test_dequantize_odd_rows_unaligned_blocks(g, wt):
    # K = one block per row: Q6_K (210 B), Q8_0 (34 B) and Q4_0 (18 B) rows
    # alternate alignment; MXFP4 rows (17 B) start at every byte offset
    k = 32 if wt in (oracle.Q8_0, oracle.Q4_0, oracle.MXFP4) else 256
    w = _weights(wt, 33, k, seed=8, safe=True)
    ref = oracle.dequantize(wt, w, k, oracle.F32)
    got = g.gguf_dequantize(_u8(w), wt, 33, k).cpu().numpy()
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
def test_get_rows_bit_exact(g, wt):
    rows, k = 1000, 512
    w = _weights(wt, rows, k, seed=9, safe=True)
    ids = np.array([0, 999, 3, 3, -1, 1000, 517, 42], dtype=np.int32)
    ref = oracle.get_rows(wt, w, k, ids, oracle.BF16)
    got = _bits(g.gguf_get_rows(_u8(w), wt, rows, k, _u8(ids), out_dtype=torch.bfloat16))
    np.testing.assert_array_equal(got, ref)


def test_get_rows_llama_embedding_shape(g):
    # tied embedding table 128256 x 3072 (Q6_K), ids at both ends
    rows, k = 128256, 3072
    w = synth.safe_blocks(oracle.Q6_K, rows, k, seed=10)
    ids = np.array([0, 128255, 64000, 1, 77777, 128254, 5, 99999], dtype=np.int32)
    ref = oracle.get_rows(oracle.Q6_K, w, k, ids, oracle.BF16)
    got = _bits(g.gguf_get_rows(_u8(w), oracle.Q6_K, rows, k, _u8(ids), out_dtype=torch.bfloat16))
    np.testing.assert_array_equal(got, ref)


# ---------------------------------------------------------------- block dots

@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
def test_block_dots_bit_exact(g, wt):
    n, k, m = 19, 1024, 3
    w = _weights(wt, n, k, seed=11, safe=True)
    x = synth.activations(m, k, seed=12, dtype=torch.float32)
    xq = oracle.quantize_q8_1(x.numpy())
    ref = oracle.block_dots(wt, w, k, xq)
    got = g.gguf_debug_block_dots(_u8(w), wt, n, k, _u8(xq), m).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


# ---------------------------------------------------------------- mul_mat (MMVQ)

@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("safe", [False, True])
def test_mmvq_fp32(g, wt, m, safe):
    n, k = 301, 2048
    w = _weights(wt, n, k, seed=20 + m, safe=safe)
    x = synth.activations(m, k, seed=30 + m, dtype=torch.float32)
    ref = oracle.mul_mat(wt, w, k, oracle.quantize_q8_1(x.numpy()))
    y = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV)).cpu().numpy()
    assert_close(y, ref, TOL_F32, f"mmvq type {wt} m {m}")


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
@pytest.mark.parametrize("k", [256, 768, 3072, 8192, 16384])
@pytest.mark.parametrize("m", [1, 4, 7])
def test_mmvq_k_range_bf16(g, wt, k, m):
    # covers every CTA shape: 64-value pieces up to 256 threads, 32-value
    # pieces up to 512 threads, 1 or 2 threads per piece, ragged warps
    n = 129
    w = _weights(wt, n, k, seed=k, safe=True)
    x = synth.activations(m, k, seed=k + 1, dtype=torch.bfloat16)
    ref = oracle.mul_mat(wt, w, k, oracle.quantize_q8_1(x.float().numpy()))
    y = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV))
    assert y.dtype == torch.bfloat16        # output in the activation dtype
    assert_close(y.float().cpu().numpy(), ref, TOL_BF16, f"mmvq bf16 type {wt} k {k} m {m}")


@pytest.mark.parametrize("wt", [oracle.Q4_0, oracle.MXFP4])
@pytest.mark.parametrize("k", [32, 96, 2080, 16352])
@pytest.mark.parametrize("m", [1, 3, 5, 8])
def test_mmvq_two_block_pieces_odd_block_count(g, wt, k, m):
    # Q4_0 / MXFP4 pieces are block pairs: an odd number of blocks per row
    # leaves a last piece of one block (k = 32: a single half piece; 16352:
    # 511 blocks); MXFP4 rows of an odd number of blocks start at odd bytes
    n = 197
    w = _weights(wt, n, k, seed=k + m, safe=True)
    x = synth.activations(m, k, seed=k - m, dtype=torch.float32)
    ref = oracle.mul_mat(wt, w, k, oracle.quantize_q8_1(x.numpy()))
    y = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV)).cpu().numpy()
    assert_close(y, ref, TOL_F32, f"mmvq type {wt} k {k} m {m}")


@pytest.mark.parametrize("wt", [oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.Q8_0, oracle.Q4_0, oracle.MXFP4])
@pytest.mark.parametrize("k", [256, 1024, 3072, 8192])
@pytest.mark.parametrize("m", [5, 8])
def test_mmvq_tensor_core_vs_dp4a(g, wt, k, m):
    # 5..8 tokens of Q4_K / Q5_K / Q8_0 / Q4_0 / MXFP4 rows (n >= 2048; MXFP4
    # rows of whole 512-value items) and of Q6_K rows (n >= 32768) run on the
    # tensor-core MMVQ by default; the dp4a kernel (option mmvq_tc = 0)
    # computes the same formula
    n = 32768 + 37 if wt == oracle.Q6_K else 2100
    if wt == oracle.Q6_K and k > 1024:
        pytest.skip("tall Q6_K rows: k up to 1024 keeps the oracle fast")
    w = _weights(wt, n, k, seed=k + m)
    x = synth.activations(m, k, seed=k, dtype=torch.float32)
    ref = oracle.mul_mat(wt, w, k, oracle.quantize_q8_1(x.numpy()))
    a = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV)).cpu().numpy()
    g.gguf_set_option("mmvq_tc", 0)
    try:
        b = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV)).cpu().numpy()
    finally:
        g.gguf_set_option("mmvq_tc", 1)
    assert_close(a, ref, TOL_F32, f"tensor-core mmvq type {wt} k {k} m {m}")
    assert_close(b, ref, TOL_F32, f"dp4a mmvq type {wt} k {k} m {m}")


@pytest.mark.parametrize("m", [9, 12, 16, 17, 24, 32])
@pytest.mark.parametrize("n,k", [(300, 256), (2100, 3072), (700, 4096)])
def test_mmvq_wide_tensor_core(g, m, n, k):
    # 9..32 tokens of Q4_K rows: one tensor-core MMVQ launch with 2 or 4
    # n-tiles (option mmvq_tc_max_m at 32); with the option at 8 the same
    # product runs on MMQ, and both match the oracle
    w = _weights(oracle.Q4_K, n, k, seed=m + n)
    x = synth.activations(m, k, seed=k + m, dtype=torch.float32)
    ref = oracle.mul_mat(oracle.Q4_K, w, k, oracle.quantize_q8_1(x.numpy()))
    saved = g.gguf_get_option("mmvq_tc_max_m")
    try:
        g.gguf_set_option("mmvq_tc_max_m", 32)
        a = g.gguf_mul_mat(_u8(w), oracle.Q4_K, n, k, x.to(DEV)).cpu().numpy()
        g.gguf_set_option("mmvq_tc_max_m", 8)
        b = g.gguf_mul_mat(_u8(w), oracle.Q4_K, n, k, x.to(DEV)).cpu().numpy()
    finally:
        g.gguf_set_option("mmvq_tc_max_m", saved)
    assert_close(a, ref, TOL_F32, f"wide mmvq m {m} n {n} k {k}")
    assert_close(b, ref, TOL_F32, f"mmq m {m} n {n} k {k}")


def _q4_k_plain_nibbles(nib):
    # Q4_K rows with d = 1, dmin = 0 and every sub-block scale 1, min 0: the
    # blocks hold the nibbles themselves (chunk c of 64 values: byte i has
    # value 64c + i in its low and 64c + 32 + i in its high nibble)
    n, k = nib.shape
    blk = np.zeros((n, k // 256, 144), np.uint8)
    blk[:, :, 1] = 0x3C                                   # d = fp16 1.0 (0x3C00)
    blk[:, :, 4:8] = 1                                    # scales of sub-blocks 0..3
    blk[:, :, 12:16] = 1                                  # scales of sub-blocks 4..7 (low bits)
    q = nib.reshape(n, k // 256, 4, 2, 32).astype(np.uint8)
    blk[:, :, 16:] = (q[:, :, :, 0, :] | (q[:, :, :, 1, :] << 4)).reshape(n, k // 256, 128)
    return blk.reshape(n, -1)


@pytest.mark.parametrize("m", [5, 8, 16])
def test_mmvq_tensor_core_exact_integer_sums(g, m):
    # With plain-nibble Q4_K rows and integer activations whose every 32-block
    # reaches 127 (so d_a = 1 and q = x), y is the integer product W . X, below
    # 2^24 and so exact in fp32.  The tensor-core MMVQ sums every block exactly
    # and combines the sums in fp32 without rounding here, so y must match the
    # int64 product bit for bit (5..8 tokens: one n-tile; 16 tokens: two).
    n, k = 2048, 4096
    rng = np.random.default_rng(m)
    nib = rng.integers(0, 16, size=(n, k), dtype=np.int64)
    xi = rng.integers(-127, 128, size=(m, k), dtype=np.int64)
    xi[:, ::32] = 127
    w = _q4_k_plain_nibbles(nib)
    assert np.array_equal(oracle.dequantize_f32(oracle.Q4_K, w, k), nib.astype(np.float32))
    want = (xi @ nib.T).astype(np.float64)
    assert np.abs(want).max() < 2 ** 24
    x = torch.from_numpy(xi.astype(np.float32))
    assert np.array_equal(oracle.mul_mat(oracle.Q4_K, w, k, oracle.quantize_q8_1(xi.astype(np.float32))), want)
    y = g.gguf_mul_mat(_u8(w), oracle.Q4_K, n, k, x.to(DEV)).cpu().numpy()
    assert np.array_equal(y.astype(np.float64), want), f"max diff {np.abs(y - want).max()}"


def _q5_k_plain(q5):
    # Q5_K rows with d = 1, dmin = 0, every sub-block scale 1 and min 0: the
    # blocks hold the 5-bit quants themselves (value 64c + 32h + l of a block:
    # low 4 bits in the nibble h of byte 32c + l, fifth bit in bit 2c + h of
    # high-bit byte l)
    n, k = q5.shape
    v = q5.reshape(n, k // 256, 4, 2, 32).astype(np.uint8)     # [row][sb][c][h][l]
    blk = np.zeros((n, k // 256, 176), np.uint8)
    blk[:, :, 1] = 0x3C                                         # d = fp16 1.0
    blk[:, :, 4:8] = 1
    blk[:, :, 12:16] = 1
    qh = np.zeros((n, k // 256, 32), np.uint8)
    for c in range(4):
        for h in range(2):
            qh |= ((v[:, :, c, h, :] >> 4) & 1) << (2 * c + h)
    blk[:, :, 16:48] = qh
    blk[:, :, 48:] = ((v[:, :, :, 0, :] & 15) | ((v[:, :, :, 1, :] & 15) << 4)).reshape(n, k // 256, 128)
    return blk.reshape(n, -1)


@pytest.mark.parametrize("m", [5, 8])
@pytest.mark.parametrize("n", [2048, 2061])
def test_mmvq_tensor_core_q5_k_exact_integer_sums(g, m, n):
    # Q5_K rows with unit scales, zero mins and integer activations whose every
    # 32-block reaches 127 (d_a = 1, q = x): y is the integer product q5 . X,
    # below 2^24, so the tensor-core MMVQ must match the int64 product bit for
    # bit (2061 rows: a ragged last 16-row tile)
    k = 1024
    rng = np.random.default_rng(m + n)
    q5 = rng.integers(0, 32, size=(n, k), dtype=np.int64)
    xi = rng.integers(-127, 128, size=(m, k), dtype=np.int64)
    xi[:, ::32] = 127
    w = _q5_k_plain(q5)
    assert np.array_equal(oracle.dequantize_f32(oracle.Q5_K, w, k), q5.astype(np.float32))
    want = (xi @ q5.T).astype(np.float64)
    assert np.abs(want).max() < 2 ** 24
    y = g.gguf_mul_mat(_u8(w), oracle.Q5_K, n, k, torch.from_numpy(xi.astype(np.float32)).to(DEV)).cpu().numpy()
    assert np.array_equal(y.astype(np.float64), want), f"max diff {np.abs(y - want).max()}"


def _q8_0_plain(q8):
    # Q8_0 rows with d = 1: the blocks hold the int8 quants themselves
    n, k = q8.shape
    blk = np.zeros((n, k // 32, 34), np.uint8)
    blk[:, :, 1] = 0x3C                                         # d = fp16 1.0
    blk[:, :, 2:] = q8.reshape(n, k // 32, 32).astype(np.int8).view(np.uint8)
    return blk.reshape(n, -1)


def _mxfp4_plain(codes):
    # MXFP4 rows with exponent byte 128 (scale 2^(128-127) on e2m1, so a code's
    # value is the integer 2 * e2m1(code)); code l of a block in byte l (low
    # nibble, l < 16) or l - 16 (high)
    n, k = codes.shape
    v = codes.reshape(n, k // 32, 2, 16).astype(np.uint8)
    blk = np.zeros((n, k // 32, 17), np.uint8)
    blk[:, :, 0] = 128
    blk[:, :, 1:] = v[:, :, 0, :] | (v[:, :, 1, :] << 4)
    return blk.reshape(n, -1)


def _q4_0_plain(q4):
    # Q4_0 rows with d = 1: value l of a block is q4 - 8, its nibble in byte
    # l (low, l < 16) or l - 16 (high)
    n, k = q4.shape
    v = q4.reshape(n, k // 32, 2, 16).astype(np.uint8)
    blk = np.zeros((n, k // 32, 18), np.uint8)
    blk[:, :, 1] = 0x3C
    blk[:, :, 2:] = v[:, :, 0, :] | (v[:, :, 1, :] << 4)
    return blk.reshape(n, -1)


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.MXFP4])
@pytest.mark.parametrize("m", [5, 8])
@pytest.mark.parametrize("n", [2048, 2061])
def test_mmvq_tensor_core_small_block_exact_integer_sums(g, wt, m, n):
    # Q8_0 / Q4_0 rows with d = 1, MXFP4 rows with unit scale, and integer
    # activations whose every 32-block reaches 127 (d_a = 1, q = x): y is the
    # integer product, below 2^24, so the tensor-core MMVQ must match the
    # int64 product bit for bit (2061 rows: a ragged last 16-row tile)
    k = 512
    rng = np.random.default_rng(m + n + wt)
    if wt == oracle.Q8_0:
        qv = rng.integers(-128, 128, size=(n, k), dtype=np.int64)   # the full int8 range
        w, vals = _q8_0_plain(qv), qv
    elif wt == oracle.Q4_0:
        qv = rng.integers(0, 16, size=(n, k), dtype=np.int64)
        w, vals = _q4_0_plain(qv), qv - 8
    else:
        w = _mxfp4_plain(rng.integers(0, 16, size=(n, k), dtype=np.int64))
        vals = oracle.dequantize_f32(wt, w, k).astype(np.int64)
    xi = rng.integers(-127, 128, size=(m, k), dtype=np.int64)
    xi[:, ::32] = 127
    assert np.array_equal(oracle.dequantize_f32(wt, w, k), vals.astype(np.float32))
    want = (xi @ vals.T).astype(np.float64)
    assert np.abs(want).max() < 2 ** 24
    y = g.gguf_mul_mat(_u8(w), wt, n, k, torch.from_numpy(xi.astype(np.float32)).to(DEV)).cpu().numpy()
    assert np.array_equal(y.astype(np.float64), want), f"max diff {np.abs(y - want).max()}"


def _q6_k_plain(q6):
    # Q6_K rows with d = 1 and every scale 1: the blocks hold q6 - 32 (q6 in
    # 0..63); value 128h + 32q + l of a block takes its low 4 bits from
    # ql[64h + 32(q & 1) + l] (low nibble for q < 2, high for q >= 2) and its
    # high 2 bits from bits 2q, 2q + 1 of qh[32h + l]
    n, k = q6.shape
    v = q6.reshape(n, k // 256, 2, 4, 32).astype(np.uint8)     # [row][sb][h][q][l]
    ql = np.zeros((n, k // 256, 2, 2, 32), np.uint8)            # [row][sb][h][q & 1][l]
    qh = np.zeros((n, k // 256, 2, 32), np.uint8)
    for q in range(4):
        ql[:, :, :, q & 1, :] |= (v[:, :, :, q, :] & 15) << (4 * (q >> 1))
        qh |= (v[:, :, :, q, :] >> 4) << (2 * q)
    blk = np.zeros((n, k // 256, 210), np.uint8)
    blk[:, :, :128] = ql.reshape(n, k // 256, 128)
    blk[:, :, 128:192] = qh.reshape(n, k // 256, 64)
    blk[:, :, 192:208] = 1
    blk[:, :, 209] = 0x3C                                      # d = fp16 1.0 (0x3C00)
    return blk.reshape(n, -1)


@pytest.mark.parametrize("m", [5, 8])
@pytest.mark.parametrize("n", [32768, 32781])
def test_mmvq_tensor_core_q6_k_exact_integer_sums(g, m, n):
    # Q6_K rows with unit scales and integer activations whose every 32-block
    # reaches 127 (d_a = 1, q = x): y is the integer product (q6 - 32) . X,
    # below 2^24, so the tensor-core MMVQ (u8 quants, the 32 * sum correction,
    # int32 scale sums) must match the int64 product bit for bit.  32781 rows:
    # a ragged last tile and the guarded end of the view.
    k = 512
    rng = np.random.default_rng(m + n)
    q6 = rng.integers(0, 64, size=(n, k), dtype=np.int64)
    xi = rng.integers(-127, 128, size=(m, k), dtype=np.int64)
    xi[:, ::32] = 127
    w = _q6_k_plain(q6)
    assert np.array_equal(oracle.dequantize_f32(oracle.Q6_K, w, k), (q6 - 32).astype(np.float32))
    want = (xi @ (q6 - 32).T).astype(np.float64)
    assert np.abs(want).max() < 2 ** 24
    y = g.gguf_mul_mat(_u8(w), oracle.Q6_K, n, k, torch.from_numpy(xi.astype(np.float32)).to(DEV)).cpu().numpy()
    assert np.array_equal(y.astype(np.float64), want), f"max diff {np.abs(y - want).max()}"


@pytest.mark.parametrize("wt,n,k", [(oracle.Q6_K, 40000, 3072), (oracle.Q4_K, 20000, 3072),
                                    (oracle.Q5_K, 20000, 3072), (oracle.Q4_0, 20000, 4096),
                                    (oracle.MXFP4, 20000, 4128)])
@pytest.mark.parametrize("m", [1, 2, 8])
def test_mmvq_tall_sampled(g, wt, n, k, m):
    # tall matrices take the R = 1 / R = 4 row groupings; rows sampled for the oracle
    w = synth.safe_blocks(wt, n, k, seed=n + m)
    x = synth.activations(m, k, seed=m, dtype=torch.float32)
    y = g.gguf_mul_mat(_u8(w), wt, n, k, x.to(DEV)).cpu().numpy()
    rows = np.sort(np.random.default_rng(m).choice(n, 64, replace=False))
    rows[0], rows[-1] = 0, n - 1
    ref = oracle.mul_mat(wt, w[rows], k, oracle.quantize_q8_1(x.numpy()))
    assert_close(y[:, rows], ref, TOL_F32, f"mmvq tall type {wt} m {m}")


def test_mmvq_q8_0_config(g):
    # Q8_0 512 x 1024, X 8 x 1024 fp32 ~ N(0,1), output 8 x 512 fp32
    wf = synth.normal((512, 1024), 0.02, seed=0)
    w = oracle.quantize_weights(oracle.Q8_0, wf)
    x = synth.activations(8, 1024, seed=1, dtype=torch.float32)
    xq = oracle.quantize_q8_1(x.numpy())
    ref = oracle.mul_mat(oracle.Q8_0, w, 1024, xq)
    y = g.gguf_mul_mat(_u8(w), oracle.Q8_0, 512, 1024, x.to(DEV))
    assert y.shape == (8, 512) and y.dtype == torch.float32
    assert_close(y.cpu().numpy(), ref, TOL_F32, "Q8_0 512x1024 m=8")


@pytest.mark.parametrize("n", [4096, 14336])
@pytest.mark.parametrize("m", [1, 2, 4, 8])
def test_mmvq_q4_k_decode_full_size_sampled(g, n, m):
    # decode MMVQ shapes: Q4_K n x 4096 from N(0, 0.02), bf16 activations
    k = 4096
    w = oracle.quantize_weights(oracle.Q4_K, synth.normal((n, k), 0.02, seed=n))
    x = synth.activations(m, k, seed=n + m, dtype=torch.bfloat16)
    xq = oracle.quantize_q8_1(x.float().numpy())
    y = g.gguf_mul_mat(_u8(w), oracle.Q4_K, n, k, x.to(DEV)).float().cpu().numpy()
    rows = np.sort(np.random.default_rng(n + m).choice(n, 256, replace=False))
    rows[0], rows[-1] = 0, n - 1
    ref = oracle.mul_mat(oracle.Q4_K, w[rows], k, xq)
    assert_close(y[:, rows], ref, TOL_BF16, f"Q4_K {n}x{k} m={m}")


def test_mmvq_prequantized_segments(g):
    """One q8_1 quantization reused by three weight segments that write column
    slices of one output (the fused-Linear use)."""
    k, m = 3072, 8
    x = synth.activations(m, k, seed=40, dtype=torch.bfloat16)
    xq_ref = oracle.quantize_q8_1(x.float().numpy())
    xq = g.gguf_quantize_q8_1(x.to(DEV))
    segs = [(oracle.Q4_K, 3072), (oracle.Q4_K, 1024), (oracle.Q6_K, 1024)]
    out = torch.zeros(m, sum(n for _, n in segs), dtype=torch.bfloat16, device=DEV)
    col = 0
    refs = []
    for i, (wt, n) in enumerate(segs):
        w = _weights(wt, n, k, seed=41 + i)
        g.gguf_mul_mat(_u8(w), wt, n, k, xq, xt=oracle.Q8_1, m=m, out=out[:, col:col + n])
        refs.append(oracle.mul_mat(wt, w, k, xq_ref))
        col += n
    assert_close(out.float().cpu().numpy(), np.concatenate(refs, axis=1), TOL_BF16, "segments")


def test_mmvq_edge_cases(g):
    w = _weights(oracle.Q4_K, 1, 256, seed=50)
    x = synth.activations(1, 256, seed=51, dtype=torch.float32)
    y = g.gguf_mul_mat(_u8(w), oracle.Q4_K, 1, 256, x.to(DEV)).cpu().numpy()
    assert_close(y, oracle.mul_mat(oracle.Q4_K, w, 256, oracle.quantize_q8_1(x.numpy())), TOL_F32, "1x256")
    # zero activations give exact zeros
    w = _weights(oracle.Q6_K, 7, 512, seed=52, safe=True)
    y = g.gguf_mul_mat(_u8(w), oracle.Q6_K, 7, 512, torch.zeros(3, 512, device=DEV)).cpu().numpy()
    assert np.all(y == 0)
    # m = 0 is a no-op
    y = g.gguf_mul_mat(_u8(w), oracle.Q6_K, 7, 512, torch.zeros(0, 512, device=DEV))
    assert y.shape == (0, 7)


def test_no_read_past_weight_view(g):
    """A weight view fenced on both sides by 0xFF bytes (NaN fp16 scales) gives
    the same result as a clean copy: no kernel reads outside the view."""
    for wt, n, k in [(oracle.Q6_K, 9, 256), (oracle.Q8_0, 7, 96), (oracle.Q4_K, 5, 512)]:
        w = _weights(wt, n, k, seed=60, safe=True)
        nb = w.nbytes
        off = 4096
        fenced = torch.full((off + nb + 4096,), 0xFF, dtype=torch.uint8, device=DEV)
        fenced[off:off + nb] = _u8(w.reshape(-1))
        view = fenced[off:off + nb]
        x = synth.activations(3, k, seed=61, dtype=torch.float32).to(DEV)
        y = g.gguf_mul_mat(view, wt, n, k, x).cpu().numpy()
        assert np.all(np.isfinite(y))
        ref = oracle.mul_mat(wt, w, k, oracle.quantize_q8_1(x.cpu().numpy()))
        assert_close(y, ref, TOL_F32, f"fenced type {wt}")
        d = g.gguf_dequantize(view, wt, n, k).cpu().numpy()
        np.testing.assert_array_equal(d.view(np.uint32), oracle.dequantize(wt, w, k, oracle.F32).view(np.uint32))
