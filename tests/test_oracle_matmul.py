"""Pins of the oracle's per-block integer dots, blockwise matmul and MoE.

  * block dots on blocks whose scales are 1 reduce to plain integer dot
    products of the quants (numpy int64 brute force);
  * the blockwise fp64 formula equals the plain fp64 dot product of the
    dequantized operands (Q8_0, Q6_K: exactly up to fp64 rounding; Q4_K: up to
    the fp16 rounding of the activation's s = d * sum(q), bounded below);
  * quantized matmul approximates the fp32 matmul within the quantization error;
  * MoE special cases: E = 1, top_k = 1 is a dense GEMM + SwiGLU; a repeated
    expert id is two independent routes; id -1 and weight 0 contribute nothing.
"""
import numpy as np
import pytest

from gguf_block_quantized_quantize_gb300 import synth


def _unit_scale_blocks(orc, t, n, k, seed):
    """Random quants with every scale 1 (and min 0): dequant == the raw quants."""
    p = synth.safe_blocks(t, n, k, seed).reshape(n, -1, orc.block_bytes(t)).copy()
    if t in (orc.Q8_0, orc.Q4_0):
        p[:, :, 0:2] = [0x00, 0x3C]
    elif t in (orc.Q4_K, orc.Q5_K):
        p[:, :, 0:4] = [0x00, 0x3C, 0x00, 0x00]
        p[:, :, 4:16] = [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1]
    elif t == orc.Q6_K:
        p[:, :, 192:208] = 1
        p[:, :, 208:210] = [0x00, 0x3C]
    elif t == orc.MXFP4:
        p[:, :, 0] = 128            # scale 2: the value is the integer quant 2 * e2m1
    elif t == orc.Q5_0:
        p[:, :, 0:2] = [0x00, 0x3C]
    elif t in (orc.Q4_1, orc.Q5_1):
        p[:, :, 0:4] = [0x00, 0x3C, 0x00, 0x00]   # d = 1, m = 0
    return np.ascontiguousarray(p.reshape(n, -1))


@pytest.mark.parametrize("tname", ["Q8_0", "Q4_0", "Q4_K", "Q5_K", "Q6_K", "MXFP4", "Q4_1", "Q5_0", "Q5_1"])
def test_block_dots_brute_force(orc, tname):
    t = getattr(orc, tname)
    k, n, m = 512, 6, 3
    w = _unit_scale_blocks(orc, t, n, k, seed=31)
    qw = orc.dequantize_f32(t, w, k).astype(np.int64)      # raw quants (q, q - 8, q, q - 32 or 2 * e2m1)
    assert np.all(qw == orc.dequantize_f32(t, w, k))      # integral
    xq = orc.quantize_q8_1(synth.normal((m, k), 1.0, seed=32))
    _, _, qa = orc.q8_1_fields(xq)
    qa = qa.reshape(m, k).astype(np.int64)
    sub = orc.sub_elems(t)
    want = (qa.reshape(m, 1, k // sub, sub) * qw.reshape(1, n, k // sub, sub)).sum(axis=3)
    got = orc.block_dots(t, w, k, xq)
    np.testing.assert_array_equal(got, want)
    # extreme values stay exact in int32: all quants at their extremes
    if t == orc.Q8_0:
        w2 = w.reshape(n, -1, 34).copy()
        w2[:, :, 2:] = 0x81                                 # -127
        w2 = np.ascontiguousarray(w2.reshape(n, -1))
        x = np.full((1, k), -1.0, np.float32)
        got = orc.block_dots(t, w2, k, orc.quantize_q8_1(x))
        assert np.all(got == 32 * 127 * 127)


@pytest.mark.parametrize("tname", ["Q8_0", "Q4_0", "Q6_K", "MXFP4", "Q5_0"])
def test_blockwise_equals_dequant_dot(orc, tname):
    t = getattr(orc, tname)
    k = 1024
    w = synth.safe_blocks(t, 24, k, seed=41)
    xq = orc.quantize_q8_1(synth.normal((5, k), 1.0, seed=42))
    y = orc.mul_mat(t, w, k, xq)
    ref = orc.dequantize_f64(t, w, k) @ orc.dequantize_f64(orc.Q8_1, xq, k).T
    ref = ref.T
    scale = np.abs(orc.dequantize_f64(t, w, k)).sum(axis=1)[None, :] * np.abs(orc.dequantize_f64(orc.Q8_1, xq, k)).max(axis=1)[:, None]
    assert np.all(np.abs(y - ref) <= 1e-13 * scale)


@pytest.mark.parametrize("tname", ["Q4_K", "Q5_K"])
def test_blockwise_affine_min_term(orc, tname):
    """Q4_K / Q5_K: blockwise y = dequant-dot + sum_j dmin*m_j*(d_a*sum(q_a) - s_a),
    and the difference is bounded by the fp16 rounding of d_a and s_a."""
    t = getattr(orc, tname)
    k = 1024
    w = synth.safe_blocks(t, 16, k, seed=43)
    xq = orc.quantize_q8_1(synth.normal((4, k), 1.0, seed=44))
    y = orc.mul_mat(t, w, k, xq)
    ref = orc.mul_mat_dequant_f64(t, w, k, xq)
    # bound: |d_a sum q - s_a| <= |sum q| * |d_a| * 2^-10 per 32-block (two fp16 roundings)
    dbits, sbits, qa = orc.q8_1_fields(xq)
    da = dbits.view(np.float16).astype(np.float64)
    qsum = np.abs(qa.astype(np.int64).sum(axis=2))
    blk = w.reshape(16, -1, orc.block_bytes(t))
    dmin = blk[:, :, 2:4].copy().view(np.float16)[..., 0].astype(np.float64)   # [n, nsb]
    per_block = (qsum * np.abs(da) * 2.0 ** -10 + 1e-300)                       # [m, k/32]
    bound = (per_block.reshape(4, 1, -1, 8).sum(axis=3) * dmin[None] * 63).sum(axis=2)
    assert np.all(np.abs(y - ref) <= bound + 1e-12)
    assert np.abs(y - ref).max() > 0        # the term is real, not identically zero


@pytest.mark.parametrize("tname,tol", [("Q8_0", 0.02), ("Q4_0", 0.12), ("Q4_K", 0.15), ("Q5_K", 0.08),
                                       ("Q6_K", 0.05), ("MXFP4", 0.2), ("Q4_1", 0.12), ("Q5_0", 0.08),
                                       ("Q5_1", 0.06)])
def test_quantized_matmul_tracks_fp32(orc, tname, tol):
    t = getattr(orc, tname)
    k = 2048
    wf = synth.normal((64, k), 0.02, seed=45)
    xf = synth.normal((4, k), 1.0, seed=46)
    y = orc.mul_mat(t, orc.quantize_weights(t, wf), k, orc.quantize_q8_1(xf))
    ref = xf.astype(np.float64) @ wf.T.astype(np.float64)
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert rel < tol, rel


def test_mul_mat_row_subset_and_threads(orc):
    k = 512
    w = synth.safe_blocks(orc.Q6_K, 33, k, seed=47)
    xq = orc.quantize_q8_1(synth.normal((3, k), 1.0, seed=48))
    full = orc.mul_mat(orc.Q6_K, w, k, xq)
    part = orc.mul_mat(orc.Q6_K, w, k, xq, rows=(5, 20), nthreads=4)
    np.testing.assert_array_equal(part[:, 5:20], full[:, 5:20])
    assert np.all(part[:, :5] == 0) and np.all(part[:, 20:] == 0)


# --------------------------------------------------------------------------
# MoE
# --------------------------------------------------------------------------

def _bf16_round(a):
    """fp64 -> nearest bf16 value (ties to even), rounded once: 8 significant
    bits, by exact power-of-two scaling and numpy's round-half-even."""
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)                       # a = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                  # below the normal range the quantum stays 2^-133
    return np.ldexp(np.round(np.ldexp(a, 8 - e)), e - 8)


def _bf16_round_via_f32(a):
    """The same after an fp32 step: differs from _bf16_round when the fp32
    value lands on a bf16 tie that the fp64 value was not on."""
    return _bf16_round(np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64))


def _q8_0_rows(d_bits, q):
    """Q8_0 rows of one block each: fp16 scale bits d_bits[i], int8 quants q[i]."""
    out = np.zeros((len(d_bits), 34), np.uint8)
    out[:, 0:2] = np.array(d_bits, np.uint16).astype("<u2").view(np.uint8).reshape(-1, 2)
    out[:, 2:] = np.array(q, np.int8).view(np.uint8)
    return out


def test_moe_single_expert_is_dense_swiglu(orc):
    H, I, T = 256, 256, 5
    wgu = orc.quantize_weights(orc.Q4_K, synth.normal((2 * I, H), 0.02, seed=51))
    wd = orc.quantize_weights(orc.Q6_K, synth.normal((H, I), 0.02, seed=52))
    xq = orc.quantize_q8_1(synth.normal((T, H), 1.0, seed=53))
    ids = np.zeros((T, 1), np.int32)
    rw = np.full((T, 1), 0.75, np.float32)
    h, hq = orc.moe_gate_up(orc.Q4_K, wgu, 1, wgu.nbytes, 2 * I, H, xq, ids)
    g = orc.mul_mat(orc.Q4_K, wgu[:I], H, xq)
    u = orc.mul_mat(orc.Q4_K, wgu[I:], H, xq)
    silu = g / (1.0 + np.exp(-g))                        # textbook SiLU
    np.testing.assert_array_equal(h, _bf16_round(silu * u))
    np.testing.assert_array_equal(hq, orc.quantize_q8_1(h))
    y = orc.moe_down(orc.Q6_K, wd, 1, wd.nbytes, H, I, hq, ids, rw)
    np.testing.assert_allclose(y, 0.75 * orc.mul_mat(orc.Q6_K, wd, I, hq), rtol=1e-15, atol=1e-300)


def test_moe_swiglu_rounds_fp64_to_bf16_once(orc):
    """h = bf16(silu(g) * u) is one rounding of the fp64 value.  The first three
    gate / up row pairs are hand-picked so that silu(g) * u lies off a bf16 tie
    that its fp32 rounding lands on exactly: an fp32 step in between would
    round those three the other way."""
    H, I = 32, 32
    rng = np.random.default_rng(81)
    # (gate d, gate q, up d, up q) against x = e_0, whose q8_1 block is d = fp16(1/127), q_0 = 127
    picked = [(0x240F, -49, 0x2085, -111), (0x2054, -13, 0x2340, -86), (0x1BCA, 44, 0x1D46, -27)]
    dg = [p[0] for p in picked] + [0x2000] * (I - 3)
    du = [p[2] for p in picked] + [0x2000] * (I - 3)
    qg = rng.integers(-127, 128, (I, 32))
    qu = rng.integers(-127, 128, (I, 32))
    for i, p in enumerate(picked):
        qg[i] = 0; qu[i] = 0
        qg[i, 0] = p[1]; qu[i, 0] = p[3]
    bank = np.concatenate([_q8_0_rows(dg, qg), _q8_0_rows(du, qu)]).reshape(-1)
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    xq = orc.quantize_q8_1(x)
    h, _ = orc.moe_gate_up(orc.Q8_0, bank, 1, bank.nbytes, 2 * I, H, xq, np.zeros((1, 1), np.int32))
    # independent expectation: fp64 dot of the dequantized rows and activation, textbook SiLU
    d_x = np.float16(np.float32(1.0) / np.float32(127.0)).astype(np.float64)
    wg = np.array(dg, np.uint16).view(np.float16).astype(np.float64)[:, None] * qg
    wu = np.array(du, np.uint16).view(np.float16).astype(np.float64)[:, None] * qu
    xv = np.zeros(H)
    xv[0] = d_x * 127.0
    g, u = wg @ xv, wu @ xv
    v = g / (1.0 + np.exp(-g)) * u
    np.testing.assert_array_equal(h[0], _bf16_round(v))
    # the pin is sensitive: an fp32 step would change exactly the picked rows here
    assert np.all(_bf16_round_via_f32(v[:3]) != _bf16_round(v[:3]))


def test_moe_repeated_and_inactive_routes(orc):
    H, I, E, T, K = 256, 256, 3, 4, 3
    bank_gu = np.concatenate([orc.quantize_weights(orc.Q4_K, synth.normal((2 * I, H), 0.02, seed=60 + e)) for e in range(E)])
    bank_d = np.concatenate([orc.quantize_weights(orc.Q6_K, synth.normal((H, I), 0.02, seed=70 + e)) for e in range(E)])
    sgu, sd = bank_gu.nbytes // E, bank_d.nbytes // E
    xq = orc.quantize_q8_1(synth.normal((T, H), 1.0, seed=61))
    ids = np.array([[1, 1, 2], [0, -1, 2], [2, 2, 2], [-1, -1, -1]], np.int32)
    rw = np.array([[0.25, 0.5, 0.25], [0.5, 9.0, 0.5], [0.125, 0.375, 0.0], [1.0, 1.0, 1.0]], np.float32)
    h, hq = orc.moe_gate_up(orc.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids)
    hrows = h.reshape(T, K, I)
    # a repeated id computes the same row twice
    np.testing.assert_array_equal(hrows[0, 0], hrows[0, 1])
    np.testing.assert_array_equal(hrows[2, 0], hrows[2, 2])
    # id -1 gives a zero row
    assert np.all(hrows[1, 1] == 0) and np.all(hrows[3] == 0)
    y = orc.moe_down(orc.Q6_K, bank_d, E, sd, H, I, hq, ids, rw)
    single = lambda e, r: orc.mul_mat(orc.Q6_K, bank_d[e * H:(e + 1) * H], I, hq[r:r + 1])[0]
    np.testing.assert_allclose(y[0], 0.75 * single(1, 0) + 0.25 * single(2, 2), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(y[1], 0.5 * single(0, 3) + 0.5 * single(2, 5), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(y[2], 0.5 * single(2, 6), rtol=1e-12, atol=1e-15)   # weight 0 dropped
    assert np.all(y[3] == 0)
    # ids >= E are inactive too
    ids2 = ids.copy()
    ids2[0, 0] = E
    y2 = orc.moe_down(orc.Q6_K, bank_d, E, sd, H, I, hq, ids2, rw)
    np.testing.assert_allclose(y2[0], 0.5 * single(1, 1) + 0.25 * single(2, 2), rtol=1e-12, atol=1e-15)


def test_route_recipe(orc):
    ids, w = synth.routes(1000, 256, 8, seed=2)
    assert ids.shape == (1000, 8) and ids.dtype == np.int32
    assert all(len(set(r)) == 8 for r in ids)
    assert ids.min() >= 0 and ids.max() < 256
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-6)
    assert np.all(w > 0)


def test_moe_plain_rows(orc):
    """mul_mat_id without the weighted sum: each active route's row equals the
    dense product of its expert with its token's row; the route-weighted sum
    of the rows equals moe_down fed the token rows per route; inactive routes
    are zero rows."""
    E, T, K, n, k = 3, 5, 2, 64, 512
    bank = np.concatenate([orc.quantize_weights(orc.Q4_K, synth.normal((n, k), 0.02, seed=80 + e)) for e in range(E)])
    stride = bank.nbytes // E
    xq = orc.quantize_q8_1(synth.normal((T, k), 1.0, seed=84))
    ids, rw = synth.routes(T, E, K, seed=85)
    ids[0] = [2, 2]
    ids[1, 1] = -1
    ids[2, 0] = E + 1
    y = orc.moe_plain(orc.Q4_K, bank, E, stride, n, k, xq, ids)
    assert y.shape == (T * K, n)
    for t in range(T):
        for j in range(K):
            r, e = t * K + j, ids[t, j]
            if 0 <= e < E:
                np.testing.assert_array_equal(y[r], orc.mul_mat(orc.Q4_K, bank[e * n:(e + 1) * n], k, xq[t:t + 1])[0])
            else:
                assert np.all(y[r] == 0)
    ref = orc.moe_down(orc.Q4_K, bank, E, stride, n, k, np.repeat(xq, K, axis=0), ids, rw)
    got = (y.reshape(T, K, n) * rw.astype(np.float64)[:, :, None]).sum(axis=1)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-300)



@pytest.mark.parametrize("tname", ["Q4_1", "Q5_1"])
def test_blockwise_plus_min_term(orc, tname):
    """Q4_1 / Q5_1: blockwise y = dequant-dot - sum_b m_b*(d_a*sum(q_a) - s_a):
    the +m term uses the stored s_a, so the difference is bounded by its fp16
    rounding, and is real."""
    t = getattr(orc, tname)
    k = 1024
    w = synth.safe_blocks(t, 16, k, seed=48)
    xq = orc.quantize_q8_1(synth.normal((4, k), 1.0, seed=49))
    y = orc.mul_mat(t, w, k, xq)
    ref = orc.mul_mat_dequant_f64(t, w, k, xq)
    dbits, _, qa = orc.q8_1_fields(xq)
    da = dbits.view(np.float16).astype(np.float64)
    qsum = np.abs(qa.astype(np.int64).sum(axis=2))
    m = np.abs(w.reshape(16, -1, orc.block_bytes(t))[:, :, 2:4].copy().view(np.float16)[..., 0].astype(np.float64))
    bound = (qsum[:, None, :] * np.abs(da)[:, None, :] * 2.0 ** -10 * m[None]).sum(axis=2)
    assert np.all(np.abs(y - ref) <= bound + 1e-12)
    assert np.abs(y - ref).max() > 0
