"""Pins of the oracle's number formats, block layouts and quantizers.

These tests check the oracle against what the format definitions and plain
mathematics fix, never against itself:
  * fp16 / bf16 conversion against numpy's float16 and torch's bfloat16;
  * hand-built blocks (tests/golden/*.txt) whose values were derived by hand;
  * quantize -> dequantize error bounds, code reachability, and the
    round-half-away-from-zero rule against a brute-force nearest search.
"""
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN
from gguf_block_quantized_quantize_gb300 import synth


# --------------------------------------------------------------------------
# binary16 / bfloat16
# --------------------------------------------------------------------------

def _specials():
    return np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.9, 65520.0, 1e6, 6.1e-5, 6.0e-8, 2.98e-8, 3.0e-8,
                     1e-10, 0.1, 1.0 / 3.0, 2049.0, 2051.0, 4097.0, -2.5e-6, 3.0e38, 1.5e-45],
                    dtype=np.float32)


def test_f16_matches_numpy(orc):
    rng = np.random.default_rng(0)
    vals = np.concatenate([_specials(), rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-9, 6, 20000)])
    vals = vals.astype(np.float32)
    ours = np.array([orc.f16_bits(float(v)) for v in vals], dtype=np.uint16)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    # decode every finite binary16 pattern
    bits = np.arange(0, 65536, dtype=np.uint32)
    finite = (bits & 0x7C00) != 0x7C00
    dec = np.array([orc.f16_value(int(b)) for b in bits[finite]], dtype=np.float32)
    np.testing.assert_array_equal(dec, bits[finite].astype(np.uint16).view(np.float16).astype(np.float32))


def test_bf16_matches_torch(orc):
    rng = np.random.default_rng(1)
    vals = np.concatenate([_specials(), rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000)])
    vals = vals.astype(np.float32)
    ours = np.array([orc.bf16_bits(float(v)) for v in vals], dtype=np.uint16)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    bits = np.array([0x0000, 0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4049, 0x8001], dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    for b, w in zip(bits, want):
        assert orc.bf16_value(int(b)) == w


# --------------------------------------------------------------------------
# hand-built blocks
# --------------------------------------------------------------------------

def _parse_blocks(name):
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "type":
                cur = {"type": tok[1], "hex": None, "expect": {}}
            elif tok[0] == "hex":
                cur["hex"] = bytes.fromhex(tok[1])
            elif tok[0] == "value":
                cur["expect"][int(tok[1])] = float(tok[2])
            elif tok[0] == "range":
                for i in range(int(tok[1]), int(tok[1]) + int(tok[2])):
                    cur["expect"][i] = float(tok[3])
            elif tok[0] == "end":
                blocks.append(cur)
                cur = None
    if cur is not None:
        blocks.append(cur)
    return blocks


@pytest.mark.parametrize("fname,tname,k", [("q8_0_hand_block.txt", "Q8_0", 32),
                                           ("q4_0_hand_blocks.txt", "Q4_0", 32),
                                           ("q4_k_hand_blocks.txt", "Q4_K", 256),
                                           ("q5_k_hand_blocks.txt", "Q5_K", 256),
                                           ("mxfp4_hand_blocks.txt", "MXFP4", 32),
                                           ("q4_1_q5_0_q5_1_hand_blocks.txt", None, 32),
                                           ("q6_k_hand_blocks.txt", "Q6_K", 256)])
def test_hand_built_blocks(orc, fname, tname, k):
    blocks = _parse_blocks(fname)
    assert blocks
    for b in blocks:
        t = getattr(orc, tname if tname is not None else b["type"])
        raw = np.frombuffer(b["hex"], dtype=np.uint8).reshape(1, -1)
        assert raw.shape[1] == orc.block_bytes(t)
        got = orc.dequantize_f32(t, raw, k)[0]
        got64 = orc.dequantize_f64(t, raw, k)[0]
        for i, v in b["expect"].items():
            assert got[i] == v, (fname, i, got[i], v)
            assert got64[i] == v


def _parse_q8_1_cases():
    cases = []
    with open(os.path.join(GOLDEN, "q8_1_hand_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line.startswith("case"):
                continue
            parts = [p.strip() for p in line.split("|")]
            name = parts[0].split()[1]
            x = np.zeros(32, dtype=np.float32)
            for kv in parts[1].split()[1:]:
                i, v = kv.split("=")
                x[int(i)] = float(v)
            d = int(parts[2].split()[1], 16)
            s = int(parts[3].split()[1], 16)
            q = np.zeros(32, dtype=np.int8)
            for kv in parts[4].split()[1:]:
                i, v = kv.split("=")
                q[int(i)] = int(v)
            cases.append((name, x, d, s, q))
    return cases


def test_q8_1_hand_blocks(orc):
    cases = _parse_q8_1_cases()
    assert len(cases) >= 6
    for name, x, d, s, q in cases:
        blk = orc.quantize_q8_1(x.reshape(1, 32))
        dd, ss, qq = orc.q8_1_fields(blk)
        assert int(dd[0, 0]) == d, name
        assert int(ss[0, 0]) == s, name
        np.testing.assert_array_equal(qq[0, 0], q, err_msg=name)


# --------------------------------------------------------------------------
# q8_1 invariants
# --------------------------------------------------------------------------

def test_q8_1_invariants_and_rounding(orc):
    x = synth.normal((64, 512), 1.0, seed=11)
    x[3, :32] = 0.0                       # an all-zero block
    x[5, 64:96] = np.float32(1e-30)       # a tiny block
    blk = orc.quantize_q8_1(x)
    dbits, sbits, q = orc.q8_1_fields(blk)
    xb = x.reshape(64, 16, 32)
    amax = np.abs(xb).max(axis=2)
    d32 = amax / np.float32(127.0)        # the fp32 d the quantizer divides by
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    # |x - d*q| <= d/2 (before the fp16 rounding of d), as the rounding rule implies
    err = np.abs(xb.astype(np.float64) - d32[..., None].astype(np.float64) * q)
    assert np.all(err <= d32[..., None].astype(np.float64) * 0.5 * (1 + 1e-6) + 1e-45)
    # stored d is the fp16 rounding of the fp32 d
    np.testing.assert_array_equal(dbits, d32.astype(np.float16).view(np.uint16))
    # brute force: q is the nearest integer to x/d, ties away from zero
    r = (xb / np.where(d32 == 0, 1, d32)[..., None]).astype(np.float32)
    cand = np.arange(-128, 129)
    for idx in [(0, 0), (7, 3), (63, 15), (5, 2)]:
        for j in range(32):
            v = float(r[idx][j])
            if d32[idx] == 0:
                assert q[idx][j] == 0
                continue
            dist = np.abs(cand - v)
            best = cand[dist == dist.min()]
            want = best.max() if v > 0 else best.min()
            assert q[idx][j] == want
    # s is the fp16 of fp32(d * sum q)
    ssum = q.astype(np.int32).sum(axis=2).astype(np.float32)
    np.testing.assert_array_equal(sbits, (d32 * ssum).astype(np.float32).astype(np.float16).view(np.uint16))


# --------------------------------------------------------------------------
# weight quantizers: reconstruction bounds and reachability
# --------------------------------------------------------------------------

def test_q8_0_roundtrip_bound(orc):
    w = synth.normal((32, 1024), 0.02, seed=3)
    p = orc.quantize_weights(orc.Q8_0, w)
    dq = orc.dequantize_f32(orc.Q8_0, p, 1024)
    wb = w.reshape(32, 32, 32)
    d = np.abs(wb).max(axis=2, keepdims=True) / 127.0
    # half a step plus the fp16 rounding of d applied to |q| <= 127
    bound = d * 0.5 + 127 * d * 2.0 ** -11
    assert np.all(np.abs(dq.reshape(32, 32, 32) - wb) <= bound * (1 + 1e-5))


def test_q4_k_roundtrip_bound_and_codes(orc):
    w = synth.normal((64, 2048), 0.02, seed=4) * synth.lognormal_row_scale(64, seed=5)
    p = orc.quantize_weights(orc.Q4_K, w)
    dq = orc.dequantize_f32(orc.Q4_K, p, 2048)
    wb = w.reshape(64, 8, 8, 32)
    lo = np.minimum(0, wb.min(axis=3))
    step = (wb.max(axis=3) - lo) / 15.0
    # the 6-bit scale/min rounding moves the grid by at most half a 6-bit unit of
    # d (resp. dmin) times 15 (resp. 1); bound = that + half a step
    d = step.max(axis=2, keepdims=True) / 63.0
    dmin = (-lo).max(axis=2, keepdims=True) / 63.0
    # fp16 storage of d / dmin: relative 2^-11, or half the subnormal quantum 2^-25
    ed, edm = np.maximum(d * 2.0 ** -11, 2.0 ** -25), np.maximum(dmin * 2.0 ** -11, 2.0 ** -25)
    grid_off = 0.5 * d + 63 * ed          # |step_j - d_h * s_j|
    min_off = 0.5 * dmin + 63 * edm       # |min_j - dmin_h * m_j|
    # half a grid step, the clamp at code 15 when the grid is finer than the step,
    # and the shifted min
    bound = 0.5 * (step + grid_off) + 15 * grid_off + min_off
    err = np.abs(dq.reshape(64, 8, 8, 32) - wb).max(axis=3)
    assert np.all(err <= bound * 1.001)
    # every 4-bit code and many 6-bit scales/mins are reached
    blocks = p.reshape(-1, 144)
    qs = blocks[:, 16:]
    codes = set(np.unique(qs & 15)) | set(np.unique(qs >> 4))
    assert codes == set(range(16))


def test_q6_k_roundtrip_bound_and_codes(orc):
    w = synth.normal((64, 2048), 0.02, seed=6) * synth.lognormal_row_scale(64, seed=7)
    p = orc.quantize_weights(orc.Q6_K, w)
    dq = orc.dequantize_f32(orc.Q6_K, p, 2048)
    wb = w.reshape(64, 8, 16, 16)
    scale = np.abs(wb).max(axis=3) / 31.0
    d = scale.max(axis=2, keepdims=True) / 127.0
    # the grid step d_h*sc_j sits within d/2 + 127*e_d of scale_j (int8 rounding of
    # sc_j; fp16 storage of d with e_d = max(d*2^-11, 2^-25), the subnormal case);
    # a half step plus the clamp at 31 steps when the grid is finer gives the bound
    ed = np.maximum(d * 2.0 ** -11, 2.0 ** -25)
    grid_off = 0.5 * d + 127 * ed
    bound = 0.5 * (scale + grid_off) + 31 * grid_off
    err = np.abs(dq.reshape(64, 8, 16, 16) - wb).max(axis=3)
    assert np.all(err <= bound * 1.001 + 1e-12)
    blocks = p.reshape(-1, 210)
    ql, qh = blocks[:, :128], blocks[:, 128:192]
    lows = set(np.unique(ql & 15)) | set(np.unique(ql >> 4))
    highs = set()
    for g in range(4):
        highs |= set(np.unique((qh >> (2 * g)) & 3))
    assert lows == set(range(16)) and highs == set(range(4))


def test_q4_0_roundtrip_bound_and_codes(orc):
    w = synth.normal((32, 1024), 0.02, seed=8) * synth.lognormal_row_scale(32, seed=9)
    p = orc.quantize_weights(orc.Q4_0, w)
    dq = orc.dequantize_f32(orc.Q4_0, p, 1024).reshape(32, 32, 32).astype(np.float64)
    wb = w.reshape(32, 32, 32).astype(np.float64)
    blocks = p.reshape(32, 32, 18)
    dh = np.abs(blocks[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64))[..., None]
    err = np.abs(dq - wb)
    # codes 0..15 are q - 8 = -8..7: the extreme value v sets d = v / -8, so every
    # value lies within 8 steps of 0 (fp16 d: 2^-11 relative); values that do
    # not reach the +8 side are rounded to the nearest step (half a step), those
    # beyond +7.5 steps are clamped to +7 (at most 1 + 2^-9 steps)
    assert np.all(err <= dh * (1.0 + 2.0 ** -9) + 1e-30)
    r = np.abs(wb) / np.where(dh == 0, 1, dh)
    inner = r < 7.4
    assert np.all(err[inner] <= 0.5 * dh.repeat(32, axis=2)[inner] * (1 + 1e-6))
    # the extreme value of each block is reproduced up to the fp16 rounding of d
    amax = np.abs(wb).max(axis=2)
    ext = np.take_along_axis(dq, np.abs(wb).argmax(axis=2)[..., None], axis=2)[..., 0]
    assert np.all(np.abs(np.abs(ext) - amax) <= amax * 2.0 ** -11 * 1.001)
    qs = blocks[:, :, 2:]
    codes = set(np.unique(qs & 15)) | set(np.unique(qs >> 4))
    assert codes == set(range(16))


def test_q5_k_roundtrip_bound_and_codes(orc):
    w = synth.normal((64, 2048), 0.02, seed=10) * synth.lognormal_row_scale(64, seed=12)
    p = orc.quantize_weights(orc.Q5_K, w)
    dq = orc.dequantize_f32(orc.Q5_K, p, 2048)
    wb = w.reshape(64, 8, 8, 32)
    lo = np.minimum(0, wb.min(axis=3))
    step = (wb.max(axis=3) - lo) / 31.0
    # as for Q4_K, with 31 steps per sub-block
    d = step.max(axis=2, keepdims=True) / 63.0
    dmin = (-lo).max(axis=2, keepdims=True) / 63.0
    ed, edm = np.maximum(d * 2.0 ** -11, 2.0 ** -25), np.maximum(dmin * 2.0 ** -11, 2.0 ** -25)
    grid_off = 0.5 * d + 63 * ed
    min_off = 0.5 * dmin + 63 * edm
    bound = 0.5 * (step + grid_off) + 31 * grid_off + min_off
    err = np.abs(dq.reshape(64, 8, 8, 32) - wb).max(axis=3)
    assert np.all(err <= bound * 1.001)
    # the fifth bit halves the Q4_K step: the mean error is well below Q4_K's
    e4 = np.abs(orc.dequantize_f32(orc.Q4_K, orc.quantize_weights(orc.Q4_K, w), 2048) - w).mean()
    assert np.abs(dq - w).mean() < 0.6 * e4
    blocks = p.reshape(-1, 176)
    qh, qs = blocks[:, 16:48], blocks[:, 48:]
    codes = set()
    for j in range(8):
        nib = (qs[:, 32 * (j // 2):32 * (j // 2) + 32] >> (4 * (j % 2))) & 15
        codes |= set(np.unique(nib | (((qh >> j) & 1) << 4)))
    assert codes == set(range(32))


def test_mxfp4_codes_are_the_ocp_e2m1_values(orc):
    """Every e2m1 code at scale 1 against the OCP table of FP4 E2M1 values,
    and the scale as an exact power of two over the whole E8M0 range."""
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    codes = bytes([l | ((l ^ 8) << 4) for l in range(16)])      # value l: code l; value 16 + l: code l ^ 8
    for e in range(0, 255):
        raw = np.frombuffer(bytes([e]) + codes, np.uint8).reshape(1, -1)
        v64 = orc.dequantize_f64(orc.MXFP4, raw, 32)[0]
        v32 = orc.dequantize_f32(orc.MXFP4, raw, 32)[0]
        for l in range(16):
            want = (table[l & 7] if l < 8 else -table[l & 7]) * 2.0 ** (e - 127)
            assert v64[l] == want and v64[16 + l] == -want, (e, l)
            # fp32: the same product, exact while it fits, inf past the fp32 range
            w32 = np.float32(want) if abs(want) < 3.4028234663852886e38 else np.float32(np.copysign(np.inf, want))
            assert v32[l] == w32, (e, l, v32[l], w32)


def test_mxfp4_roundtrip_bound_and_codes(orc):
    w = synth.normal((32, 1024), 0.02, seed=13) * synth.lognormal_row_scale(32, seed=14)
    p = orc.quantize_weights(orc.MXFP4, w)
    blocks = p.reshape(32, 32, 17)
    e = blocks[:, :, 0].astype(np.float64)
    s = 2.0 ** (e - 127)
    wb = np.abs(w.reshape(32, 32, 32)).astype(np.float64)
    # the chosen scale is the smallest power of two with 6 * s >= amax
    amax = wb.max(axis=2)
    assert np.all(6 * s >= amax) and np.all(6 * s / 2 < amax)
    dq = orc.dequantize_f32(orc.MXFP4, p, 1024).reshape(32, 32, 32).astype(np.float64)
    # nearest e2m1 magnitude: within half the widest gap of the grid (1.0 between 4 and 6)
    # below 4 s, and half a gap elsewhere: gaps are 0.5 below 2, 1 from 2 to 4, 2 from 4 to 6
    r = wb / s[..., None]
    half_gap = np.where(r <= 2, 0.25, np.where(r <= 4, 0.5, 1.0))
    assert np.all(np.abs(np.abs(dq) - wb) <= half_gap * s[..., None] * (1 + 1e-12))
    assert np.all((np.sign(dq) == np.sign(w.reshape(32, 32, 32))) | (dq == 0))
    codes = set(np.unique(blocks[:, :, 1:] & 15)) | set(np.unique(blocks[:, :, 1:] >> 4))
    assert codes >= set(range(1, 8)) | set(range(9, 16))


def test_layout_each_quant_nibble_moves_one_value(orc):
    """Perturbing one quant field changes exactly one dequantized value, and
    across a block every value is hit once (pins that the layout is a bijection)."""
    for t, nbytes, qrange in [(orc.Q4_K, 144, range(16, 144)), (orc.Q6_K, 210, range(0, 128))]:
        base = bytearray(nbytes)
        if t == orc.Q4_K:
            base[0:2] = bytes.fromhex("003c")           # d = 1
            base[4:16] = bytes([1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1])   # all s = 1, m = 0
        else:
            base[192:208] = bytes([1] * 16)
            base[208:210] = bytes.fromhex("003c")
        ref = orc.dequantize_f32(t, np.frombuffer(bytes(base), np.uint8).reshape(1, -1), 256)[0]
        hit = np.zeros(256, dtype=np.int32)
        for pos in qrange:
            for shift in (0, 4):
                b = bytearray(base)
                b[pos] ^= (1 << shift)
                v = orc.dequantize_f32(t, np.frombuffer(bytes(b), np.uint8).reshape(1, -1), 256)[0]
                changed = np.nonzero(v != ref)[0]
                assert changed.size == 1, (t, pos, shift, changed)
                hit[changed[0]] += 1
        assert np.all(hit == 1), t
    # Q4_0: the low bit of each nibble of qs moves exactly one of the 32 values
    base = bytearray(18)
    base[0:2] = bytes.fromhex("003c")
    ref = orc.dequantize_f32(orc.Q4_0, np.frombuffer(bytes(base), np.uint8).reshape(1, -1), 32)[0]
    hit = np.zeros(32, dtype=np.int32)
    for pos in range(2, 18):
        for shift in (0, 4):
            b = bytearray(base)
            b[pos] ^= (1 << shift)
            v = orc.dequantize_f32(orc.Q4_0, np.frombuffer(bytes(b), np.uint8).reshape(1, -1), 32)[0]
            changed = np.nonzero(v != ref)[0]
            assert changed.size == 1
            hit[changed[0]] += 1
    assert np.all(hit == 1)
    # MXFP4: every bit of every code (all codes 1 = 0.5, so the sign bit moves
    # the value too) moves exactly one of the 32 values
    base = bytearray([127] + [0x11] * 16)
    ref = orc.dequantize_f32(orc.MXFP4, np.frombuffer(bytes(base), np.uint8).reshape(1, -1), 32)[0]
    for bit in range(4):
        hit = np.zeros(32, dtype=np.int32)
        for pos in range(1, 17):
            for shift in (0, 4):
                b = bytearray(base)
                b[pos] ^= (1 << (bit + shift))
                v = orc.dequantize_f32(orc.MXFP4, np.frombuffer(bytes(b), np.uint8).reshape(1, -1), 32)[0]
                changed = np.nonzero(v != ref)[0]
                assert changed.size == 1, (bit, pos, shift)
                hit[changed[0]] += 1
        assert np.all(hit == 1), bit
    # Q5_K: each nibble of qs and each bit of qh moves exactly one value; each
    # set covers all 256 values once
    base = bytearray(176)
    base[0:2] = bytes.fromhex("003c")
    base[4:16] = bytes([1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1])
    ref = orc.dequantize_f32(orc.Q5_K, np.frombuffer(bytes(base), np.uint8).reshape(1, -1), 256)[0]
    for positions, bits in [(range(48, 176), (0, 4)), (range(16, 48), range(8))]:
        hit = np.zeros(256, dtype=np.int32)
        for pos in positions:
            for bit in bits:
                b = bytearray(base)
                b[pos] ^= (1 << bit)
                v = orc.dequantize_f32(orc.Q5_K, np.frombuffer(bytes(b), np.uint8).reshape(1, -1), 256)[0]
                changed = np.nonzero(v != ref)[0]
                assert changed.size == 1, (pos, bit, changed)
                hit[changed[0]] += 1
        assert np.all(hit == 1)
    # Q6_K high-bit bytes: each 2-bit pair moves exactly one value
    base = bytearray(210)
    base[192:208] = bytes([1] * 16)
    base[208:210] = bytes.fromhex("003c")
    ref = orc.dequantize_f32(orc.Q6_K, np.frombuffer(bytes(base), np.uint8).reshape(1, -1), 256)[0]
    hit = np.zeros(256, dtype=np.int32)
    for pos in range(128, 192):
        for pair in range(4):
            b = bytearray(base)
            b[pos] ^= (1 << (2 * pair))
            v = orc.dequantize_f32(orc.Q6_K, np.frombuffer(bytes(b), np.uint8).reshape(1, -1), 256)[0]
            changed = np.nonzero(v != ref)[0]
            assert changed.size == 1
            hit[changed[0]] += 1
    assert np.all(hit == 1)


def test_dequantize_out_dtypes_are_rne(orc):
    for t, k in [(orc.Q8_0, 256), (orc.Q4_0, 256), (orc.Q4_K, 512), (orc.Q5_K, 512), (orc.Q6_K, 512),
                 (orc.MXFP4, 256)]:
        p = synth.safe_blocks(t, 16, k, seed=21)
        f = orc.dequantize(t, p, k, orc.F32)
        h = orc.dequantize(t, p, k, orc.F16)
        b = orc.dequantize(t, p, k, orc.BF16)
        np.testing.assert_array_equal(h, f.astype(np.float16).view(np.uint16))
        np.testing.assert_array_equal(b, torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
        # the fp32 values are exact: they equal the fp64 evaluation of the same fields
        np.testing.assert_array_equal(f.astype(np.float64), orc.dequantize_f64(t, p, k)) if t not in (orc.Q4_K, orc.Q5_K) else None


def test_get_rows_is_row_gather_of_dequantize(orc):
    p = synth.safe_blocks(orc.Q6_K, 40, 512, seed=22)
    full = orc.dequantize(orc.Q6_K, p, 512, orc.BF16)
    ids = np.array([3, 0, 39, 3, 17], dtype=np.int32)
    np.testing.assert_array_equal(orc.get_rows(orc.Q6_K, p, 512, ids, orc.BF16), full[ids])
    # out-of-range ids give zero rows
    z = orc.get_rows(orc.Q6_K, p, 512, np.array([-1, 40], dtype=np.int32), orc.F32)
    assert np.all(z == 0)


@pytest.mark.parametrize("tname", ["Q8_0", "Q4_0", "Q4_K", "Q5_K", "Q6_K", "MXFP4", "Q4_1", "Q5_0", "Q5_1"])
def test_safe_blocks_give_weight_sized_finite_values(orc, tname):
    """The random-but-safe packed blocks (host and device generators; the
    device one runs on the CPU here) dequantize to finite values of the size
    quantized N(0, 0.02) weights have, so no test or bench input overflows."""
    t = getattr(orc, tname)
    k = 512
    for blocks in (synth.safe_blocks(t, 64, k, seed=90),
                   synth.safe_blocks_device(t, 64, k, seed=91, device="cpu").numpy()):
        assert blocks.shape == (64, synth.row_bytes(t, k))
        v = orc.dequantize_f64(t, np.ascontiguousarray(blocks), k)
        assert np.all(np.isfinite(v))
        assert 1e-4 < np.abs(v).max() < 1.0, (tname, np.abs(v).max())



@pytest.mark.parametrize("tname,levels", [("Q4_1", 15), ("Q5_1", 31)])
def test_q4_1_q5_1_roundtrip_bound_and_codes(orc, tname, levels):
    t = getattr(orc, tname)
    w = synth.normal((32, 1024), 0.02, seed=15) * synth.lognormal_row_scale(32, seed=16)
    p = orc.quantize_weights(t, w)
    dq = orc.dequantize_f64(t, p, 1024).reshape(32, 32, 32)
    wb = w.reshape(32, 32, 32).astype(np.float64)
    step = (wb.max(axis=2) - wb.min(axis=2)) / levels
    # half a step, plus the fp16 roundings of d (times up to `levels`) and of m
    ed = np.maximum(step * 2.0 ** -11, 2.0 ** -25)
    em = np.maximum(np.abs(wb.min(axis=2)) * 2.0 ** -11, 2.0 ** -25)
    bound = 0.5 * (step + ed) + levels * ed + em
    assert np.all(np.abs(dq - wb).max(axis=2) <= bound * 1.001)
    codes = orc.dequantize_f64(t, _unit_scale(orc, t, p), 1024)
    assert set(np.unique(codes).astype(int)) == set(range(levels + 1))


def test_q5_0_roundtrip_bound_and_codes(orc):
    w = synth.normal((32, 1024), 0.02, seed=17) * synth.lognormal_row_scale(32, seed=18)
    p = orc.quantize_weights(orc.Q5_0, w)
    dq = orc.dequantize_f64(orc.Q5_0, p, 1024).reshape(32, 32, 32)
    wb = w.reshape(32, 32, 32).astype(np.float64)
    dh = np.abs(p.reshape(32, 32, 22)[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64))[..., None]
    # as Q4_0 with 16 steps each side: within a step (1 + 2^-9 for the clamp at +15)
    assert np.all(np.abs(dq - wb) <= dh * (1.0 + 2.0 ** -9) + 1e-30)
    codes = orc.dequantize_f64(orc.Q5_0, _unit_scale(orc, orc.Q5_0, p), 1024)
    assert set(np.unique(codes).astype(int)) == set(range(-16, 16))


def _unit_scale(orc, t, p):
    """The same quants with d = 1 (and m = 0): dequantize gives the raw codes."""
    b = p.reshape(p.shape[0], -1, orc.block_bytes(t)).copy()
    b[:, :, 0:2] = [0x00, 0x3C]
    if t in (orc.Q4_1, orc.Q5_1):
        b[:, :, 2:4] = 0
    return np.ascontiguousarray(b.reshape(p.shape[0], -1))


@pytest.mark.parametrize("tname", ["Q4_1", "Q5_0", "Q5_1"])
def test_q4_1_q5_0_q5_1_layout_bijection(orc, tname):
    """Every quant bit (nibble bits and high bits) moves exactly one of the 32
    values, and each set of bits covers all 32 once."""
    t = getattr(orc, tname)
    nb = orc.block_bytes(t)
    qs0 = {"Q4_1": 4, "Q5_0": 6, "Q5_1": 8}[tname]
    qh0 = {"Q4_1": None, "Q5_0": 2, "Q5_1": 4}[tname]
    base = bytearray(nb)
    base[0:2] = bytes.fromhex("003c")
    ref = orc.dequantize_f32(t, np.frombuffer(bytes(base), np.uint8).reshape(1, -1), 32)[0]
    groups = [[(pos, bit) for pos in range(qs0, qs0 + 16) for bit in (0, 4)]]
    if qh0 is not None:
        groups.append([(pos, bit) for pos in range(qh0, qh0 + 4) for bit in range(8)])
    for group in groups:
        hit = np.zeros(32, dtype=np.int32)
        for pos, bit in group:
            b = bytearray(base)
            b[pos] ^= (1 << bit)
            v = orc.dequantize_f32(t, np.frombuffer(bytes(b), np.uint8).reshape(1, -1), 32)[0]
            changed = np.nonzero(v != ref)[0]
            assert changed.size == 1, (tname, pos, bit)
            hit[changed[0]] += 1
        assert np.all(hit == 1)
