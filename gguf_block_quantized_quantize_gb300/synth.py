"""Seeded synthetic inputs for the tests and ``bench.py``.

This module draws random numbers and fills byte fields; it holds none of the
quantize / dequantize / dot-product arithmetic of the method.  Both the oracle
side (tests) and the CUDA side take their inputs from here.

Recipes (one seed per input; torch CPU generators, so the bytes are identical
on every machine):
  * weights      fp32 ~ N(0, 0.02)           (later quantized by the oracle)
  * activations  ~ N(0, 1) in fp32 / bf16 / fp16
  * routes       top_k distinct experts per token, uniform; weights are the
                 softmax of top_k N(0, 1) logits
  * safe blocks  random packed Q8_0 / Q4_0 / Q4_K / Q5_K / Q6_K / MXFP4 bytes whose fp16 scale fields
                 are finite and of the size quantized N(0, 0.02) weights have,
                 so that no value overflows (the "random-but-safe packed bytes"
                 of FreeToken PR #196, section "Testing")
"""
from __future__ import annotations

import numpy as np
import torch

F32, F16, Q4_0, Q8_0, Q8_1, Q4_K, Q5_K, Q6_K, BF16, MXFP4 = 0, 1, 2, 8, 9, 12, 13, 14, 30, 39
Q4_1, Q5_0, Q5_1 = 3, 6, 7

BLOCK_ELEMS = {Q4_0: 32, Q8_0: 32, Q8_1: 32, Q4_K: 256, Q5_K: 256, Q6_K: 256, MXFP4: 32, Q4_1: 32, Q5_0: 32,
               Q5_1: 32}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q8_1: 36, Q4_K: 144, Q5_K: 176, Q6_K: 210, MXFP4: 17, Q4_1: 20, Q5_0: 22,
               Q5_1: 24}


def row_bytes(t: int, k: int) -> int:
    be = BLOCK_ELEMS[t]
    if k % be:
        raise ValueError(f"k={k} not a multiple of {be}")
    return k // be * BLOCK_BYTES[t]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int) -> np.ndarray:
    """fp32 N(0, std^2) array."""
    return (torch.randn(*shape, generator=_gen(seed), dtype=torch.float32) * std).numpy()


def activations(m: int, k: int, seed: int, dtype: torch.dtype = torch.bfloat16, std: float = 1.0) -> torch.Tensor:
    """CPU tensor [m, k] ~ N(0, std^2) in ``dtype`` (rounded from fp32)."""
    x = torch.randn(m, k, generator=_gen(seed), dtype=torch.float32) * std
    return x.to(dtype)


def routes(n_tokens: int, n_experts: int, top_k: int, seed: int):
    """ids int32 [T, top_k] (distinct per token, uniform) and fp32 weights [T, top_k]."""
    g = _gen(seed)
    ids = torch.rand(n_tokens, n_experts, generator=g).argsort(dim=1)[:, :top_k].to(torch.int32)
    logits = torch.randn(n_tokens, top_k, generator=g, dtype=torch.float32)
    w = torch.softmax(logits, dim=1)
    return ids.numpy(), w.numpy().astype(np.float32)


def _f16_bits(a: np.ndarray) -> np.ndarray:
    return a.astype(np.float16).view(np.uint16)


def safe_blocks(t: int, rows: int, k: int, seed: int) -> np.ndarray:
    """Random packed bytes [rows, row_bytes(t, k)] with safe fp16 scale fields."""
    rng = np.random.default_rng(int(seed))
    nb = k // BLOCK_ELEMS[t]
    bb = BLOCK_BYTES[t]
    blk = rng.integers(0, 256, size=(rows, nb, bb), dtype=np.uint8)
    if t == Q8_0:
        # fp16 d at bytes 0..1 (either sign); int8 quants anywhere in [-128, 127]
        d = rng.uniform(1.0e-4, 6.0e-4, size=(rows, nb)) * rng.choice([-1.0, 1.0], size=(rows, nb))
        blk[:, :, 0:2] = _f16_bits(d).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
    elif t == Q4_0:
        # fp16 d at 0..1 (either sign); 16 nibble bytes random
        d = rng.uniform(2.0e-3, 1.2e-2, size=(rows, nb)) * rng.choice([-1.0, 1.0], size=(rows, nb))
        blk[:, :, 0:2] = _f16_bits(d).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
    elif t in (Q4_1, Q5_1):
        # fp16 d at 0..1 (positive), fp16 m at 2..3 (the block minimum, negative); the rest random
        levels = 15 if t == Q4_1 else 31
        d = rng.uniform(4.0, 8.0, size=(rows, nb)) * 0.02 / levels
        m = -rng.uniform(0.03, 0.07, size=(rows, nb))
        blk[:, :, 0:2] = _f16_bits(d).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
        blk[:, :, 2:4] = _f16_bits(m).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
    elif t == Q5_0:
        # fp16 d at 0..1 (either sign); high-bit and quant bytes random
        d = rng.uniform(1.0e-3, 6.0e-3, size=(rows, nb)) * rng.choice([-1.0, 1.0], size=(rows, nb))
        blk[:, :, 0:2] = _f16_bits(d).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
    elif t == MXFP4:
        # E8M0 exponent byte at 0: block scales 2^-9 .. 2^-3, the range of quantized N(0, 0.02)
        # weights; the 16 code bytes random
        blk[:, :, 0] = rng.integers(118, 125, size=(rows, nb), dtype=np.uint8)
    elif t == Q5_K:
        # fp16 d at 0..1, fp16 dmin at 2..3 (non-negative); scale, high-bit and quant bytes random
        d = rng.uniform(1.0e-5, 1.0e-4, size=(rows, nb))
        dmin = rng.uniform(0.0, 1.2e-3, size=(rows, nb))
        blk[:, :, 0:2] = _f16_bits(d).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
        blk[:, :, 2:4] = _f16_bits(dmin).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
    elif t == Q4_K:
        # fp16 d at 0..1, fp16 dmin at 2..3 (non-negative); 12 scale bytes and 128 quant bytes random
        d = rng.uniform(2.0e-5, 2.0e-4, size=(rows, nb))
        dmin = rng.uniform(0.0, 1.2e-3, size=(rows, nb))
        blk[:, :, 0:2] = _f16_bits(d).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
        blk[:, :, 2:4] = _f16_bits(dmin).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
    elif t == Q6_K:
        # fp16 d at 208..209 (either sign); int8 scales at 192..207 anywhere in [-128, 127]
        d = rng.uniform(5.0e-6, 2.0e-5, size=(rows, nb)) * rng.choice([-1.0, 1.0], size=(rows, nb))
        blk[:, :, 208:210] = _f16_bits(d).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
    elif t == Q8_1:
        d = rng.uniform(5.0e-3, 3.0e-2, size=(rows, nb))
        blk[:, :, 0:2] = _f16_bits(d).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
        s = rng.uniform(-1.0, 1.0, size=(rows, nb))
        blk[:, :, 2:4] = _f16_bits(s).reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
    else:
        raise ValueError(f"unsupported type {t}")
    return np.ascontiguousarray(blk.reshape(rows, nb * bb))


def lognormal_row_scale(rows: int, seed: int, sigma: float = 1.0) -> np.ndarray:
    """Per-row multiplicative scale exp(N(0, sigma^2)), used to spread block
    scales over a wider range than uniform N(0, 0.02) weights give."""
    return np.exp(normal((rows, 1), sigma, seed)).astype(np.float32)


def safe_blocks_device(t: int, rows: int, k: int, seed: int, device) -> torch.Tensor:
    """Random-but-safe packed blocks generated on the device (for multi-GB
    benchmark weights): random bytes, then the fp16 scale fields overwritten
    with a few safe values of the size quantized N(0, 0.02) weights have."""
    nb = k // BLOCK_ELEMS[t]
    bb = BLOCK_BYTES[t]
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    blk = torch.randint(0, 256, (rows, nb, bb), dtype=torch.uint8, device=device, generator=g)
    def field(vals, lo, hi):
        bits = torch.from_numpy(_f16_bits(np.asarray(vals, dtype=np.float64)).view(np.uint8).reshape(-1, 2))
        choice = torch.randint(0, len(vals), (rows, nb), device=device, generator=g)
        blk[:, :, lo:hi] = bits.to(device)[choice]
    if t == Q8_0:
        field([1.5e-4, -2.5e-4, 3.5e-4, -4.5e-4], 0, 2)
    elif t == Q4_0:
        field([4.0e-3, -6.0e-3, 8.0e-3, -1.0e-2], 0, 2)
    elif t == MXFP4:
        blk[:, :, 0] = torch.randint(118, 125, (rows, nb), dtype=torch.uint8, device=device, generator=g)
    elif t in (Q4_1, Q5_1):
        levels = 15 if t == Q4_1 else 31
        field([0.1 / levels, 0.12 / levels, 0.14 / levels, 0.16 / levels], 0, 2)
        field([-0.035, -0.045, -0.055, -0.065], 2, 4)
    elif t == Q5_0:
        field([2.0e-3, -3.0e-3, 4.0e-3, -5.0e-3], 0, 2)
    elif t == Q5_K:
        field([1.5e-5, 3.0e-5, 5.5e-5, 8.0e-5], 0, 2)
        field([0.0, 3.0e-4, 6.0e-4, 9.0e-4], 2, 4)
    elif t == Q4_K:
        field([3.0e-5, 6.0e-5, 1.1e-4, 1.6e-4], 0, 2)
        field([0.0, 3.0e-4, 6.0e-4, 9.0e-4], 2, 4)
    elif t == Q6_K:
        field([7.0e-6, -1.1e-5, 1.4e-5, -1.8e-5], 208, 210)
    else:
        raise ValueError(f"unsupported type {t}")
    return blk.reshape(rows, nb * bb)
