"""GPU tests of gguf_copy_async, the SM copy between pinned host memory and
device memory: every byte arrives for any size and alignment, in both
directions and device to device, in stream order with the path's kernels;
pageable host memory and overlapping ranges are refused before any launch."""
import numpy as np
import pytest
import torch

import oracle
from _util import TOL_BF16, assert_close
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


def _bytes(n, seed):
    return torch.from_numpy(np.random.default_rng(seed).integers(0, 256, size=n, dtype=np.uint8))


@pytest.mark.parametrize("n", [1, 15, 16, 17, 255, 4096, 65537, (1 << 20) + 7, 553000])
@pytest.mark.parametrize("off", [0, 1, 8])
@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
def test_copy_every_byte(g, n, off, direction):
    src_host = _bytes(n + off, n + off)
    if direction == "h2d":
        src = src_host.pin_memory()
        dst = torch.full((n + 16,), 0xA5, dtype=torch.uint8, device=DEV)
    elif direction == "d2h":
        src = src_host.to(DEV)
        dst = torch.full((n + 16,), 0xA5, dtype=torch.uint8).pin_memory()
    else:
        src = src_host.to(DEV)
        dst = torch.full((n + 16,), 0xA5, dtype=torch.uint8, device=DEV)
    # unaligned views at `off` (src) and 16 - off (dst) bytes
    g.gguf_copy(dst[16 - off:16 - off + n] if off else dst[:n], src[off:off + n])
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    want = src_host.numpy()[off:off + n]
    lo = 16 - off if off else 0
    assert np.array_equal(got[lo:lo + n], want)
    # nothing outside the destination range was written
    assert (got[:lo] == 0xA5).all() and (got[lo + n:] == 0xA5).all()


def test_copy_in_stream_order_with_the_path(g):
    # host activations -> device (SM copy) -> q8_1 -> MMVQ -> host (SM copy),
    # repeated with new inputs each time: every step sees its own inputs
    k, n = 1024, 600
    w = oracle.quantize_weights(oracle.Q4_K, synth.normal((n, k), 0.02, seed=3))
    wd = torch.from_numpy(w).to(DEV)
    dx = torch.empty((4, k), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((4, n), dtype=torch.bfloat16, device=DEV)
    for step in range(3):
        hx = synth.activations(4, k, seed=10 + step, dtype=torch.bfloat16).pin_memory()
        hy = torch.empty((4, n), dtype=torch.bfloat16).pin_memory()
        g.gguf_copy(dx, hx)
        xq = g.gguf_quantize_q8_1(dx)
        g.gguf_mul_mat(wd, oracle.Q4_K, n, k, xq, xt=oracle.Q8_1, m=4, out=y)
        g.gguf_copy(hy, y)
        torch.cuda.synchronize()
        want = oracle.mul_mat(oracle.Q4_K, w, k, oracle.quantize_q8_1(hx.float().numpy()))
        got = hy.float().numpy()
        assert_close(got, want, TOL_BF16, f"step {step}")
        assert torch.equal(hy, y.cpu())


def test_copy_refuses_pageable_and_overlap(g):
    L = g.load_library()
    pageable = torch.zeros(64, dtype=torch.uint8)
    d = torch.zeros(64, dtype=torch.uint8, device=DEV)
    assert L.gguf_copy_async(d.data_ptr(), pageable.data_ptr(), 64, None) == 1
    assert L.gguf_copy_async(pageable.data_ptr(), d.data_ptr(), 64, None) == 1
    assert L.gguf_copy_async(d.data_ptr() + 8, d.data_ptr(), 32, None) == 1   # overlapping ranges
    with pytest.raises(ValueError):
        g.gguf_copy(d, pageable)
    torch.cuda.synchronize()
