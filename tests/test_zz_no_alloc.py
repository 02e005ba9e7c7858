"""GPU parity of gguf_mul_mat_noalloc, the allocation-free decode entry point.

It must give what gguf_mul_mat gives for the same decode-sized product (the
same MMVQ kernels), on consecutive calls that reuse the fixed scratch with
different sizes, and refuse sizes its scratch does not cover.  This file is
collected last so that it also runs after every other GPU test in the session.
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


@pytest.mark.parametrize("wt,n,k", [(oracle.Q4_K, 1000, 4096), (oracle.Q6_K, 333, 2048), (oracle.Q8_0, 517, 16384),
                                    (oracle.Q4_0, 301, 4128), (oracle.Q5_K, 257, 2048), (oracle.MXFP4, 263, 4128)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_mul_mat_on_consecutive_calls(g, wt, n, k, dtype):
    w = _u8(oracle.quantize_weights(wt, synth.normal((n, k), 0.02, seed=n)))
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    # the larger call first, then a smaller one that reads only part of the
    # scratch the first call left behind
    for call, m in enumerate((8, 3)):
        x = synth.activations(m, k, seed=100 * call + m, dtype=dtype).to(DEV)
        y_noalloc = g.gguf_mul_mat_noalloc(w, wt, n, k, x)
        y_ref = g.gguf_mul_mat(w, wt, n, k, x)
        torch.cuda.synchronize()
        assert y_noalloc.dtype == dtype
        a, b = y_noalloc.float().cpu().numpy(), y_ref.float().cpu().numpy()
        assert_close(a, b, tol, f"noalloc vs mul_mat call {call}")


def test_noalloc_against_oracle(g):
    wt, n, k, m = oracle.Q4_K, 256, 1024, 5
    wq = oracle.quantize_weights(wt, synth.normal((n, k), 0.02, seed=7))
    x = synth.activations(m, k, seed=8, dtype=torch.bfloat16)
    ref = oracle.mul_mat(wt, wq, k, oracle.quantize_q8_1(x.float().numpy()))
    y = g.gguf_mul_mat_noalloc(_u8(wq), wt, n, k, x.to(DEV), out_dtype=torch.float32)
    assert_close(y.cpu().numpy(), ref, TOL_F32, "noalloc vs oracle")


@pytest.mark.parametrize("m,k", [(9, 256), (1, 16384 + 256)])
def test_noalloc_rejects_sizes_beyond_scratch(g, m, k):
    # checked on the host before any launch: nothing runs on the device
    w = torch.zeros(8 * (k // 256) * 144, dtype=torch.uint8, device=DEV)
    x = torch.zeros(m, k, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(g.GgufError) as e:
        g.gguf_mul_mat_noalloc(w, oracle.Q4_K, 8, k, x)
    assert e.value.status == 5, str(e.value)          # GGUF_ERR_WORKSPACE
