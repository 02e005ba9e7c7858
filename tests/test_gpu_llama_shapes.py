"""GPU parity of the Llama-3.2-3B-shaped decode step's linears at full size,
issued as the benchmark issues them: q + k (Q4_K) as one segment call on the
attention input, v (Q6_K), o (Q4_K), gate + up (Q4_K) as one segment call on
the FFN input, down (Q6_K, K = 8192), and the tied Q6_K LM head (128256 rows,
sampled), at 1, 8 and 32 tokens (MMVQ, the tensor-core MMVQ and MMQ)."""
import numpy as np
import pytest
import torch

import oracle
from _util import TOL_BF16, assert_close
from gguf_block_quantized_quantize_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
D, F, V, KV = 3072, 8192, 128256, 1024


@pytest.fixture(scope="module")
def g():
    from gguf_block_quantized_quantize_gb300 import build

    build.build()
    import gguf_block_quantized_quantize_gb300 as g

    g.load_library()
    return g


@pytest.fixture(scope="module")
def layer():
    Q4, Q6 = oracle.Q4_K, oracle.Q6_K
    shapes = {"q": (Q4, D, D), "k": (Q4, KV, D), "v": (Q6, KV, D), "o": (Q4, D, D), "gate": (Q4, F, D),
              "up": (Q4, F, D), "down": (Q6, D, F)}
    host = {nm: (wt, n, k, synth.safe_blocks(wt, n, k, seed=1000 + i)) for i, (nm, (wt, n, k)) in enumerate(shapes.items())}
    dev = {nm: torch.from_numpy(w).to(DEV) for nm, (_, _, _, w) in host.items()}
    return host, dev


@pytest.mark.parametrize("m", [1, 8, 32])
def test_llama_layer_linears_as_benchmarked(g, layer, m):
    host, dev = layer
    act_d = synth.activations(m, D, seed=m, dtype=torch.bfloat16)
    act_f = synth.activations(m, F, seed=m + 1, dtype=torch.bfloat16)
    xd, xf = g.gguf_quantize_q8_1(act_d.to(DEV)), g.gguf_quantize_q8_1(act_f.to(DEV))
    out = {nm: torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV) for nm, (_, n, _, _) in host.items()}
    ws = torch.empty(256 << 20, dtype=torch.uint8, device=DEV)
    Q4, Q6 = oracle.Q4_K, oracle.Q6_K
    g.gguf_mul_mat_segments(Q4, D, xd, [(dev["q"], D, out["q"]), (dev["k"], KV, out["k"])], xt=g.Q8_1, m=m, ws=ws)
    g.gguf_mul_mat(dev["v"], Q6, KV, D, xd, xt=g.Q8_1, m=m, out=out["v"], ws=ws)
    g.gguf_mul_mat(dev["o"], Q4, D, D, xd, xt=g.Q8_1, m=m, out=out["o"], ws=ws)
    g.gguf_mul_mat_segments(Q4, D, xd, [(dev["gate"], F, out["gate"]), (dev["up"], F, out["up"])], xt=g.Q8_1, m=m,
                            ws=ws)
    g.gguf_mul_mat(dev["down"], Q6, D, F, xf, xt=g.Q8_1, m=m, out=out["down"], ws=ws)
    torch.cuda.synchronize()
    xrd, xrf = oracle.quantize_q8_1(act_d.float().numpy()), oracle.quantize_q8_1(act_f.float().numpy())
    rng = np.random.default_rng(m)
    for nm, (wt, n, k, w) in host.items():
        rows = np.sort(rng.choice(n, min(n, 192), replace=False))
        rows[0], rows[-1] = 0, n - 1
        ref = oracle.mul_mat(wt, w[rows], k, xrf if nm == "down" else xrd)
        y = out[nm].float().cpu().numpy()
        assert np.isfinite(y).all(), f"{nm}: an output was not written"
        assert_close(y[:, rows], ref, TOL_BF16, f"{nm} {n}x{k} m={m}")


@pytest.mark.parametrize("m", [1, 8, 32])
def test_llama_lm_head_sampled(g, m):
    Q6 = oracle.Q6_K
    w = synth.safe_blocks(Q6, V, D, seed=2000)
    x = synth.activations(m, D, seed=50 + m, dtype=torch.bfloat16)
    xq = g.gguf_quantize_q8_1(x.to(DEV))
    y = torch.full((m, V), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(g.gguf_mul_mat_ws_size(Q6, V, D, g.Q8_1, m, g.BF16) or 16, dtype=torch.uint8, device=DEV)
    g.gguf_mul_mat(torch.from_numpy(w).to(DEV), Q6, V, D, xq, xt=g.Q8_1, m=m, out=y, ws=ws)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(m).choice(V, 256, replace=False))
    rows[0], rows[-1] = 0, V - 1
    ref = oracle.mul_mat(Q6, w[rows], D, oracle.quantize_q8_1(x.float().numpy()))
    got = y.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert_close(got[:, rows], ref, TOL_BF16, f"LM head m={m}")
