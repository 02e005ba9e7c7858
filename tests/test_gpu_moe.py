"""GPU parity of mul_mat_id (MoE) against the oracle.

  * gate_up + SwiGLU: h (bf16) within 1e-2 of max(|r|, row rms); the q8_1
    form within one quantization step per value (the GPU's g, u come from the
    fp16 tensor-core product, so h may sit on the other side of a rounding
    boundary -- a q differs by at most 1);
  * down + weighted sum fed with the ORACLE's h_q8_1 rows: within 1e-2;
  * the fused FFN end to end against the full oracle chain: within 1e-2;
  * repeated expert ids, id -1, ids >= E (counted in the status word) and
    weight-0 routes; the full-size configuration (E = 256, top-8, H = 2048,
    I = 512, 8192 tokens) on sampled tokens.
"""
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


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _bank(wt, E, rows, cols, seed, safe):
    if safe:
        return np.ascontiguousarray(synth.safe_blocks(wt, E * rows, cols, seed))
    return np.concatenate([oracle.quantize_weights(wt, synth.normal((rows, cols), 0.02, seed + e)) for e in range(E)])


def _small_case(safe=False):
    E, K, H, I, T = 5, 3, 256, 128, 37
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 100, safe)
    bank_d = _bank(oracle.Q6_K, E, H, I, 200, safe) if I % 256 == 0 else None
    ids, rw = synth.routes(T, E, K, seed=3)
    ids[0] = [1, 1, 1]          # the same expert three times
    ids[1, 2] = -1              # inactive slot
    ids[2] = [-1, -1, -1]       # a token with no active route
    rw[3, 0] = 0.0              # weight 0
    x = synth.activations(T, H, seed=4, dtype=torch.bfloat16)
    return E, K, H, I, T, bank_gu, bank_d, ids, rw, x


def test_gate_up_swiglu_bf16_and_q8_1(g):
    E, K, H, I, T, bank_gu, _, ids, rw, x = _small_case()
    sgu = bank_gu.nbytes // E
    xq = oracle.quantize_q8_1(x.float().numpy())
    h_ref, hq_ref = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids)
    hb = g.gguf_mul_mat_id(_u8(bank_gu), g.Q4_K, E, sgu, 2 * I, H, x.to(DEV), _u8(ids), g.GATE_UP_SWIGLU)
    assert hb.shape == (T * K, I) and hb.dtype == torch.bfloat16
    hb = hb.float().cpu().numpy()
    active = ids.reshape(-1) >= 0
    assert np.all(hb[~active] == 0)
    assert_close(hb[active], h_ref[active], TOL_BF16, "gate_up bf16 h")
    # repeated ids give identical rows
    np.testing.assert_array_equal(hb[0], hb[1])
    np.testing.assert_array_equal(hb[0], hb[2])
    hq = g.gguf_mul_mat_id(_u8(bank_gu), g.Q4_K, E, sgu, 2 * I, H, x.to(DEV), _u8(ids), g.GATE_UP_SWIGLU,
                           out_type=g.Q8_1).cpu().numpy()
    d1, _, q1 = oracle.q8_1_fields(hq)
    d0, _, q0 = oracle.q8_1_fields(hq_ref)
    assert np.all(np.abs(q1.astype(int) - q0.astype(int))[active] <= 1)
    dd1, dd0 = d1.view(np.float16).astype(np.float64), d0.view(np.float16).astype(np.float64)
    assert np.all(np.abs(dd1 - dd0)[active] <= 0.02 * np.abs(dd0)[active] + 1e-12)
    assert np.all(hq[~active] == 0)


def test_down_weighted_sum_from_oracle_h(g):
    E, K, H, T = 4, 3, 512, 29
    I = 256
    bank_d = _bank(oracle.Q6_K, E, H, I, 300, safe=False)
    sd = bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=5)
    ids[0] = [2, 2, 0]
    ids[1, 1] = -1
    rw[2, 2] = 0.0
    # the down GEMM's input comes from the oracle (q8_1 h rows of random activations)
    hq = oracle.quantize_q8_1(synth.normal((T * K, I), 1.0, seed=6))
    ref = oracle.moe_down(oracle.Q6_K, bank_d, E, sd, H, I, hq, ids, rw)
    y = g.gguf_mul_mat_id(_u8(bank_d), g.Q6_K, E, sd, H, I, _u8(hq), _u8(ids), g.DOWN_WEIGHTED_SUM,
                          route_w=_u8(rw), xt=g.Q8_1, out_type=g.F32)
    assert y.shape == (T, H)
    # the fp16 operand path: 3e-3 of the row rms for fp32 outputs (see test_gpu_mmq)
    assert_close(y.cpu().numpy(), ref, 3e-3, "down weighted sum")


@pytest.mark.parametrize("safe", [False, True])
def test_moe_ffn_end_to_end_small(g, safe):
    E, K, H, T = 6, 4, 256, 41
    I = 256
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 400, safe)
    bank_d = _bank(oracle.Q6_K, E, H, I, 500, safe)
    sgu, sd = bank_gu.nbytes // E, bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=7)
    ids[0] = [3, 3, 3, 3]
    ids[1, :2] = -1
    ids[2, 0] = E + 5                  # out of range: inactive, counted
    rw[4, 1] = 0.0
    x = synth.activations(T, H, seed=8, dtype=torch.bfloat16)
    xq = oracle.quantize_q8_1(x.float().numpy())
    _, hq = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids)
    ref = oracle.moe_down(oracle.Q6_K, bank_d, E, sd, H, I, hq, ids, rw)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = g.gguf_moe_ffn(_u8(bank_gu), g.Q4_K, sgu, _u8(bank_d), g.Q6_K, sd, E, H, I, x.to(DEV), _u8(ids),
                       _u8(rw), dev_status=status)
    assert y.dtype == torch.bfloat16
    assert_close(y.float().cpu().numpy(), ref, TOL_BF16, "moe ffn")
    assert int(status.item()) == 1


def test_moe_empty_and_all_inactive(g):
    E, H, I = 2, 256, 256
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 600, True)
    bank_d = _bank(oracle.Q6_K, E, H, I, 601, True)
    ids = np.full((5, 2), -1, np.int32)
    rw = np.ones((5, 2), np.float32)
    x = synth.activations(5, H, seed=9, dtype=torch.bfloat16).to(DEV)
    y = g.gguf_moe_ffn(_u8(bank_gu), g.Q4_K, bank_gu.nbytes // E, _u8(bank_d), g.Q6_K, bank_d.nbytes // E, E, H, I,
                       x, _u8(ids), _u8(rw))
    assert torch.all(y == 0)
    y0 = g.gguf_moe_ffn(_u8(bank_gu), g.Q4_K, bank_gu.nbytes // E, _u8(bank_d), g.Q6_K, bank_d.nbytes // E, E, H,
                        I, x[:0], _u8(ids[:0]), _u8(rw[:0]))
    assert y0.shape == (0, H)


def test_moe_full_size_sampled(g):
    # E = 256 experts, top-8, H = 2048, I = 512; gate_up Q4_K [1024 x 2048],
    # down Q6_K [2048 x 512]; 8192 bf16 tokens; softmax route weights
    E, K, H, I, T = 256, 8, 2048, 512, 8192
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 700, True)
    bank_d = _bank(oracle.Q6_K, E, H, I, 701, True)
    sgu, sd = bank_gu.nbytes // E, bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=2)
    x = synth.activations(T, H, seed=1, dtype=torch.bfloat16)
    y = g.gguf_moe_ffn(_u8(bank_gu), g.Q4_K, sgu, _u8(bank_d), g.Q6_K, sd, E, H, I, x.to(DEV), _u8(ids), _u8(rw))
    y = y.float().cpu().numpy()
    assert np.all(np.isfinite(y))
    xq = oracle.quantize_q8_1(x.float().numpy())
    for t in [0, 1, 4095, 8191, 777]:
        _, hq = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids, routes=(t * K, t * K + K),
                                   nthreads=8)
        ref = oracle.moe_down(oracle.Q6_K, bank_d, E, sd, H, I, hq, ids, rw, tokens=(t, t + 1), nthreads=8)
        assert_close(y[t:t + 1], ref[t:t + 1], TOL_BF16, f"moe token {t}")
