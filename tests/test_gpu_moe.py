"""GPU parity of mul_mat_id (MoE) against the oracle.

  * gate_up + SwiGLU: h (bf16) within 1e-2 of max(|r|, row rms); the q8_1
    form within half a quantization step of each side plus one bf16 ulp (g, u
    come from the precise hi + lo tensor-core product, so a bf16 rounding of h
    can still land on the other side of a tie);
  * down + weighted sum fed with the ORACLE's h_q8_1 rows: within 1e-2;
  * the fused FFN end to end against the full oracle chain: norm-wise per
    token within 1e-2 (the re-quantized intermediate, see _util.py);
  * repeated expert ids, id -1, ids >= E (counted in the status word) and
    weight-0 routes; the full-size configuration (E = 256, top-8, H = 2048,
    I = 512, 8192 tokens) on sampled tokens;
  * the route-batched MMVQ (vector) path of small token counts (option
    moe_vec_max_tokens): the same checks, and agreement with the tensor-core
    path on the same inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from _util import TOL_BF16, TOL_F32, TOL_MOE_E2E_ELEM, TOL_MOE_E2E_ELEM_VEC, assert_close, assert_close_moe_e2e
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


@pytest.fixture(params=["tensor_core", "vector"])
def path(request, g):
    """Runs the test through the tensor-core grouped GEMM (option
    moe_vec_max_tokens = 0) and through the route-batched MMVQ (option at
    its maximum), whatever the token count."""
    saved = g.gguf_get_option("moe_vec_max_tokens")
    g.gguf_set_option("moe_vec_max_tokens", 0 if request.param == "tensor_core" else 256)
    yield request.param
    g.gguf_set_option("moe_vec_max_tokens", saved)


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


@pytest.fixture(params=[1, 0])
def gate_up_precise(request, g):
    """The grouped gate_up GEMM on hi + lo operands (option
    moe_gate_up_precise = 1, three MMAs per K step) and on one fp16 operand
    per side (0)."""
    saved = g.gguf_get_option("moe_gate_up_precise")
    g.gguf_set_option("moe_gate_up_precise", request.param)
    yield request.param
    g.gguf_set_option("moe_gate_up_precise", saved)


def test_gate_up_swiglu_bf16_and_q8_1(g, path, gate_up_precise):
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
    # The two h differ by the tensor-core rounding and at most one bf16 ulp
    # (2^-7 relative); each q8_1 dequantization is within d/2 of its h.  So the
    # dequantized values agree within d_gpu/2 + d_ref/2 + |h| 2^-7 + 2e-3 rms.
    assert np.all(hq[~active] == 0)
    d1 = oracle.q8_1_fields(hq)[0].view(np.float16).astype(np.float64)
    d0 = oracle.q8_1_fields(hq_ref)[0].view(np.float16).astype(np.float64)
    v1 = oracle.dequantize_f64(oracle.Q8_1, hq, I)
    v0 = oracle.dequantize_f64(oracle.Q8_1, hq_ref, I)
    rms = np.sqrt((h_ref.astype(np.float64) ** 2).mean(axis=1, keepdims=True))
    bound = (np.repeat(d1, 32, axis=1) + np.repeat(d0, 32, axis=1)) / 2 + np.abs(h_ref) * 2.0 ** -7 + 2e-3 * rms
    assert np.all((np.abs(v1 - v0) <= bound * 1.0001)[active])


def test_down_weighted_sum_from_oracle_h(g, path):
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
    # fp32 output: the precise (hi + lo) operand mode
    assert_close(y.cpu().numpy(), ref, TOL_F32, "down weighted sum")


@pytest.mark.parametrize("safe", [False, True])
def test_moe_ffn_end_to_end_small(g, path, safe):
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
    assert_close_moe_e2e(y.float().cpu().numpy(), ref, "moe ffn",
                         TOL_MOE_E2E_ELEM_VEC if path == "vector" else TOL_MOE_E2E_ELEM)
    assert int(status.item()) == 1


def test_moe_empty_and_all_inactive(g, path):
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
    # the first and last 8 tokens and 32 more across the range
    toks = sorted(set(list(range(8)) + list(range(T - 8, T)) +
                      np.random.default_rng(11).choice(np.arange(8, T - 8), 32, replace=False).tolist()))
    for t in toks:
        _, hq = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids, routes=(t * K, t * K + K),
                                   nthreads=8)
        ref = oracle.moe_down(oracle.Q6_K, bank_d, E, sd, H, I, hq, ids, rw, tokens=(t, t + 1), nthreads=8)
        assert_close_moe_e2e(y[t:t + 1], ref[t:t + 1], f"moe token {t}")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_moe_ffn_q4_k_down_bank(g, path, out_dtype):
    """Both banks Q4_K: the down GEMM needs the min-term correction columns of
    the q8_1 intermediate; fp32 output runs the precise down product."""
    E, K, H, T, I = 4, 2, 512, 23, 256
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 800, False)
    bank_d = _bank(oracle.Q4_K, E, H, I, 801, False)
    sgu, sd = bank_gu.nbytes // E, bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=9)
    ids[0] = [1, 1]
    x = synth.activations(T, H, seed=10, dtype=torch.float32)
    xq = oracle.quantize_q8_1(x.numpy())
    _, hq = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids)
    ref = oracle.moe_down(oracle.Q4_K, bank_d, E, sd, H, I, hq, ids, rw)
    out = torch.empty(T, H, dtype=out_dtype, device=DEV)
    y = g.gguf_moe_ffn(_u8(bank_gu), g.Q4_K, sgu, _u8(bank_d), g.Q4_K, sd, E, H, I, x.to(DEV), _u8(ids), _u8(rw),
                       out=out)
    assert_close_moe_e2e(y.float().cpu().numpy(), ref, f"moe ffn q4_k down {out_dtype}")


@pytest.mark.parametrize("out_type", ["f32", "bf16"])
def test_down_q4_k_from_oracle_h(g, path, out_type):
    """Q4_K down bank through the DOWN mode (q8_1 rows from the oracle): the
    operand conversion appends the min-term correction columns."""
    E, K, H, T, I = 4, 2, 512, 23, 256
    bank_d = _bank(oracle.Q4_K, E, H, I, 801, False)
    sd = bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=9)
    ids[0] = [1, 1]
    hq = oracle.quantize_q8_1(synth.normal((T * K, I), 1.0, seed=12))
    ref = oracle.moe_down(oracle.Q4_K, bank_d, E, sd, H, I, hq, ids, rw)
    yt = g.F32 if out_type == "f32" else g.BF16
    y = g.gguf_mul_mat_id(_u8(bank_d), g.Q4_K, E, sd, H, I, _u8(hq), _u8(ids), g.DOWN_WEIGHTED_SUM,
                          route_w=_u8(rw), xt=g.Q8_1, out_type=yt)
    assert_close(y.float().cpu().numpy(), ref, TOL_F32 if yt == g.F32 else TOL_BF16, f"down q4_k {out_type}")


def test_gate_up_h512(g, path):
    E, K, H, T, I = 4, 2, 512, 23, 256
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 800, False)
    sgu = bank_gu.nbytes // E
    ids, _ = synth.routes(T, E, K, seed=9)
    x = synth.activations(T, H, seed=10, dtype=torch.float32)
    h_ref, _ = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, oracle.quantize_q8_1(x.numpy()), ids)
    hb = g.gguf_mul_mat_id(_u8(bank_gu), g.Q4_K, E, sgu, 2 * I, H, x.to(DEV), _u8(ids), g.GATE_UP_SWIGLU)
    assert_close(hb.float().cpu().numpy(), h_ref, TOL_BF16, "gate_up H=512")
    # precise gate_up (tensor-core hi + lo, or the exact block sums of the
    # vector path): the bf16 h agrees bit for bit with the oracle's except near
    # rounding ties (fp32 accumulation, ~1e-6 relative: ~0.1% of values)
    same = (hb.float().cpu().numpy() == h_ref)
    assert same.mean() > 0.995, same.mean()


@pytest.mark.parametrize("wt", [oracle.Q4_0, oracle.Q5_K, oracle.Q8_0, oracle.Q6_K, oracle.MXFP4])
def test_gate_up_bank_types(g, path, wt):
    """gate_up with every weight type of the bank, through both paths: the
    bf16 h against the oracle's, inactive routes zero."""
    E, K, H, I, T = 4, 3, 512, 128, 21
    bank_gu = _bank(wt, E, 2 * I, H, 300 + wt, False)
    sgu = bank_gu.nbytes // E
    ids, _ = synth.routes(T, E, K, seed=wt)
    ids[0] = [2, 2, 2]
    ids[1, 0] = -1
    x = synth.activations(T, H, seed=wt + 1, dtype=torch.bfloat16)
    h_ref, _ = oracle.moe_gate_up(wt, bank_gu, E, sgu, 2 * I, H, oracle.quantize_q8_1(x.float().numpy()), ids)
    active = ids.reshape(-1) >= 0
    hb = g.gguf_mul_mat_id(_u8(bank_gu), wt, E, sgu, 2 * I, H, x.to(DEV), _u8(ids), g.GATE_UP_SWIGLU)
    hb = hb.float().cpu().numpy()
    assert np.all(hb[~active] == 0)
    assert_close(hb[active], h_ref[active], TOL_BF16, f"gate_up type {wt} ({path})")


@pytest.mark.parametrize("wt", [oracle.Q4_0, oracle.MXFP4])
def test_vec_down_two_block_pieces_odd_blocks(g, wt):
    # a Q4_0 / MXFP4 down bank with I = 96 (three blocks per row): the
    # route-batched MMVQ's last piece holds one block
    E, K, H, I, T = 3, 2, 256, 96, 5
    bank_d = _bank(wt, E, H, I, 77, True)
    sd = bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=78)
    hq = oracle.quantize_q8_1(synth.normal((T * K, I), 1.0, seed=79))
    ref = oracle.moe_down(wt, bank_d, E, sd, H, I, hq, ids, rw)
    y = g.gguf_mul_mat_id(_u8(bank_d), wt, E, sd, H, I, _u8(hq), _u8(ids), g.DOWN_WEIGHTED_SUM,
                          route_w=_u8(rw), xt=g.Q8_1, out_type=g.F32).cpu().numpy()
    assert_close(y, ref, TOL_F32, f"vec down type {wt} I=96")


@pytest.mark.parametrize("wt", [oracle.Q4_K, oracle.Q6_K, oracle.MXFP4])
@pytest.mark.parametrize("out_type", ["f32", "bf16"])
def test_plain_rows(g, path, wt, out_type):
    """mul_mat_id without the weighted sum: one output row per route against
    the oracle; inactive and out-of-range ids give zero rows and the latter
    are counted; route weights are ignored."""
    E, K, n, k, T = 4, 3, 256, 512, 21
    bank = _bank(wt, E, n, k, 400 + wt, False)
    stride = bank.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=wt + 3)
    ids[0] = [1, 1, 1]
    ids[1, 2] = -1
    ids[2, 0] = E + 5
    rw[3, 0] = 0.0                      # a weight of 0 does not skip a PLAIN route
    x = synth.activations(T, k, seed=wt + 4, dtype=torch.float32 if out_type == "f32" else torch.bfloat16)
    ref = oracle.moe_plain(wt, bank, E, stride, n, k, oracle.quantize_q8_1(x.float().numpy()), ids)
    active = ((ids >= 0) & (ids < E)).reshape(-1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = g.gguf_mul_mat_id(_u8(bank), wt, E, stride, n, k, x.to(DEV), _u8(ids), g.PLAIN, route_w=_u8(rw),
                          out_type=g.F32 if out_type == "f32" else g.BF16, dev_status=status)
    assert y.shape == (T * K, n)
    y = y.float().cpu().numpy()
    assert np.all(y[~active] == 0)
    assert_close(y[active], ref[active], TOL_F32 if out_type == "f32" else TOL_BF16, f"plain type {wt} ({path})")
    np.testing.assert_array_equal(y[0], y[1])          # the same expert and token
    assert int(status.item()) == 1
    # pre-quantized token rows give the same result
    xq = g.gguf_quantize_q8_1(x.to(DEV))
    y2 = g.gguf_mul_mat_id(_u8(bank), wt, E, stride, n, k, xq, _u8(ids), g.PLAIN, xt=g.Q8_1,
                           out_type=g.F32 if out_type == "f32" else g.BF16).float().cpu().numpy()
    np.testing.assert_array_equal(y2, y)


# ---------------------------------------------------------------- vector path (few tokens)

class _vec_off:
    """Runs the block with the tensor-core path for every token count."""

    def __init__(self, g):
        self.g = g

    def __enter__(self):
        self.saved = self.g.gguf_get_option("moe_vec_max_tokens")
        self.g.gguf_set_option("moe_vec_max_tokens", 0)

    def __exit__(self, *a):
        self.g.gguf_set_option("moe_vec_max_tokens", self.saved)


def _q8_1_close(hq, hq_ref, h_ref, active, I):
    # as in test_gate_up_swiglu_bf16_and_q8_1: each dequantized value within
    # d/2 of its h on each side, plus one bf16 ulp of h and 2e-3 of the row rms
    d1 = oracle.q8_1_fields(hq)[0].view(np.float16).astype(np.float64)
    d0 = oracle.q8_1_fields(hq_ref)[0].view(np.float16).astype(np.float64)
    v1 = oracle.dequantize_f64(oracle.Q8_1, hq, I)
    v0 = oracle.dequantize_f64(oracle.Q8_1, hq_ref, I)
    rms = np.sqrt((h_ref.astype(np.float64) ** 2).mean(axis=1, keepdims=True))
    bound = (np.repeat(d1, 32, axis=1) + np.repeat(d0, 32, axis=1)) / 2 + np.abs(h_ref) * 2.0 ** -7 + 2e-3 * rms
    return bool(np.all((np.abs(v1 - v0) <= bound * 1.0001)[active]))


@pytest.mark.parametrize("T", [1, 3, 16])
def test_vec_gate_up_outputs(g, T):
    E, K, H, I = 5, 3, 512, 128
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 900 + T, False)
    sgu = bank_gu.nbytes // E
    ids, _ = synth.routes(T, E, K, seed=T)
    ids[0, 1] = ids[0, 0]                 # a repeated expert
    if T > 1:
        ids[1, 2] = -1                    # an inactive slot
    x = synth.activations(T, H, seed=T + 1, dtype=torch.bfloat16)
    xq = oracle.quantize_q8_1(x.float().numpy())
    h_ref, hq_ref = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids)
    active = ids.reshape(-1) >= 0
    args = (_u8(bank_gu), g.Q4_K, E, sgu, 2 * I, H, x.to(DEV), _u8(ids), g.GATE_UP_SWIGLU)
    hb = g.gguf_mul_mat_id(*args).float().cpu().numpy()
    assert np.all(hb[~active] == 0)
    assert_close(hb[active], h_ref[active], TOL_BF16, f"vec gate_up bf16 T {T}")
    np.testing.assert_array_equal(hb[0], hb[1])
    hq = g.gguf_mul_mat_id(*args, out_type=g.Q8_1).cpu().numpy()
    assert np.all(hq[~active] == 0)
    assert _q8_1_close(hq, hq_ref, h_ref, active, I)
    # F16: the dequantized q8_1 values d16 * q of the same rows
    hf = g.gguf_mul_mat_id(*args, out_type=g.F16).float().cpu().numpy()
    deq = oracle.dequantize_f32(oracle.Q8_1, hq, I).astype(np.float16).astype(np.float32)
    np.testing.assert_array_equal(hf, deq)
    # the tensor-core path on the same inputs
    with _vec_off(g):
        hb2 = g.gguf_mul_mat_id(*args).float().cpu().numpy()
    assert_close(hb2[active], hb[active], TOL_BF16, f"vec vs tensor-core gate_up T {T}")


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
@pytest.mark.parametrize("T", [1, 5, 16])
def test_vec_down_from_oracle_h(g, wt, T):
    E, K, H, I = 4, 3, 512, 256
    bank_d = _bank(wt, E, H, I, 950 + T, False)
    sd = bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=T + 7)
    ids[0] = [2, 2, 0]
    if T > 1:
        ids[1, 1] = -1
        rw[1, 0] = 0.0
    hq = oracle.quantize_q8_1(synth.normal((T * K, I), 1.0, seed=T + 8))
    ref = oracle.moe_down(wt, bank_d, E, sd, H, I, hq, ids, rw)
    args = (_u8(bank_d), wt, E, sd, H, I, _u8(hq), _u8(ids), g.DOWN_WEIGHTED_SUM)
    y = g.gguf_mul_mat_id(*args, route_w=_u8(rw), xt=g.Q8_1, out_type=g.F32).cpu().numpy()
    assert_close(y, ref, TOL_F32, f"vec down type {wt} T {T}")
    with _vec_off(g):
        y2 = g.gguf_mul_mat_id(*args, route_w=_u8(rw), xt=g.Q8_1, out_type=g.F32).cpu().numpy()
    assert_close(y2, ref, TOL_F32, f"tensor-core down type {wt} T {T}")


@pytest.mark.parametrize("T", [1, 2, 16])
@pytest.mark.parametrize("down", [oracle.Q6_K, oracle.Q4_K, oracle.Q5_K, oracle.Q4_0, oracle.MXFP4])
def test_vec_moe_ffn_end_to_end(g, T, down):
    E, K, H, I = 6, 4, 256, 256
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 1000 + T, False)
    bank_d = _bank(down, E, H, I, 1100 + T, False)
    sgu, sd = bank_gu.nbytes // E, bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=T + 20)
    ids[0, :2] = [3, 3]
    if T > 1:
        ids[1, 0] = -1
        ids[1, 1] = E + 2              # out of range: inactive, counted
        rw[1, 2] = 0.0
    x = synth.activations(T, H, seed=T + 21, dtype=torch.bfloat16)
    xq = oracle.quantize_q8_1(x.float().numpy())
    _, hq = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids)
    ref = oracle.moe_down(down, bank_d, E, sd, H, I, hq, ids, rw)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    args = (_u8(bank_gu), g.Q4_K, sgu, _u8(bank_d), down, sd, E, H, I, x.to(DEV), _u8(ids), _u8(rw))
    y = g.gguf_moe_ffn(*args, dev_status=status).float().cpu().numpy()
    assert_close_moe_e2e(y, ref, f"vec moe ffn T {T} down {down}", TOL_MOE_E2E_ELEM_VEC)
    assert int(status.item()) == (1 if T > 1 else 0)
    with _vec_off(g):
        y2 = g.gguf_moe_ffn(*args).float().cpu().numpy()
    assert_close_moe_e2e(y2, ref, f"tensor-core moe ffn T {T} down {down}")


def test_vec_moe_full_size_decode(g):
    # the full-size expert banks (E = 256, top-8, H = 2048, I = 512) at 16
    # decode tokens through the vector path, every token against the oracle
    E, K, H, I, T = 256, 8, 2048, 512, 16
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 700, True)
    bank_d = _bank(oracle.Q6_K, E, H, I, 701, True)
    sgu, sd = bank_gu.nbytes // E, bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=3)
    x = synth.activations(T, H, seed=4, dtype=torch.bfloat16)
    y = g.gguf_moe_ffn(_u8(bank_gu), g.Q4_K, sgu, _u8(bank_d), g.Q6_K, sd, E, H, I, x.to(DEV), _u8(ids), _u8(rw))
    y = y.float().cpu().numpy()
    xq = oracle.quantize_q8_1(x.float().numpy())
    _, hq = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids, nthreads=8)
    ref = oracle.moe_down(oracle.Q6_K, bank_d, E, sd, H, I, hq, ids, rw, nthreads=8)
    assert_close_moe_e2e(y, ref, "vec moe full size", TOL_MOE_E2E_ELEM_VEC)


def _e2e_error_stats(y, ref):
    from _util import rel_err
    e = rel_err(y, ref)
    q = np.percentile(e, [50, 99, 99.9, 99.99])
    return {"max": float(e.max()), "p50": float(q[0]), "p99": float(q[1]), "p99.9": float(q[2]),
            "p99.99": float(q[3]), "frac_gt_1e-2": float((e > 1e-2).mean()), "frac_gt_3e-3": float((e > 3e-3).mean()),
            "n": int(e.size)}


@pytest.mark.parametrize("T,vec,precise", [(8192, False, 1), (8192, False, 0), (256, True, 1)])
def test_moe_full_size_error_distribution(g, T, vec, precise):
    """Per-element error of the fused FFN against the full oracle chain on the
    full-size expert block (E = 256, top-8, H = 2048, I = 512): 64 tokens,
    the first 16, the last 16 and 32 spread between (printed with -s); the
    tensor-core path with the gate_up GEMM on hi + lo operands and on one
    fp16 operand per side."""
    E, K, H, I = 256, 8, 2048, 512
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 700, True)
    bank_d = _bank(oracle.Q6_K, E, H, I, 701, True)
    sgu, sd = bank_gu.nbytes // E, bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=2)
    x = synth.activations(T, H, seed=1, dtype=torch.bfloat16)
    saved = (g.gguf_get_option("moe_vec_max_tokens"), g.gguf_get_option("moe_gate_up_precise"))
    g.gguf_set_option("moe_vec_max_tokens", 256 if vec else 0)
    g.gguf_set_option("moe_gate_up_precise", precise)
    try:
        y = g.gguf_moe_ffn(_u8(bank_gu), g.Q4_K, sgu, _u8(bank_d), g.Q6_K, sd, E, H, I, x.to(DEV), _u8(ids),
                           _u8(rw)).float().cpu().numpy()
    finally:
        g.gguf_set_option("moe_vec_max_tokens", saved[0])
        g.gguf_set_option("moe_gate_up_precise", saved[1])
    toks = sorted(set(list(range(16)) + list(range(T - 16, T)) +
                      np.random.default_rng(5).choice(np.arange(16, T - 16), 32, replace=False).tolist()))
    xq = oracle.quantize_q8_1(x[toks].float().numpy())
    sub_ids, sub_rw = ids[toks], rw[toks]
    _, hq = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, sub_ids, nthreads=16)
    ref = oracle.moe_down(oracle.Q6_K, bank_d, E, sd, H, I, hq, sub_ids, sub_rw, nthreads=16)
    st = _e2e_error_stats(y[toks], ref)
    print(f"\nmoe e2e error T={T} {'vector' if vec else 'tensor-core'} gate_up precise={precise}: {st}")
    # one fp16 operand per side in gate_up (opt-in): measured max 2.0e-2, p99 8.6e-3
    # elementwise at this size, against 1.0e-2 / 3.4e-3 on hi + lo operands; only
    # the per-token norm-wise bound is asserted for it
    tol = TOL_MOE_E2E_ELEM_VEC if vec else (TOL_MOE_E2E_ELEM if precise else None)
    assert_close_moe_e2e(y[toks], ref, f"moe e2e T={T}", tol)


def test_device_error_word_is_clear_after_moe(g, path):
    g.gguf_device_errors(clear=True)
    E, K, H, I, T, bank_gu, _, ids, rw, x = _small_case()
    sgu = bank_gu.nbytes // E
    g.gguf_mul_mat_id(_u8(bank_gu), g.Q4_K, E, sgu, 2 * I, H, x.to(DEV), _u8(ids), g.GATE_UP_SWIGLU)
    assert g.gguf_device_errors(clear=True) == 0


@pytest.mark.parametrize("H,I,down", [(256, 256, oracle.Q6_K), (2048, 512, oracle.Q6_K), (512, 256, oracle.Q4_K)])
def test_moe_staged_weights(g, H, I, down):
    """The grouped GEMMs with packed weight rows staged by bulk tensor copies
    (option mmq_stage, the default) and loaded by the producer warps: both
    against the oracle chain, and against each other."""
    E, K, T = 7, 4, 300
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 900, True)
    bank_d = _bank(down, E, H, I, 901, True)
    sgu, sd = bank_gu.nbytes // E, bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=31)
    ids[0] = [2, 2, 5, 5]
    ids[1, 1] = -1
    x = synth.activations(T, H, seed=32, dtype=torch.bfloat16)
    xq = oracle.quantize_q8_1(x.float().numpy())
    _, hq = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids, nthreads=8)
    ref = oracle.moe_down(down, bank_d, E, sd, H, I, hq, ids, rw, nthreads=8)
    saved = (g.gguf_get_option("mmq_stage"), g.gguf_get_option("moe_vec_max_tokens"),
             g.gguf_get_option("moe_deterministic"))
    g.gguf_set_option("moe_vec_max_tokens", 0)
    g.gguf_set_option("moe_deterministic", 1)
    ys = []
    try:
        for stage in (1, 0):
            g.gguf_set_option("mmq_stage", stage)
            y = g.gguf_moe_ffn(_u8(bank_gu), g.Q4_K, sgu, _u8(bank_d), down, sd, E, H, I, x.to(DEV), _u8(ids),
                               _u8(rw)).float().cpu().numpy()
            assert_close_moe_e2e(y, ref, f"moe staged={stage} H {H} I {I}")
            ys.append(y)
    finally:
        g.gguf_set_option("mmq_stage", saved[0])
        g.gguf_set_option("moe_vec_max_tokens", saved[1])
        g.gguf_set_option("moe_deterministic", saved[2])
    # the same operand values either way, and a fixed order of the sums
    np.testing.assert_array_equal(ys[0], ys[1])


def test_moe_deterministic_option(g):
    """Option moe_deterministic = 1 (the default): per-route rows summed in
    slot order, the same bits on every run; 0: the weighted rows added into
    the token rows by bulk reduce-adds in the down GEMM's epilogue, which
    agrees with it to fp32 rounding of the sum's order."""
    E, K, H, I, T = 9, 8, 512, 256, 400
    bank_gu = _bank(oracle.Q4_K, E, 2 * I, H, 950, True)
    bank_d = _bank(oracle.Q6_K, E, H, I, 951, True)
    sgu, sd = bank_gu.nbytes // E, bank_d.nbytes // E
    ids, rw = synth.routes(T, E, K, seed=41)
    x = synth.activations(T, H, seed=42, dtype=torch.float32).to(DEV)
    args = (_u8(bank_gu), g.Q4_K, sgu, _u8(bank_d), g.Q6_K, sd, E, H, I, x, _u8(ids), _u8(rw))
    saved = (g.gguf_get_option("moe_deterministic"), g.gguf_get_option("moe_vec_max_tokens"))
    g.gguf_set_option("moe_vec_max_tokens", 0)
    try:
        g.gguf_set_option("moe_deterministic", 1)
        y1 = g.gguf_moe_ffn(*args).cpu().numpy()
        y2 = g.gguf_moe_ffn(*args).cpu().numpy()
        g.gguf_set_option("moe_deterministic", 0)
        y3 = g.gguf_moe_ffn(*args).cpu().numpy()
    finally:
        g.gguf_set_option("moe_deterministic", saved[0])
        g.gguf_set_option("moe_vec_max_tokens", saved[1])
    np.testing.assert_array_equal(y1, y2)
    assert_close(y3, y1, 1e-5, "atomic vs slot-order weighted sum")
    xq = oracle.quantize_q8_1(x.cpu().numpy())
    _, hq = oracle.moe_gate_up(oracle.Q4_K, bank_gu, E, sgu, 2 * I, H, xq, ids, nthreads=8)
    ref = oracle.moe_down(oracle.Q6_K, bank_d, E, sd, H, I, hq, ids, rw, nthreads=8)
    assert_close_moe_e2e(y3, ref, "moe fp32 out, fused sum")


@pytest.mark.parametrize("n", [510, 500])
def test_down_fused_sum_row_lengths(g, n):
    """The fused weighted sum (option moe_deterministic = 0) for output rows
    whose length is a multiple of 4 (bulk reduce-adds of 16-byte runs) and one
    that is not (fp32 atomics), against the oracle; a partial last column tile
    in both."""
    E, K, T, I = 6, 4, 150, 256
    packed = _bank(oracle.Q6_K, E, n, I, 960, safe=True).reshape(E, -1)
    sd = (packed.shape[1] + 15) // 16 * 16     # expert matrices on 16-byte boundaries
    bank_d = np.zeros((E, sd), dtype=np.uint8)
    bank_d[:, :packed.shape[1]] = packed
    bank_d = bank_d.reshape(-1)
    ids, rw = synth.routes(T, E, K, seed=43)
    ids[0] = [3, 3, 1, 1]
    ids[1, 2] = -1
    rw[2, 1] = 0.0
    hq = oracle.quantize_q8_1(synth.normal((T * K, I), 1.0, seed=44))
    ref = oracle.moe_down(oracle.Q6_K, bank_d, E, sd, n, I, hq, ids, rw)
    saved = (g.gguf_get_option("moe_deterministic"), g.gguf_get_option("moe_vec_max_tokens"))
    g.gguf_set_option("moe_vec_max_tokens", 0)
    try:
        out = {}
        for det in (1, 0):
            g.gguf_set_option("moe_deterministic", det)
            out[det] = g.gguf_mul_mat_id(_u8(bank_d), g.Q6_K, E, sd, n, I, _u8(hq), _u8(ids), g.DOWN_WEIGHTED_SUM,
                                         route_w=_u8(rw), xt=g.Q8_1, out_type=g.F32).cpu().numpy()
    finally:
        g.gguf_set_option("moe_deterministic", saved[0])
        g.gguf_set_option("moe_vec_max_tokens", saved[1])
    assert_close(out[0], ref, TOL_F32, f"fused weighted sum n={n}")
    assert_close(out[0], out[1], 1e-5, f"fused vs slot-order sum n={n}")
