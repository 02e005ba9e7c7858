"""GPU parity of gguf_mul_mat_segments: several weight matrices on one input.

Each segment's output must equal the oracle's product for that weight, in
every path: dp4a MMVQ (1..4 tokens), the int8 tensor-core MMVQ (5..8 tokens of
Q4_K, where 16-row tiles straddle segment boundaries), MMVQ in 8-row chunks,
and MMQ (one GEMM per segment on the shared operand).
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


@pytest.mark.parametrize("wt", [oracle.Q8_0, oracle.Q4_0, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K, oracle.MXFP4])
@pytest.mark.parametrize("m", [1, 3, 6, 8, 40])
def test_segments_match_oracle(g, wt, m):
    k = 1024
    ns = [2100, 0, 517, 64] if wt == oracle.Q4_K else [300, 0, 517, 64]
    ws_ = [oracle.quantize_weights(wt, synth.normal((n, k), 0.02, seed=11 + i)) if n else None for i, n in enumerate(ns)]
    x = synth.activations(m, k, seed=m, dtype=torch.float32)
    xq = oracle.quantize_q8_1(x.numpy())
    # outputs: column slices of one wide row-major tensor
    wide = torch.zeros(m, sum(ns) + 5, dtype=torch.float32, device=DEV)
    segs, c0 = [], 0
    for w, n in zip(ws_, ns):
        segs.append((_u8(w) if n else torch.zeros(16, dtype=torch.uint8, device=DEV), n, wide[:, c0:c0 + n]))
        c0 += n
    g.gguf_mul_mat_segments(wt, k, x.to(DEV), segs)
    got = wide.cpu().numpy()
    c0 = 0
    for i, (w, n) in enumerate(zip(ws_, ns)):
        if n:
            ref = oracle.mul_mat(wt, w, k, xq)
            assert_close(got[:, c0:c0 + n], ref, TOL_F32, f"segment {i} type {wt} m {m}")
        c0 += n
    assert np.all(got[:, c0:] == 0)   # columns past the segments untouched


@pytest.mark.parametrize("m", [5, 8])
def test_segments_q6_k_tensor_core_tall(g, m):
    # tall Q6_K segments (>= 32768 rows in all) take the tensor-core Q6_K
    # MMVQ; the 16-row tiles straddle the segment boundaries at 20001 and
    # 20001 + 12799, and the last row of every segment is the guarded end of
    # its view.  Each segment's output is checked against the oracle on
    # sampled rows (the boundary rows included) and against the dp4a kernel.
    k = 512
    ns = [20001, 12799, 37]
    ws_ = [synth.safe_blocks(oracle.Q6_K, n, k, seed=31 + i) for i, n in enumerate(ns)]
    x = synth.activations(m, k, seed=m + 50, dtype=torch.float32)
    xq = oracle.quantize_q8_1(x.numpy())
    wide = torch.zeros(m, sum(ns), dtype=torch.float32, device=DEV)
    segs, c0 = [], 0
    for w, n in zip(ws_, ns):
        segs.append((_u8(w), n, wide[:, c0:c0 + n]))
        c0 += n
    g.gguf_mul_mat_segments(oracle.Q6_K, k, x.to(DEV), segs)
    got = wide.cpu().numpy()
    g.gguf_set_option("mmvq_tc", 0)
    try:
        wide2 = torch.zeros_like(wide)
        segs2 = [(w_, n, wide2[:, c:c + n]) for (w_, n, _), c in zip(segs, np.cumsum([0] + ns[:-1]))]
        g.gguf_mul_mat_segments(oracle.Q6_K, k, x.to(DEV), segs2)
        dp4a = wide2.cpu().numpy()
    finally:
        g.gguf_set_option("mmvq_tc", 1)
    assert_close(got, dp4a, TOL_F32, f"tensor-core vs dp4a m {m}")
    c0 = 0
    rng = np.random.default_rng(m)
    for i, (w, n) in enumerate(zip(ws_, ns)):
        rows = np.unique(np.concatenate([[0, n - 1], rng.choice(n, min(n, 48), replace=False)]))
        ref = oracle.mul_mat(oracle.Q6_K, w[rows], k, xq)
        assert_close(got[:, c0 + rows], ref, TOL_F32, f"segment {i} m {m}")
        c0 += n


def test_segments_equal_separate_calls_bf16(g):
    # the decode shape: two Q4_K matrices on one q8_1 copy, bf16 out
    k = 4096
    w1 = _u8(synth.safe_blocks(oracle.Q4_K, 4096, k, seed=1))
    w2 = _u8(synth.safe_blocks(oracle.Q4_K, 2560, k, seed=2))   # both >= 2048 rows: same kernel at 8 tokens
    for m in (1, 2, 4, 8):
        x = synth.activations(m, k, seed=m, dtype=torch.bfloat16).to(DEV)
        xq = g.gguf_quantize_q8_1(x)
        y1 = torch.empty(m, 4096, dtype=torch.bfloat16, device=DEV)
        y2 = torch.empty(m, 2560, dtype=torch.bfloat16, device=DEV)
        g.gguf_mul_mat_segments(oracle.Q4_K, k, xq, [(w1, 4096, y1), (w2, 2560, y2)], xt=oracle.Q8_1, m=m)
        r1 = g.gguf_mul_mat(w1, oracle.Q4_K, 4096, k, xq, xt=oracle.Q8_1, m=m, out_dtype=torch.bfloat16)
        r2 = g.gguf_mul_mat(w2, oracle.Q4_K, 2560, k, xq, xt=oracle.Q8_1, m=m, out_dtype=torch.bfloat16)
        # same kernels, same per-row arithmetic and reduction order
        assert torch.equal(y1, r1) and torch.equal(y2, r2), m


def test_segments_reject_bad_count(g):
    x = torch.zeros(1, 256, dtype=torch.bfloat16, device=DEV)
    y = torch.zeros(1, 8, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(8 * 144, dtype=torch.uint8, device=DEV)
    with pytest.raises(g.GgufError) as e:
        g.gguf_mul_mat_segments(oracle.Q4_K, 256, x, [(w, 8, y)] * 9)
    assert e.value.status == 1


@pytest.mark.parametrize("wt", [oracle.Q4_K, oracle.Q6_K, oracle.Q8_0])
def test_mul_mat_batch_matches_segment_calls(g, wt):
    """A batch of decode-sized jobs (chained launches) gives exactly what the
    same jobs give as separate segment calls, and the oracle's products; a
    kernel queued after the batch sees every job's output."""
    k = 2048
    shapes = [(300, 1), (1000, 2)]
    ws = {n: _u8(oracle.quantize_weights(wt, synth.normal((n, k), 0.02, seed=n + s))) for n, s in shapes}
    jobs, refs, sep = [], [], []
    for j, m in enumerate((1, 2, 4, 8, 3)):
        x = synth.activations(m, k, seed=40 + j, dtype=torch.bfloat16)
        xq = g.gguf_quantize_q8_1(x.to(DEV))
        outs = [torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV) for n, _ in shapes]
        jobs.append((xq, [(ws[n], n, o) for (n, _), o in zip(shapes, outs)]))
        xq_ref = oracle.quantize_q8_1(x.float().numpy())
        refs.append([oracle.mul_mat(wt, ws[n].cpu().numpy(), k, xq_ref) for n, _ in shapes])
        sep.append([torch.empty((m, n), dtype=torch.bfloat16, device=DEV) for n, _ in shapes])
        g.gguf_mul_mat_segments(wt, k, xq, [(ws[n], n, o) for (n, _), o in zip(shapes, sep[-1])], xt=g.Q8_1, m=m)
    outs = g.gguf_mul_mat_batch(wt, k, jobs)
    sums = [sum(o.float().sum() for o in job_outs) for job_outs in outs]   # queued right after the batch
    torch.cuda.synchronize()
    for j, job_outs in enumerate(outs):
        for o, s, r in zip(job_outs, sep[j], refs[j]):
            assert torch.equal(o, s), f"job {j}: batch differs from the segment call"
            assert_close(o.float().cpu().numpy(), r, TOL_BF16, f"batch job {j}")
        assert torch.isfinite(sums[j])
    # the same batch with its arguments marshalled once, run twice into cleared outputs
    prep = g.PreparedBatch(wt, k, jobs)
    for _ in range(2):
        for job_outs in outs:
            for o in job_outs:
                o.fill_(float("nan"))
        prep.run()
        torch.cuda.synchronize()
        for j, job_outs in enumerate(outs):
            for o, s_ in zip(job_outs, sep[j]):
                assert torch.equal(o, s_), f"prepared batch job {j} differs from the segment call"


def test_decode_step_as_benchmarked_full_size_sampled(g):
    """The benchmarked decode step itself: bench.py's Decode object (Q4_K
    4096x4096 and 14336x4096, K = 4096, random packed blocks with safe scales,
    copies rotating past L2), one q8_1 quantization of the 15 activation rows,
    and the four M-products as one gguf_mul_mat_batch chain in the timed order.
    Every output matrix is checked against the oracle on 256 sampled rows plus
    the first and last, for every token."""
    import bench

    dec = bench.Decode(torch, g, synth, torch.device(DEV))
    for y in dec.ys.values():
        y.fill_(float("nan"))
    dec.step()
    torch.cuda.synchronize()
    k = dec.k
    for (n, kk) in bench.DECODE_SHAPES:
        assert kk == k
        base = synth.safe_blocks(oracle.Q4_K, n, k, seed=n)   # every rotating copy holds these bytes
        assert torch.equal(dec.pools[(n, k)][0].cpu(), torch.from_numpy(base))
        rows = np.sort(np.random.default_rng(n).choice(n, 256, replace=False))
        rows[0], rows[-1] = 0, n - 1
        for m in bench.DECODE_MS:
            xq_ref = oracle.quantize_q8_1(dec.xs[m].float().cpu().numpy())
            assert np.array_equal(dec.xqs[m].cpu().numpy(), xq_ref.reshape(m, -1)), f"q8_1 rows of M = {m}"
            ref = oracle.mul_mat(oracle.Q4_K, base[rows], k, xq_ref)
            y = dec.ys[(n, m)].float().cpu().numpy()
            assert np.isfinite(y).all(), f"{n} x {k}, M = {m}: an output was not written"
            assert_close(y[:, rows], ref, TOL_BF16, f"decode step {n} x {k}, M = {m}")


@pytest.mark.parametrize("m", [1, 2, 5, 8])
def test_mul_mat_batch_typed_mixed_types(g, m):
    """Products of different weight types and K on their q8_1 inputs in one
    chain (a layer's q + k in Q4_K and v in Q6_K on the attention input, and a
    Q8_0 product with another K): each job equals its separate segment call bit
    for bit and matches the oracle."""
    D, KV, k2 = 3072, 1024, 1024
    wq = oracle.quantize_weights(oracle.Q4_K, synth.normal((D, D), 0.02, seed=1))
    wk = oracle.quantize_weights(oracle.Q4_K, synth.normal((KV, D), 0.02, seed=2))
    wv = oracle.quantize_weights(oracle.Q6_K, synth.normal((KV, D), 0.02, seed=3))
    w8 = oracle.quantize_weights(oracle.Q8_0, synth.normal((300, k2), 0.02, seed=4))
    x = synth.activations(m, D, seed=m, dtype=torch.bfloat16)
    x2 = synth.activations(m, k2, seed=m + 9, dtype=torch.bfloat16)
    xq, xq2 = g.gguf_quantize_q8_1(x.to(DEV)), g.gguf_quantize_q8_1(x2.to(DEV))
    out = {nm: torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
           for nm, n in (("q", D), ("k", KV), ("v", KV), ("e", 300))}
    dw = {nm: _u8(w) for nm, w in (("q", wq), ("k", wk), ("v", wv), ("e", w8))}
    g.gguf_mul_mat_batch_typed([(oracle.Q4_K, D, xq, [(dw["q"], D, out["q"]), (dw["k"], KV, out["k"])]),
                                (oracle.Q6_K, D, xq, [(dw["v"], KV, out["v"])]),
                                (oracle.Q8_0, k2, xq2, [(dw["e"], 300, out["e"])])])
    sep = {nm: torch.empty_like(o) for nm, o in out.items()}
    g.gguf_mul_mat_segments(oracle.Q4_K, D, xq, [(dw["q"], D, sep["q"]), (dw["k"], KV, sep["k"])], xt=g.Q8_1, m=m)
    g.gguf_mul_mat(dw["v"], oracle.Q6_K, KV, D, xq, xt=g.Q8_1, m=m, out=sep["v"])
    g.gguf_mul_mat(dw["e"], oracle.Q8_0, 300, k2, xq2, xt=g.Q8_1, m=m, out=sep["e"])
    torch.cuda.synchronize()
    xr, xr2 = oracle.quantize_q8_1(x.float().numpy()), oracle.quantize_q8_1(x2.float().numpy())
    refs = {"q": oracle.mul_mat(oracle.Q4_K, wq, D, xr), "k": oracle.mul_mat(oracle.Q4_K, wk, D, xr),
            "v": oracle.mul_mat(oracle.Q6_K, wv, D, xr), "e": oracle.mul_mat(oracle.Q8_0, w8, k2, xr2)}
    for nm in out:
        assert torch.equal(out[nm], sep[nm]), f"{nm}: typed batch differs from the separate call"
        assert_close(out[nm].float().cpu().numpy(), refs[nm], TOL_BF16, f"typed batch {nm} m={m}")
