"""Benchmark of the GGUF block-quantized matmul hot path on GB300.

Default workload (one "step"): the decode MMVQ configuration -- Q4_K weights of
shape 4096 x 4096 and 14336 x 4096, bf16 activations with M in {1, 2, 4, 8};
the step's 15 activation rows are quantized once (bf16 -> q8_1) and both
weight matrices run the MMVQ kernel on each M's row slice, all through the
library's C ABI.  The metric is the HBM bandwidth of
the path in GB/s: algorithmic bytes (packed weights + activations + q8_1 +
outputs; the weights are >99% of them) / step time.  Weight copies rotate so
that no launch finds its weights in L2 (the rotation set is > 4x L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--no-secondary] [--no-cpu-baseline]

Beside the headline, the line carries "secondary" results measured in the same
run: the Q8_0 512x1024 product, the two prefill MMQ products (TOPS), the MoE
FFN (TOPS on routed rows) and a Llama-3.2-3B-shaped decode step of all 196
linears plus the tied LM head at M = 1, 8, 32 (GB/s of weights).

Under torchrun each rank runs the same per-GPU workload (replicas, weak
scaling); rank 0 prints one JSON line with the whole-job value.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# the headline metric's name, as the benchmark configuration states it
METRIC = "GGUF matmul: weight-read HBM GB/s (MMVQ) and int8 TOPS (MMQ/MoE) on 1 GB300"
DECODE_SHAPES = [(4096, 4096), (14336, 4096)]
DECODE_MS = [1, 2, 4, 8]
# launch order of the step's batch call: the 8-token tensor-core launch first,
# then the dp4a ones (measured on GB300: 51.1 us per step against 53.7 us in
# the order 1, 2, 4, 8)
DECODE_CHAIN = (8, 1, 2, 4)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# decode workload (MMVQ) -- the headline
# --------------------------------------------------------------------------

def _l2_bytes(torch):
    try:
        return int(torch.cuda.get_device_properties(0).L2_cache_size)
    except Exception:
        return 126 * 2 ** 20


class Decode:
    """Q4_K 4096x4096 and 14336x4096 with bf16 activations, M in {1, 2, 4, 8}.

    The step's activations (the four M-row batches, 15 rows) sit in one bf16
    matrix; one quantize pass turns all of them into q8_1, and each batch's
    row slice feeds both weight matrices (every weight that reads the same
    activations shares one quantization).  Weight copies rotate over more
    than 4x L2 per shape, so no launch finds its weights in L2.

    Each M is one segment-table MMVQ launch over both weight matrices (four
    MMVQ launches per step).  They depend only on the quantized rows, so the
    step issues them as one gguf_mul_mat_batch call: a chain of programmatic
    dependent launches in which each starts as the previous one drains, closed
    by an empty ordinary launch.  Measured on GB300 before the batch call: 59.4
    us per step on four CUDA streams, 63.1 us serially.  `mode` selects the
    batch (default), four streams ("streams") or serial segment calls
    ("serial")."""

    def __init__(self, torch, g, synth, dev):
        self.g = g
        l2 = _l2_bytes(torch)
        self.pools, self.counters = {}, {}
        for (n, k) in DECODE_SHAPES:
            rb = g.gguf_row_size(g.Q4_K, k)
            copies = max(4, -(-4 * l2 // (n * rb)))
            base = torch.from_numpy(synth.safe_blocks(g.Q4_K, n, k, seed=n)).to(dev)
            pool = torch.empty((copies, n, rb), dtype=torch.uint8, device=dev)
            for c in range(copies):
                pool[c].copy_(base)
            self.pools[(n, k)] = pool
            self.counters[(n, k)] = 0
        k = DECODE_SHAPES[0][1]
        self.k = k
        self.x_all = torch.cat([synth.activations(m, k, seed=100 + m, dtype=torch.bfloat16) for m in DECODE_MS]).to(dev)
        self.xq_all = torch.empty((self.x_all.shape[0], g.gguf_row_size(g.Q8_1, k)), dtype=torch.uint8, device=dev)
        self.rows = {}
        r0 = 0
        for m in DECODE_MS:
            self.rows[m] = (r0, r0 + m)
            r0 += m
        self.xs = {m: self.x_all[a:b] for m, (a, b) in self.rows.items()}
        self.xqs = {m: self.xq_all[a:b] for m, (a, b) in self.rows.items()}
        # all outputs in one buffer (one device-to-host read in the e2e loop)
        sizes = [(n, m) for m in DECODE_MS for (n, _) in DECODE_SHAPES]
        self.y_all = torch.empty(sum(n * m for n, m in sizes), dtype=torch.bfloat16, device=dev)
        self.ys, off = {}, 0
        for (n, m) in sizes:
            self.ys[(n, m)] = self.y_all[off:off + n * m].view(m, n)
            off += n * m
        self.n_phase = max(p.shape[0] for p in self.pools.values())
        self.torch = torch
        self.sides = [torch.cuda.Stream(device=dev) for _ in range(len(DECODE_MS) - 1)]
        # MMVQ on q8_1 input needs no workspace; passing one skips the size query
        self.ws = torch.empty(256, dtype=torch.uint8, device=dev)

    def weight(self, n, k):
        pool = self.pools[(n, k)]
        c = self.counters[(n, k)]
        self.counters[(n, k)] = (c + 1) % pool.shape[0]
        return pool[c]

    def _segments(self, ms):   # one call (and launch) per M for both weight matrices
        g = self.g
        for m in ms:
            segs = [(self.weight(n, k), n, self.ys[(n, m)]) for (n, k) in DECODE_SHAPES]
            g.gguf_mul_mat_segments(g.Q4_K, self.k, self.xqs[m], segs, xt=g.Q8_1, m=m, ws=self.ws)

    def prepared_batches(self, count):
        """`count` consecutive steps' batch calls with their arguments marshalled
        once (the weight copies rotate as in the timed step)."""
        return [self.g.PreparedBatch(self.g.Q4_K, self.k,
                                     [(self.xqs[m], [(self.weight(n, k), n, self.ys[(n, m)]) for (n, k) in DECODE_SHAPES])
                                      for m in DECODE_CHAIN])
                for _ in range(count)]

    def _batch(self, ms):   # one call: the M-products as chained launches
        self.g.gguf_mul_mat_batch(self.g.Q4_K, self.k,
                                  [(self.xqs[m], [(self.weight(n, k), n, self.ys[(n, m)]) for (n, k) in DECODE_SHAPES])
                                   for m in ms])

    def step(self, quantize=True, x_all=None, mode="batch"):
        g, torch = self.g, self.torch
        if quantize:
            g.gguf_quantize_q8_1(self.x_all if x_all is None else x_all, out=self.xq_all)
        if mode == "batch":
            self._batch(DECODE_CHAIN)
            return
        run = self._segments
        if mode == "serial":
            run(DECODE_MS)
            return
        # M = 4 on the current stream, M = 8, 2 and 1 on one side stream each
        main = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        for side, m in zip(self.sides, (8, 2, 1)):
            side.wait_event(fork)
            with torch.cuda.stream(side):
                run((m,))
        run((4,))
        for side in self.sides:
            join = torch.cuda.Event()
            join.record(side)
            main.wait_event(join)

    def mmvq_launches_per_step(self):
        return len(DECODE_MS)

    def launches_per_step(self, quantize=True):
        # the MMVQ launches, the empty launch that closes the batch, the quantize
        return self.mmvq_launches_per_step() + 1 + (1 if quantize else 0)

    def bytes_per_step(self):
        """Algorithmic bytes: packed weights + bf16 x read + q8_1 write + q8_1 read per product + y write."""
        g, k = self.g, self.k
        tot = wts = mmvq = 0
        for m in DECODE_MS:
            xq = m * g.gguf_row_size(g.Q8_1, k)
            tot += m * k * 2 + xq   # this batch's share of the quantize pass
            for (n, _) in DECODE_SHAPES:
                w = n * g.gguf_row_size(g.Q4_K, k)
                tot += w + xq + m * n * 2
                wts += w
                mmvq += w + xq + m * n * 2
        return tot, wts, mmvq


def _capture(torch, stream, fn, count):
    graphs = []
    for _ in range(count):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            fn()
        graphs.append(gr)
    return graphs


def _time_graphs(torch, stream, graphs, reps, warm=3):
    with torch.cuda.stream(stream):
        for i in range(warm):
            graphs[i % len(graphs)].replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(reps):
            graphs[i % len(graphs)].replay()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def run_ours(args, rank, world, torch, dev):
    import gguf_block_quantized_quantize_gb300 as g
    from gguf_block_quantized_quantize_gb300 import synth

    g.load_library()
    hbm_peak, tf_peak, peak_kind = _peaks()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        dec = Decode(torch, g, synth, dev)
        for _ in range(2):   # warm the launch path before capture
            dec.step()
    torch.cuda.synchronize()
    nph = min(dec.n_phase, 8)
    with torch.cuda.stream(stream):
        graphs = _capture(torch, stream, dec.step, nph)
        # the MMVQ launches alone, 8 steps per graph (the graph launch gap between
        # replays is not part of the kernels' time)
        mgraphs = _capture(torch, stream, lambda: [dec.step(quantize=False) for _ in range(8)], nph)
    torch.cuda.synchronize()
    per_step, weight_bytes, mmvq_bytes = dec.bytes_per_step()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    _barrier(world, torch)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            graphs[i % len(graphs)].replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    ms_total = ev0.elapsed_time(ev1)
    # the dominant kernel alone (MMVQ on the same q8_1 inputs, same rotation, same stream)
    ms_mmvq_step = _time_graphs(torch, stream, mgraphs, max(args.steps, 20)) / 8
    # for comparison: the same four launches as separate segment calls (no chaining)
    with torch.cuda.stream(stream):
        sgraphs = _capture(torch, stream, lambda: [dec.step(quantize=False, mode="serial") for _ in range(8)], nph)
    ms_mmvq_serial = _time_graphs(torch, stream, sgraphs, max(args.steps, 20)) / 8
    del sgraphs
    clk = clocks.stop()
    n_mmvq = dec.mmvq_launches_per_step()
    ms_mmvq = ms_mmvq_step / n_mmvq
    ms_step, value = _job_rate(ms_total, args.steps, per_step, world, torch, dev)
    achieved = (mmvq_bytes / n_mmvq) / (ms_mmvq * 1e-3) / 1e9

    # per (shape, M) detail: each MMVQ alone, 16 launches per graph
    detail = []
    for m in DECODE_MS:
        for (n, k) in DECODE_SHAPES:
            def one(n=n, k=k, m=m):
                for _ in range(16):
                    g.gguf_mul_mat(dec.weight(n, k), g.Q4_K, n, k, dec.xqs[m], xt=g.Q8_1, m=m, out=dec.ys[(n, m)])
            with torch.cuda.stream(stream):
                gr = _capture(torch, stream, one, 1)
            us = _time_graphs(torch, stream, gr, 5, warm=1) * 1e3 / 16
            by = n * g.gguf_row_size(g.Q4_K, k) + m * g.gguf_row_size(g.Q8_1, k) + m * n * 2
            detail.append({"n": n, "k": k, "m": m, "us": round(us, 3), "gbs": round(by / us / 1e3, 1),
                           "frac": round(by / us / 1e3 / hbm_peak, 3)})

    e2e = run_e2e(args, g, torch, dev, dec, per_step)

    result = {
        "metric": METRIC,
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 dot, fp32 combine", "data": "synthetic",
        "config": {"workload": "decode MMVQ: Q4_K 4096x4096 and 14336x4096, bf16 activations M in {1,2,4,8}; "
                               "step = one bf16->q8_1 quantize of the 15 activation rows, then per M one "
                               "segment-table MMVQ launch over both weight matrices (each M-row slice shared by "
                               "both), the four launches chained in one gguf_mul_mat_batch call",
                   "l2": "weight copies rotate over >4x L2 per shape (inputs larger than L2)",
                   "weights": "random-but-safe packed Q4_K blocks", "parallelism": f"replicas x{world}"},
        "weight_bytes_per_step": weight_bytes, "bytes_per_step": per_step,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": mmvq_traffic(),
                     "kernel": "MMVQ (dp4a mmvq_kernel for M<=4, int8 tensor-core for M=8), one segment-table launch "
                               "per M over both matrices, the 4 launches chained in one gguf_mul_mat_batch call "
                               "(M = 8 first); total bytes / total time of the 4, timed as 8 steps per CUDA graph",
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "frac_unchained": round(mmvq_bytes / (ms_mmvq_serial * 1e-3) / 1e9 / hbm_peak, 4)},
        "detail": detail,
        "gpu_launches": args.steps * dec.launches_per_step(),
        "clocks": clk,
        "e2e": e2e,
    }
    if not args.no_secondary:
        result["secondary"] = secondary(torch, g, synth, dev, stream, hbm_peak, tf_peak, peak_kind)
    return result


# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the
# decode MMVQ launches, averaged over the step's four segment launches, from one
# ncu capture of this bench's decode step:
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none
#       -k regex:mmvq -s 20 -c 8 python bench.py --steps 3 --warmup 3 --no-secondary --no-cpu-baseline
# together with the SHA-256 of the MMVQ sources it was taken on.  The bench
# reports the figure only while those sources are unchanged, and null otherwise.
MMVQ_TRAFFIC = {"bytes": 42528704, "sources_sha256": "dd07a10bbdcf3fa4f9dc5d2f3dd2b08587e824c26b5679504e2983bfda658b55"}
MMVQ_SOURCES = ("mmvq.cuh", "mmvq_mma.cuh", "mmvq_mma_q6k.cuh", "mmvq.cu", "mmvq_q4_k.cu", "common.cuh")


def mmvq_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for name in MMVQ_SOURCES:
        with open(os.path.join(ROOT, "gguf_block_quantized_quantize_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def mmvq_traffic():
    return MMVQ_TRAFFIC["bytes"] if MMVQ_TRAFFIC["sources_sha256"] == mmvq_sources_sha256() else None


def run_e2e(args, g, torch, dev, dec, per_step):
    """Same workload through the public API with host buffers: each step copies
    its activations from pinned host memory, quantizes them, runs the four
    M-products as one gguf_mul_mat_batch call and copies its outputs back to
    pinned host memory, on one stream.  Both copies go through gguf_copy_async
    (on the SMs, chained with the step's launches; a copy-engine copy costs
    about 5 us of latency and ends the chain).  The batch call's arguments are
    marshalled once per weight phase (PreparedBatch), as an engine replaying
    its decode step would, so the host issues four calls per step."""
    hx = dec.x_all.cpu().pin_memory()
    hy = torch.empty(dec.y_all.shape, dtype=dec.y_all.dtype).pin_memory()
    dx = torch.empty_like(dec.x_all)
    stream = torch.cuda.Stream()
    h2d = hx.numel() * hx.element_size()
    d2h = hy.numel() * hy.element_size()

    prepared = dec.prepared_batches(64)
    it = [0]

    def step():
        g.gguf_copy(dx, hx)
        g.gguf_quantize_q8_1(dx, out=dec.xq_all)
        prepared[it[0] % len(prepared)].run()
        it[0] += 1
        g.gguf_copy(hy, dec.y_all)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    return {"value": round(per_step / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 5),
            "copies": "gguf_copy_async: pinned host <-> device on the SMs, in the step's launch chain"}


# --------------------------------------------------------------------------
# secondary workloads (reported beside the headline, not part of its step)
# --------------------------------------------------------------------------

def _time_eager(torch, stream, fn, reps, flush=None, warm=2):
    """Mean device time of fn() over reps calls, CUDA events on `stream` around
    each call only; `flush` (an L2-sized write) runs between calls, untimed."""
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
        evs = []
        for _ in range(reps):
            if flush is not None:
                flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / reps


def int8_mma_peak_tops(torch):
    """The int8 warp-MMA (mma.sync m16n8k32 s8) peak: 512 ops per clock per SM
    (ncu's sm__ops_path_tensor_op_imma_src_int8 peak_sustained on GB300) x SMs x
    the maximum SM clock from the measured-peaks file."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
    except Exception:
        mhz = 2070.0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 512.0 * sms * mhz * 1e6 / 1e12


def secondary(torch, g, synth, dev, stream, hbm_peak, tf_peak, peak_kind):
    out = {}
    p_int8 = int8_mma_peak_tops(torch)
    l2 = _l2_bytes(torch)
    scrub = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def flush():
        scrub.fill_(1)

    def u8(a):
        return torch.from_numpy(a).to(dev)

    with torch.cuda.stream(stream):
        # Q8_0 512 x 1024, fp32 activations M = 8, fp32 out (a few hundred KB: launch-latency bound)
        n, k, m = 512, 1024, 8
        w = u8(synth.safe_blocks(g.Q8_0, n, k, seed=1))
        x = synth.activations(m, k, seed=2, dtype=torch.float32).to(dev)
        y = torch.empty((m, n), dtype=torch.float32, device=dev)
        ws = torch.empty(max(g.gguf_mul_mat_ws_size(g.Q8_0, n, k, g.F32, m, g.F32), 16), dtype=torch.uint8, device=dev)
        ms = _time_eager(torch, stream, lambda: g.gguf_mul_mat(w, g.Q8_0, n, k, x, out=y, ws=ws), 20, flush)
        out["q8_0_512x1024_m8_f32"] = {"us": round(ms * 1e3, 2), "note": "quantize + MMVQ, L2 flushed between calls"}
        del w

        # prefill MMQ: Q4_K 8192x2048 @ 8192 bf16 tokens, Q6_K 248320x2048 @ 2048, bf16 out
        for name, wt, n, k, m in (("mmq_q4_k_8192x2048_m8192", g.Q4_K, 8192, 2048, 8192),
                                  ("mmq_q6_k_248320x2048_m2048", g.Q6_K, 248320, 2048, 2048)):
            w = synth.safe_blocks_device(wt, n, k, seed=n, device=dev)
            x = synth.activations(m, k, seed=3, dtype=torch.bfloat16).to(dev)
            y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            ws = torch.empty(max(g.gguf_mul_mat_ws_size(wt, n, k, g.BF16, m, g.BF16), 16), dtype=torch.uint8,
                             device=dev)
            ms = _time_eager(torch, stream, lambda: g.gguf_mul_mat(w, wt, n, k, x, out=y, ws=ws), 5, flush)
            tops = 2.0 * m * n * k / (ms * 1e-3) / 1e12
            # the alternative engine on the same product: dequantize to fp16 + one library GEMM
            g.gguf_set_option("mmq_engine", 1)
            try:
                ws1 = torch.empty(max(g.gguf_mul_mat_ws_size(wt, n, k, g.BF16, m, g.BF16), 16), dtype=torch.uint8,
                                  device=dev)
                ms1 = _time_eager(torch, stream, lambda: g.gguf_mul_mat(w, wt, n, k, x, out=y, ws=ws1), 5, flush)
                # with fp16 outputs the library GEMM writes them directly (no fp32 rows)
                y16 = torch.empty((m, n), dtype=torch.float16, device=dev)
                ms2 = _time_eager(torch, stream, lambda: g.gguf_mul_mat(w, wt, n, k, x, out=y16, ws=ws1), 5, flush)
                lib_engine = {"ms": round(ms1, 4), "tops": round(2.0 * m * n * k / (ms1 * 1e-3) / 1e12, 1),
                              "ms_f16_out": round(ms2, 4),
                              "note": "option mmq_engine = 1: weights dequantized to fp16 in the workspace, then one "
                                      "cuBLAS fp16 GEMM (fp32 accumulation) on the q8_1 operand, fp32 rows converted "
                                      "to bf16; includes the dequantize"}
                del ws1, y16
            except Exception as exc:   # cuBLAS not loadable: reported, the fused number stands
                lib_engine = {"unavailable": str(exc)[:200]}
            finally:
                g.gguf_set_option("mmq_engine", 0)
            out[name] = {"ms": round(ms, 4), "tops": round(tops, 1), "library_engine": lib_engine,
                         "rate": "algorithmic 2*m*n*k ops/s (int8-equivalent); computed as fp16 tcgen05 MMAs of "
                                 "the dequantized operands",
                         "roofline": {"bound": "tensor", "achieved": round(tops, 1), "peak": tf_peak,
                                      "unit": "TFLOP/s", "frac": round(tops / tf_peak, 4),
                                      "note": f"fp16 tcgen05 MMA; peak = {peak_kind} bf16 (same rate as fp16)"},
                         "frac_of_int8_mma_peak": round(tops / p_int8, 3), "int8_mma_peak_tops": round(p_int8, 1)}
            del w, x, y, ws

        # MoE FFN: E=256, top-8, H=2048, I=512, 8192 bf16 tokens; gate_up Q4_K, down Q6_K
        E, H, I, T, K_ = 256, 2048, 512, 8192, 8
        wgu = synth.safe_blocks_device(g.Q4_K, E * 2 * I, H, seed=5, device=dev)
        wdn = synth.safe_blocks_device(g.Q6_K, E * H, I, seed=6, device=dev)
        ids_np, rw_np = synth.routes(T, E, K_, seed=7)
        ids, rw = torch.from_numpy(ids_np).to(dev), torch.from_numpy(rw_np).to(dev)
        x = synth.activations(T, H, seed=8, dtype=torch.bfloat16).to(dev)
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        gu_stride, dn_stride = 2 * I * g.gguf_row_size(g.Q4_K, H), H * g.gguf_row_size(g.Q6_K, I)
        args = g.moe_ffn_args(wgu, g.Q4_K, gu_stride, wdn, g.Q6_K, dn_stride, E, H, I, x, g.BF16, ids, K_, rw, y,
                              g.BF16, None)
        ws = torch.empty(max(g.gguf_moe_ffn_ws_size(args), 16), dtype=torch.uint8, device=dev)

        def moe():
            g.gguf_moe_ffn(wgu, g.Q4_K, gu_stride, wdn, g.Q6_K, dn_stride, E, H, I, x, ids, rw, out=y, ws=ws)
        ms = _time_eager(torch, stream, moe, 5, flush)
        ops = 2.0 * T * K_ * (2 * I * H + H * I)
        out["moe_ffn_e256_top8_h2048_i512_t8192"] = {
            "ms": round(ms, 4), "tops": round(ops / (ms * 1e-3) / 1e12, 1),
            "frac_of_bf16_peak": round(ops / (ms * 1e-3) / 1e12 / tf_peak, 4),
            "frac_of_int8_mma_peak": round(ops / (ms * 1e-3) / 1e12 / p_int8, 3),
            "note": "routed-row int8-equivalent ops 2*T*top_k*(2I*H + H*I) / time, computed as fp16 tcgen05 MMAs "
                    "of the dequantized operands; gate_up Q4_K + SwiGLU + q8_1, down Q6_K + weighted sum"}
        # the same expert block at decode token counts: the route-batched MMVQ path (each routed
        # expert's rows read once per route); GB/s of the routed experts' packed weights
        for Td in (1, 16):
            ids_np, rw_np = synth.routes(Td, E, K_, seed=11 + Td)
            ids_d, rw_d = torch.from_numpy(ids_np).to(dev), torch.from_numpy(rw_np).to(dev)
            xd = synth.activations(Td, H, seed=12, dtype=torch.bfloat16).to(dev)
            yd = torch.empty((Td, H), dtype=torch.bfloat16, device=dev)
            args_d = g.moe_ffn_args(wgu, g.Q4_K, gu_stride, wdn, g.Q6_K, dn_stride, E, H, I, xd, g.BF16, ids_d, K_,
                                    rw_d, yd, g.BF16, None)
            ws_d = torch.empty(max(g.gguf_moe_ffn_ws_size(args_d), 16), dtype=torch.uint8, device=dev)

            def moe_dec():
                g.gguf_moe_ffn(wgu, g.Q4_K, gu_stride, wdn, g.Q6_K, dn_stride, E, H, I, xd, ids_d, rw_d, out=yd,
                               ws=ws_d)
            ms = _time_eager(torch, stream, moe_dec, 20, flush)
            routed = Td * K_ * (gu_stride + dn_stride)   # each route reads its expert's matrices once
            out[f"moe_ffn_decode_e256_top8_t{Td}"] = {
                "us": round(ms * 1e3, 2), "routed_weight_mb": round(routed / 1e6, 2),
                "gbs": round(routed / (ms * 1e-3) / 1e9, 1), "frac": round(routed / (ms * 1e-3) / 1e9 / hbm_peak, 3),
                "note": "route-batched MMVQ path (quantize with the route marks, gate_up, SwiGLU + q8_1, down, weighted sum)"}
        del wgu, wdn, x, y, ws

        # dequantize (a whole Q4_K / Q6_K matrix to bf16) and get_rows (8192 random rows of a Q6_K
        # embedding table to bf16): HBM-bound, reported as GB/s of packed bytes read + values written
        for name, wt, n, k in (("dequantize_q4_k_14336x4096_bf16", g.Q4_K, 14336, 4096),
                               ("dequantize_q6_k_14336x4096_bf16", g.Q6_K, 14336, 4096)):
            w = synth.safe_blocks_device(wt, n, k, seed=9, device=dev)
            y = torch.empty((n, k), dtype=torch.bfloat16, device=dev)
            ms = _time_eager(torch, stream, lambda: g.gguf_dequantize(w, wt, n, k, out=y), 10, flush)
            by = w.numel() + y.numel() * 2
            out[name] = {"us": round(ms * 1e3, 2), "gbs": round(by / (ms * 1e-3) / 1e9, 1),
                         "frac": round(by / (ms * 1e-3) / 1e9 / hbm_peak, 3), "bytes": by}
            del w, y
        V, D, NI = 128256, 3072, 8192
        table = synth.safe_blocks_device(g.Q6_K, V, D, seed=10, device=dev)
        ids = torch.randint(0, V, (NI,), dtype=torch.int32, device=dev)
        y = torch.empty((NI, D), dtype=torch.bfloat16, device=dev)
        ms = _time_eager(torch, stream, lambda: g.gguf_get_rows(table, g.Q6_K, V, D, ids, out=y), 10, flush)
        by = NI * g.gguf_row_size(g.Q6_K, D) + NI * 4 + y.numel() * 2
        out["get_rows_q6_k_128256x3072_8192ids_bf16"] = {
            "us": round(ms * 1e3, 2), "gbs": round(by / (ms * 1e-3) / 1e9, 1),
            "frac": round(by / (ms * 1e-3) / 1e9 / hbm_peak, 3), "bytes": by}
        del table, ids, y

        # decode MMVQ of every weight type: 14336 x 4096 at 1 and 8 tokens (pre-quantized q8_1,
        # bf16 out), graph-timed with the weights rotating over more than 4x L2; GB/s of weights
        n, k = 14336, 4096
        types = {}
        for tname, wt in (("q4_0", g.Q4_0), ("q4_k", g.Q4_K), ("q5_k", g.Q5_K), ("q6_k", g.Q6_K), ("q8_0", g.Q8_0),
                          ("mxfp4", g.MXFP4)):
            wb = n * g.gguf_row_size(wt, k)
            copies = [synth.safe_blocks_device(wt, n, k, seed=20 + i, device=dev) for i in range(int(4 * l2 // wb) + 2)]
            res = {}
            for m in (1, 8):
                xq = g.gguf_quantize_q8_1(synth.activations(m, k, seed=m, dtype=torch.bfloat16).to(dev))
                y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                wsz = torch.empty(max(g.gguf_mul_mat_ws_size(wt, n, k, g.Q8_1, m, g.BF16), 16), dtype=torch.uint8,
                                  device=dev)
                idx = [0]

                def one():
                    idx[0] = (idx[0] + 1) % len(copies)
                    g.gguf_mul_mat(copies[idx[0]], wt, n, k, xq, xt=g.Q8_1, m=m, out=y, ws=wsz)
                one()
                graphs = _capture(torch, stream, lambda: [one() for _ in range(16)], (len(copies) + 15) // 16)
                us = _time_graphs(torch, stream, graphs, 4 * len(graphs), warm=2) * 1e3 / 16
                res[f"m{m}"] = {"us": round(us, 2), "gbs": round(wb / us / 1e3, 1), "frac": round(wb / us / 1e3 / hbm_peak, 3)}
                del graphs
            types[tname] = res
            del copies
        out["mmvq_types_14336x4096"] = dict(types, note="GB/s of packed weights; q8_1 input, bf16 out, graph-timed, "
                                                         "weights rotating past L2")

        # Llama-3.2-3B-shaped decode step: 28 layers of q/k/o/gate/up (Q4_K) and v/down (Q6_K), tied
        # Q6_K embedding / LM head 128256 x 3072 via get_rows + MMVQ; all linears at M in {1, 8, 32}
        out["llama32_3b_decode_linears"] = llama_decode(torch, g, synth, dev, stream, hbm_peak)
    torch.cuda.synchronize()
    return out


def llama_decode(torch, g, synth, dev, stream, hbm_peak):
    L, D, F, V, KV = 28, 3072, 8192, 128256, 1024
    Q4, Q6 = g.Q4_K, g.Q6_K
    layer_shapes = [("q", Q4, D, D), ("k", Q4, KV, D), ("v", Q6, KV, D), ("o", Q4, D, D),
                    ("gate", Q4, F, D), ("up", Q4, F, D), ("down", Q6, D, F)]
    layers = []
    seed = 1000
    for _ in range(L):
        ly = {}
        for nm, wt, n, k in layer_shapes:
            ly[nm] = synth.safe_blocks_device(wt, n, k, seed=seed, device=dev)
            seed += 1
        layers.append(ly)
    emb = synth.safe_blocks_device(Q6, V, D, seed=seed, device=dev)
    wbytes = sum(t.numel() for ly in layers for t in ly.values()) + emb.numel()
    res = []
    for m in (1, 8, 32):
        ids = torch.randint(0, V, (m,), dtype=torch.int32, device=dev)
        h = torch.empty((m, D), dtype=torch.bfloat16, device=dev)
        act_d = synth.activations(m, D, seed=m, dtype=torch.bfloat16).to(dev)
        act_f = synth.activations(m, F, seed=m + 1, dtype=torch.bfloat16).to(dev)
        xq_d = torch.empty((m, g.gguf_row_size(g.Q8_1, D)), dtype=torch.uint8, device=dev)
        xq_f = torch.empty((m, g.gguf_row_size(g.Q8_1, F)), dtype=torch.uint8, device=dev)
        outs = {nm: torch.empty((m, n), dtype=torch.bfloat16, device=dev) for nm, _, n, _ in layer_shapes}
        logits = torch.empty((m, V), dtype=torch.bfloat16, device=dev)
        wsz = max(g.gguf_mul_mat_ws_size(wt, n, k, g.Q8_1, m, g.BF16) for _, wt, n, k in layer_shapes)
        wsz = max(wsz, g.gguf_mul_mat_ws_size(Q6, V, D, g.Q8_1, m, g.BF16), 16)
        ws = torch.empty(wsz, dtype=torch.uint8, device=dev)

        def mm(w, wt, n, k, xq, out):
            g.gguf_mul_mat(w, wt, n, k, xq, xt=g.Q8_1, m=m, out=out, ws=ws)

        def seg(wt, k, xq, parts):   # weight matrices of one type on one input: one call
            g.gguf_mul_mat_segments(wt, k, xq, [(ly_w, n, o) for (ly_w, n, o) in parts], xt=g.Q8_1, m=m, ws=ws)

        def step():
            g.gguf_get_rows(emb, Q6, V, D, ids, out=h)           # token embedding rows
            for ly in layers:
                g.gguf_quantize_q8_1(act_d, out=xq_d)              # attention input, shared by q, k, v
                seg(Q4, D, xq_d, [(ly["q"], D, outs["q"]), (ly["k"], KV, outs["k"])])
                mm(ly["v"], Q6, KV, D, xq_d, outs["v"])
                g.gguf_quantize_q8_1(act_d, out=xq_d)              # attention output
                mm(ly["o"], Q4, D, D, xq_d, outs["o"])
                g.gguf_quantize_q8_1(act_d, out=xq_d)              # FFN input, shared by gate and up
                seg(Q4, D, xq_d, [(ly["gate"], F, outs["gate"]), (ly["up"], F, outs["up"])])
                g.gguf_quantize_q8_1(act_f, out=xq_f)              # FFN hidden
                mm(ly["down"], Q6, D, F, xq_f, outs["down"])
            g.gguf_quantize_q8_1(act_d, out=xq_d)
            mm(emb, Q6, V, D, xq_d, logits)                        # tied LM head

        # M = 32 runs under the default dispatch, and once more with the Q4_K
        # products on the 4-n-tile tensor-core MMVQ instead of MMQ
        variants = [("default", None)] + ([("mmvq_tc_max_m=32", 32)] if m > 16 else [])
        for label, tc_max in variants:
            saved = g.gguf_get_option("mmvq_tc_max_m")
            if tc_max is not None:
                g.gguf_set_option("mmvq_tc_max_m", tc_max)
            try:
                step()
                torch.cuda.synchronize()
                gr = _capture(torch, stream, step, 1)
                ms = _time_graphs(torch, stream, gr, 10, warm=2)
            finally:
                g.gguf_set_option("mmvq_tc_max_m", saved)
            gbs = wbytes / (ms * 1e-3) / 1e9
            res.append({"m": m, "dispatch": label, "ms": round(ms, 4), "weight_gb": round(wbytes / 1e9, 3),
                        "gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 3)})
            del gr
    return res


# --------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same workload
# --------------------------------------------------------------------------

class OracleDecode:
    """The decode MMVQ workload (Q4_K 4096x4096 and 14336x4096, bf16
    activations at M = 1, 2, 4, 8) on the oracle: one step quantizes each M's
    rows to q8_1 and computes all eight products in fp64, like the GPU step."""

    def __init__(self):
        import oracle
        import torch
        from gguf_block_quantized_quantize_gb300 import synth
        self.o = oracle
        k = DECODE_SHAPES[0][1]
        self.k = k
        self.w = {n: synth.safe_blocks(oracle.Q4_K, n, k, seed=n) for (n, _) in DECODE_SHAPES}
        self.x = {m: synth.activations(m, k, seed=100 + m, dtype=torch.bfloat16).float().numpy() for m in DECODE_MS}
        rb, qb = oracle.row_size(oracle.Q4_K, k), oracle.row_size(oracle.Q8_1, k)
        # the GPU step's algorithmic bytes: packed weights, bf16 x read, q8_1 written and read, bf16 y
        self.bytes = sum(m * k * 2 + m * qb + sum(n * rb + m * qb + m * n * 2 for (n, _) in DECODE_SHAPES)
                         for m in DECODE_MS)

    def step(self, nthreads):
        """Seconds per (n, M) product (its quantize included) and in total."""
        o, per = self.o, {}
        t_all = time.perf_counter()
        for m in DECODE_MS:
            t0 = time.perf_counter()
            xq = o.quantize_q8_1(self.x[m])
            tq = time.perf_counter() - t0
            for i, (n, _) in enumerate(DECODE_SHAPES):
                t0 = time.perf_counter()
                o.mul_mat(o.Q4_K, self.w[n], self.k, xq, nthreads=nthreads)
                per[f"{n}x{self.k}_m{m}"] = time.perf_counter() - t0 + (tq if i == 0 else 0.0)
        return per, time.perf_counter() - t_all


def _sub_rows(n, frac):
    return max(1, min(n, int(round(n * frac))))


def _time_rows(o, wt, w, k, xq, frac, nthreads):
    """Seconds for all rows of W . xq, extrapolated from the first n * frac rows."""
    n = w.shape[0]
    r = _sub_rows(n, frac)
    t0 = time.perf_counter()
    o.mul_mat(wt, w[:r], k, xq, nthreads=nthreads)
    return (time.perf_counter() - t0) * n / r


def cpu_baseline():
    """The oracle (scalar C, fp64 accumulation of the blockwise sums) on this
    host's cores, one entry per workload, single-threaded and on every core.
    The decode MMVQ step and the Q8_0 product run in full; the prefill MMQ
    products, the MoE block and the Llama-shaped step run on seeded row, token
    or layer subsets and are extrapolated linearly (the oracle's cost is
    proportional to rows x tokens); each entry states its sample.  The line's
    value is the decode MMVQ step on every core, in the GPU step's unit."""
    import oracle as o
    import torch
    from gguf_block_quantized_quantize_gb300 import synth

    cores = os.cpu_count() or 1
    t_begin = time.perf_counter()
    out = {}

    # Q8_0 512 x 1024, fp32 activations M = 8, fp32 out: in full, 5 calls each
    n, k, m = 512, 1024, 8
    w = synth.safe_blocks(o.Q8_0, n, k, seed=1)
    x = synth.activations(m, k, seed=2, dtype=torch.float32).numpy()
    e = {"sample": "in full (q8_1 quantize + fp64 blockwise product), median of 5 calls"}
    for label, nt in (("1t", 1), ("all", cores)):
        ts = []
        for _ in range(5):
            t0 = time.perf_counter()
            o.mul_mat(o.Q8_0, w, k, o.quantize_q8_1(x), nthreads=nt)
            ts.append(time.perf_counter() - t0)
        e[f"us_{label}"] = round(statistics.median(ts) * 1e6, 1)
    out["q8_0_512x1024_m8_f32"] = e

    # decode MMVQ: the whole step, single-threaded and on every core
    dec = OracleDecode()
    e = {"sample": "in full: q8_1 quantize of each M + all 8 products per step", "bytes_per_step": dec.bytes}
    for label, nt in (("1t", 1), ("all", cores)):
        per, tot = dec.step(nt)
        e[f"ms_{label}"] = round(tot * 1e3, 2)
        e[f"gbs_{label}"] = round(dec.bytes / tot / 1e9, 4)
        e[f"product_ms_{label}"] = {kk: round(v * 1e3, 2) for kk, v in per.items()}
    out["decode_mmvq_q4_k"] = e
    headline = e["gbs_all"]

    # prefill MMQ: row subsets, the q8_1 quantize of all tokens timed in full
    for name, wt, n, k, m, fr1, fra in (("mmq_q4_k_8192x2048_m8192", o.Q4_K, 8192, 2048, 8192, 4, 8),
                                        ("mmq_q6_k_248320x2048_m2048", o.Q6_K, 248320, 2048, 2048, 16, 16)):
        x = synth.activations(m, k, seed=3, dtype=torch.bfloat16).float().numpy()
        t0 = time.perf_counter()
        xq = o.quantize_q8_1(x)
        tq = time.perf_counter() - t0
        w = synth.safe_blocks(wt, max(fr1, fra * cores), k, seed=n)
        e = {"quantize_s": round(tq, 3)}
        for label, nt, rows in (("1t", 1, fr1), ("all", cores, fra * cores)):
            t0 = time.perf_counter()
            o.mul_mat(wt, w[:rows], k, xq, nthreads=nt)
            t = tq + (time.perf_counter() - t0) * n / rows
            e[f"s_{label}"] = round(t, 2)
            e[f"tops_{label}"] = round(2.0 * m * n * k / t / 1e12, 6)
        e["sample"] = (f"rows 0..{fr1} (1 thread) and 0..{fra * cores} (all cores) of {n}, each x all {m} tokens, "
                       f"time x {n} / rows + the full quantize")
        out[name] = e
        del w, x, xq

    # MoE FFN: all routes of a token subset through gate_up (Q4_K) + SwiGLU + q8_1 and down (Q6_K) +
    # weighted sum; ops as on the GPU, 2 * T * top_k * (2I * H + H * I)
    E, H, I, T, K_ = 256, 2048, 512, 8192, 8
    wgu = synth.safe_blocks(o.Q4_K, E * 2 * I, H, seed=5)
    wdn = synth.safe_blocks(o.Q6_K, E * H, I, seed=6)
    gs, ds = 2 * I * o.row_size(o.Q4_K, H), H * o.row_size(o.Q6_K, I)
    ids, rw = synth.routes(T, E, K_, seed=7)
    ops = 2.0 * T * K_ * (2 * I * H + H * I)
    e = {}
    for label, nt, ts in (("1t", 1, 2), ("all", cores, 4 * cores)):
        x = synth.activations(ts, H, seed=8, dtype=torch.bfloat16).float().numpy()
        t0 = time.perf_counter()
        xq = o.quantize_q8_1(x)
        _, hq = o.moe_gate_up(o.Q4_K, wgu, E, gs, 2 * I, H, xq, ids[:ts], nthreads=nt)
        o.moe_down(o.Q6_K, wdn, E, ds, H, I, hq, ids[:ts], rw[:ts], nthreads=nt)
        t = (time.perf_counter() - t0) * T / ts
        e[f"s_{label}"] = round(t, 2)
        e[f"tops_{label}"] = round(ops / t / 1e12, 6)
        e[f"tokens_{label}"] = ts
    e["sample"] = f"the first tokens_1t / tokens_all of {T} tokens (all {K_} routes each), time x {T} / tokens"
    out["moe_ffn_e256_top8_h2048_i512_t8192"] = e
    del wgu, wdn

    # Llama-3.2-3B-shaped decode step: one layer's seven linears (+ the four q8_1 quantizes) stand
    # for all 28 (same shapes, same cost), the LM head on a row subset; GB/s of all 28 layers'
    # weights + the head, as on the GPU
    L, D, F, V, KV = 28, 3072, 8192, 128256, 1024
    shapes = [("q", o.Q4_K, D, D), ("k", o.Q4_K, KV, D), ("v", o.Q6_K, KV, D), ("o", o.Q4_K, D, D),
              ("gate", o.Q4_K, F, D), ("up", o.Q4_K, F, D), ("down", o.Q6_K, D, F)]
    layer = {nm: synth.safe_blocks(wt, n, k, seed=1000 + i) for i, (nm, wt, n, k) in enumerate(shapes)}
    head_rows = max(_sub_rows(V, 1.0 / 16), 1)
    head = synth.safe_blocks(o.Q6_K, head_rows, D, seed=2000)
    wbytes = L * sum(v.nbytes for v in layer.values()) + V * o.row_size(o.Q6_K, D)
    rows = []
    for m in (1, 8, 32):
        xd = synth.activations(m, D, seed=m, dtype=torch.bfloat16).float().numpy()
        xf = synth.activations(m, F, seed=m + 1, dtype=torch.bfloat16).float().numpy()
        r = {"m": m}
        for label, nt, frac, hfrac in (("1t", 1, 1.0 / 16, 1.0 / 16), ("all", cores, 1.0, 1.0)):
            t0 = time.perf_counter()
            xqd = o.quantize_q8_1(xd)
            t_layer = 3 * (time.perf_counter() - t0)   # three quantizes of D-long rows per layer
            t0 = time.perf_counter()
            xqf = o.quantize_q8_1(xf)
            t_layer += time.perf_counter() - t0
            for nm, wt, n, k in shapes:
                t_layer += _time_rows(o, wt, layer[nm], k, xqf if k == F else xqd, frac, nt)
            t_head = _time_rows(o, o.Q6_K, head, D, xqd, hfrac, nt) * V / head_rows
            t = L * t_layer + t_head
            r[f"ms_{label}"] = round(t * 1e3, 1)
            r[f"gbs_{label}"] = round(wbytes / t / 1e9, 4)
        rows.append(r)
    out["llama32_3b_decode_linears"] = {
        "steps": rows, "weight_gb": round(wbytes / 1e9, 3),
        "sample": f"one layer's 7 linears x {L} (1 thread: rows 0..n/16 of each, x 16) + LM head rows "
                  f"0..{head_rows} of {V} (1 thread: 0..{_sub_rows(head_rows, 1.0 / 16)}), scaled to {V}"}

    return {"value": headline, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"decode MMVQ step in full (Q4_K 4096x4096 and 14336x4096 x M in {{1,2,4,8}}, q8_1 quantize "
                      f"+ fp64 blockwise products) on {cores} threads; per-workload entries in 'workloads'",
            "wall_s": round(time.perf_counter() - t_begin, 1), "workloads": out}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is the whole decode MMVQ step
    (the headline workload, in full) on every host core."""
    if rank != 0:
        return None
    cores = os.cpu_count() or 1
    dec = OracleDecode()
    for _ in range(args.warmup):
        dec.step(cores)
    t = [dec.step(cores)[1] for _ in range(args.steps)]
    ms = statistics.median(t) * 1e3
    v = round(dec.bytes / (ms * 1e-3) / 1e9, 4)
    sample = (f"decode MMVQ step in full per step (Q4_K 4096x4096 and 14336x4096 x M in {{1,2,4,8}}, q8_1 quantize + "
              f"fp64 blockwise products) on {cores} threads")
    return {"impl": "reference", "metric": METRIC,
            "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode MMVQ: Q4_K 4096x4096 and 14336x4096, bf16 activations M in {1,2,4,8}; "
                                   "oracle on the host cores"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------------

def _barrier(world, torch):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v, world, torch, dev):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(ms_total, steps, bytes_per_step, world, torch, dev):
    """Whole-job rate of `world` replicas: every rank processed bytes_per_step
    per step, and the job took the slowest rank's time.  Returns (ms per step,
    GB/s over all ranks)."""
    ms_step = _max_over_ranks(ms_total, world, torch, dev) / steps
    return ms_step, bytes_per_step * world / (ms_step * 1e-3) / 1e9


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true", help="skip the MMQ / MoE / Llama-shaped results")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0

    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    res = run_ours(args, rank, world, torch, dev)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
