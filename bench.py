"""Benchmark of the GGUF block-quantized matmul hot path on GB300.

Default workload (one "step"): the decode MMVQ configuration -- Q4_K weights of
shape 4096 x 4096 and 14336 x 4096, bf16 activations with M in {1, 2, 4, 8};
each of the 8 products runs the whole path (bf16 -> q8_1 quantization, then the
MMVQ kernel) through the library's C ABI.  The metric is the HBM bandwidth of
the path in GB/s: algorithmic bytes (packed weights + activations + q8_1 +
outputs; the weights are >99% of them) / step time.  Weight copies rotate so
that no launch finds its weights in L2 (the rotation set is > 4x L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload decode|mmq|moe|llama]

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

DECODE_SHAPES = [(4096, 4096), (14336, 4096)]
DECODE_MS = [1, 2, 4, 8]


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
# decode workload (MMVQ)
# --------------------------------------------------------------------------

def _l2_bytes(torch):
    try:
        return int(torch.cuda.get_device_properties(0).L2_cache_size)
    except Exception:
        return 126 * 2 ** 20


def decode_setup(torch, g, synth, dev):
    """Weight copies (random-but-safe Q4_K blocks), activations and outputs."""
    l2 = _l2_bytes(torch)
    plan = []
    pools = {}
    for (n, k) in DECODE_SHAPES:
        rb = g.gguf_row_size(g.Q4_K, k)
        nbytes = n * rb
        copies = max(4, -(-4 * l2 // nbytes))
        base = torch.from_numpy(synth.safe_blocks(g.Q4_K, n, k, seed=n)).to(dev)
        pool = torch.empty((copies, n, rb), dtype=torch.uint8, device=dev)
        for c in range(copies):
            pool[c].copy_(base)
        pools[(n, k)] = pool
    xs, ys = {}, {}
    for (n, k) in DECODE_SHAPES:
        for m in DECODE_MS:
            xs[(n, k, m)] = synth.activations(m, k, seed=100 + m, dtype=torch.bfloat16).to(dev)
            ys[(n, k, m)] = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            plan.append((n, k, m))
    ws = torch.empty(g.gguf_mul_mat_ws_size(g.Q4_K, 14336, 4096, g.BF16, 8) + 4096, dtype=torch.uint8, device=dev)
    xqs = {key: torch.empty((key[2], g.gguf_row_size(g.Q8_1, key[1])), dtype=torch.uint8, device=dev) for key in plan}
    return plan, pools, xs, ys, ws, xqs


def decode_bytes(g, n, k, m):
    w = n * g.gguf_row_size(g.Q4_K, k)
    xq = m * g.gguf_row_size(g.Q8_1, k)
    return {"weights": w, "x_bf16": m * k * 2, "xq_write": xq, "xq_read": xq, "y": m * n * 2,
            "mmvq": w + xq + m * n * 2}


def run_ours(args, rank, world, torch, dev):
    import gguf_block_quantized_quantize_gb300 as g
    from gguf_block_quantized_quantize_gb300 import synth

    g.load_library()
    hbm_peak, _, peak_kind = _peaks()
    plan, pools, xs, ys, ws, xqs = decode_setup(torch, g, synth, dev)
    counters = {key: 0 for key in pools}

    def weight(n, k):
        pool = pools[(n, k)]
        c = counters[(n, k)]
        counters[(n, k)] = (c + 1) % pool.shape[0]
        return pool[c]

    # one step = 8 products, each quantize + MMVQ through the C ABI
    def step():
        for (n, k, m) in plan:
            g.gguf_mul_mat(weight(n, k), g.Q4_K, n, k, xs[(n, k, m)], out=ys[(n, k, m)], ws=ws)

    # the MMVQ kernels alone (pre-quantized q8_1 input), for the roofline
    for (n, k, m) in plan:
        g.gguf_quantize_q8_1(xs[(n, k, m)], out=xqs[(n, k, m)])

    def mmvq_only():
        for (n, k, m) in plan:
            g.gguf_mul_mat(weight(n, k), g.Q4_K, n, k, xqs[(n, k, m)], xt=g.Q8_1, m=m, out=ys[(n, k, m)])

    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    # CUDA graphs: one graph per rotation phase so that every replay reads new copies
    n_phase = max(p.shape[0] for p in pools.values())
    graphs, mgraphs = [], []
    with torch.cuda.stream(stream):
        for _ in range(2):   # warm the launch path before capture
            step()
        torch.cuda.synchronize()
        for i in range(min(n_phase, 8)):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                step()
            graphs.append(gr)
        for i in range(min(n_phase, 8)):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                mmvq_only()
            mgraphs.append(gr)
    torch.cuda.synchronize()

    per_step = sum(sum(v for kk, v in decode_bytes(g, n, k, m).items() if kk in ("weights", "x_bf16", "xq_write", "xq_read", "y")) for (n, k, m) in plan)
    weight_bytes = sum(decode_bytes(g, n, k, m)["weights"] for (n, k, m) in plan)

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
    # dominant kernel: MMVQ launches alone, same stream, same rotation
    reps = max(args.steps, 20)
    with torch.cuda.stream(stream):
        for i in range(3):
            mgraphs[i % len(mgraphs)].replay()
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        for i in range(reps):
            mgraphs[i % len(mgraphs)].replay()
        m1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_mmvq = m0.elapsed_time(m1) / (reps * len(plan))
    ms_total = _max_over_ranks(ms_total, world, torch, dev)
    ms_step = ms_total / args.steps
    value = per_step * world / (ms_step * 1e-3) / 1e9
    mmvq_bytes = sum(decode_bytes(g, n, k, m)["mmvq"] for (n, k, m) in plan) / len(plan)
    achieved = mmvq_bytes / (ms_mmvq * 1e-3) / 1e9

    # per-shape detail: each (shape, m) MMVQ alone
    detail = []
    for (n, k, m) in plan:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gr, stream=stream):
                for _ in range(16):
                    g.gguf_mul_mat(weight(n, k), g.Q4_K, n, k, xqs[(n, k, m)], xt=g.Q8_1, m=m, out=ys[(n, k, m)])
            gr.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(5):
                gr.replay()
            b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / 80
        by = decode_bytes(g, n, k, m)["mmvq"]
        detail.append({"n": n, "k": k, "m": m, "us": round(us, 3), "gbs": round(by / us / 1e3, 1),
                       "frac": round(by / us / 1e3 / hbm_peak, 3)})

    e2e = run_e2e(args, g, torch, dev, plan, xs, ys, weight, per_step, ws)

    result = {
        "metric": "GGUF matmul: weight-read HBM GB/s (MMVQ) and int8 TOPS (MMQ/MoE) on 1 GB300",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8", "data": "synthetic",
        "config": {"workload": "decode MMVQ: Q4_K 4096x4096 and 14336x4096, bf16 activations M in {1,2,4,8}; "
                               "step = 8 x (bf16->q8_1 quantize + MMVQ)",
                   "l2": "weight copies rotate over >4x L2 per shape (inputs larger than L2)",
                   "weights": "random-but-safe packed Q4_K blocks", "parallelism": f"replicas x{world}"},
        "weight_bytes_per_step": weight_bytes, "bytes_per_step": per_step,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": None, "kernel": "mmvq_kernel (Q4_K)",
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "detail": detail,
        "gpu_launches": args.steps * 2 * len(plan),
        "clocks": clk,
        "e2e": e2e,
    }
    return result


def run_e2e(args, g, torch, dev, plan, xs, ys, weight, per_step, ws):
    """Same workload through the public API with host buffers: the step's
    activations are copied from pinned host memory and its outputs read back."""
    hx = {key: xs[key].cpu().pin_memory() for key in plan}
    hy = {key: torch.empty(ys[key].shape, dtype=ys[key].dtype).pin_memory() for key in plan}
    dx = {key: torch.empty_like(xs[key]) for key in plan}
    stream = torch.cuda.Stream()
    h2d = sum(hx[k].numel() * hx[k].element_size() for k in plan)
    d2h = sum(hy[k].numel() * hy[k].element_size() for k in plan)

    def step():
        for key in plan:
            dx[key].copy_(hx[key], non_blocking=True)
        for (n, k, m) in plan:
            g.gguf_mul_mat(weight(n, k), g.Q4_K, n, k, dx[(n, k, m)], out=ys[(n, k, m)], ws=ws)
        for key in plan:
            hy[key].copy_(ys[key], non_blocking=True)

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
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 5)}


# --------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same workload
# --------------------------------------------------------------------------

def cpu_baseline(budget_s: float = 15.0):
    import oracle
    from gguf_block_quantized_quantize_gb300 import synth

    cores = os.cpu_count() or 1
    n, k, m = 4096, 4096, 8
    w = synth.safe_blocks(oracle.Q4_K, n, k, seed=n)
    x = synth.activations(m, k, seed=108, dtype=__import__("torch").bfloat16).float().numpy()
    rows = 64
    done_bytes, t0 = 0, time.perf_counter()
    rb = oracle.row_size(oracle.Q4_K, k)
    while time.perf_counter() - t0 < budget_s and rows <= n:
        xq = oracle.quantize_q8_1(x)
        oracle.mul_mat(oracle.Q4_K, w[:rows], k, xq, nthreads=cores)
        done_bytes += rows * rb + m * k * 2 + 2 * xq.nbytes + m * rows * 2
        rows = min(n, rows * 2) if rows < n else n + 1
    dt = time.perf_counter() - t0
    return {"value": round(done_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"Q4_K 4096x4096 x M=8 bf16 (q8_1 quantize + blockwise fp64 matmul), row subsets of "
                      f"64..4096 rows for ~{budget_s:.0f} s on {cores} threads"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    per = []
    for _ in range(args.warmup):
        cpu_baseline(budget_s=2.0)
    for _ in range(args.steps):
        per.append(cpu_baseline(budget_s=max(2.0, 30.0 / max(args.steps, 1))))
    v = statistics.median(p["value"] for p in per)
    cb = dict(per[-1])
    cb["value"] = v
    return {"impl": "reference", "metric": "GGUF matmul: weight-read HBM GB/s (MMVQ) and int8 TOPS (MMQ/MoE) on 1 GB300",
            "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode MMVQ: Q4_K 4096x4096 and 14336x4096, bf16 activations M in {1,2,4,8}; "
                                   "oracle on a bounded row sample per step"},
            "cpu_baseline": cb,
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


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
