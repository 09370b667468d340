#!/usr/bin/env python3
"""Benchmark of the UFP4 hot path on GB300.

One step = one pass of the hot path over one batch of the MoE-124B-like FPROP
workload (the largest single-GPU configuration): fused RHT + E1M2 4-bit
quantization (n = 16, 1 x 16 blocks, UE8M0 scales, RTNE) of X (16384 x 7168
bf16) and W (7168 x 7168 bf16), both N(0,1) with 0.1 % element outliers x50,
then the quantized GEMM Y = Q(X H') Q(W H')^T (16384 x 7168 x 7168, fp32 out).
The quantizer launch (ufp4_rht_quantize_prepare) also writes the GEMM's
operands (E5M2 copies of the levels and the hardware scales in the
tensor-memory copy layout), so the step is two launches: that one and the
tensor-core GEMM (ufp4_gemm_prepared).

value  = fused quantizer throughput in GB/s of algorithmic bytes (bf16 read
         + packed codes + scales + the E5M2 operand + its scale cells
         written), from CUDA events around the quantizer launch inside the
         timed steps.
gemm   = quantized GEMM TFLOP/s (2 M N K per step; the tensor-core kernel,
         its operands prepared by the quantizer launch).
e2e    = the same quantizer metric through the C ABI with host buffers:
         pinned H2D of X and W, quantize + prepare, GEMM and D2H of the
         codes, scales and Y inside the timed region.
Inputs rotate over 2 copies (each copy 322 MiB > 2 x L2), so every step reads
cold data.

--impl reference runs the oracle (plain C, one host core) as the reference
arm on bounded row samples of the same workload.
--suite prints further lines (the other workloads and modes), not the headline.
Multi-GPU (torchrun): every rank runs its own replica of the step (weak
scaling, no collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "fused RHT+4-bit quantize GB/s (% of HBM peak); quantized GEMM TFLOP/s (% peak)"
M, N, K = 16384, 7168, 7168
BLOCK = 16
# algorithmic bytes per element of the row-wise quantization alone: 2 (bf16
# in) + 0.5 (codes) + 1/16 (UE8M0 scale)
BYTES_PER_ELEM = 2.0 + 0.5 + 1.0 / BLOCK
# of the fused quantize + prepare launch: also 1 (E5M2 operand) + 4/32 (one
# hardware-scale cell per 32 elements, stored four times)
BYTES_PER_ELEM_PREP = BYTES_PER_ELEM + 1.0 + 4.0 / 32
QUANT_ELEMS = (M + N) * K
QUANT_BYTES = QUANT_ELEMS * BYTES_PER_ELEM_PREP
GEMM_FLOPS = 2.0 * M * N * K
ROTATE = 2
WORKLOAD = ("MoE-124B-like FPROP operands: X 16384x7168, W 7168x7168 bf16 (N(0,1), 0.1% element outliers x50); "
            "E1M2 1x16 UE8M0 RTNE, n=16; GEMM Y = Q(X)Q(W)^T 16384x7168x7168")
L2_NOTE = "inputs rotate over 2 copies (each 322 MiB > 2x L2); the 470 MB fp32 Y is written every step"


# library kernel launches per step: quantize and prepare X and W (one
# launch), tensor-core GEMM
LAUNCHES_PER_STEP = 2


def sources_hash(files) -> str:
    """sha256 (first 16 hex digits) of the named CUDA source files, read in the
    given order from rht_bit_block_gb300/csrc: ties a recorded ncu traffic
    figure to the sources of the kernel it was measured on."""
    import hashlib
    d = os.path.join(ROOT, "rht_bit_block_gb300", "csrc")
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu capture, or None when the
    kernel's sources changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            k = json.load(f).get("kernels", {}).get(kernel)
    except (OSError, ValueError):
        return None
    if not k or k.get("sources_sha256_16") != sources_hash(k.get("sources", [])):
        return None
    return k.get("dram_bytes_per_launch")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "src": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(seconds: float, units: float, world: int, backend_device=None):
    """Whole-job throughput: units summed over ranks / max time over ranks."""
    if world == 1:
        return seconds, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=backend_device)
    u = torch.tensor([units], dtype=torch.float64, device=backend_device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------ CPU baseline
def oracle_sample(rows_x: int, rows_w: int):
    """The first rows of X and W of the dense FPROP workload and the quantizer
    arguments, generated once, outside any timed region."""
    import oracle as orc
    from rht_bit_block_gb300 import inputs
    x, w = inputs.large_sweep(M, K, N)
    xs, ws = np.ascontiguousarray(x[:rows_x]), np.ascontiguousarray(w[:rows_w])
    del x, w
    kw = dict(grid="e1m2", block=(1, BLOCK), n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=orc.SCALE_UE8M0)
    orc.quantize(xs[:16], **kw)  # build + load outside the timing
    return xs, ws, kw


def cpu_oracle_rate(sample, min_seconds: float, max_reps: int):
    """Oracle (single-threaded C) on a bounded row sample of X and W; returns
    (GB/s, elements, seconds, reps).  The GB/s count the GPU arm's bytes per
    element (BYTES_PER_ELEM_PREP), so that both arms' values are elements per
    second times the same constant; the oracle itself computes the row-wise
    quantization only."""
    import oracle as orc
    xs, ws, kw = sample
    elems = 0
    t0 = time.perf_counter()
    reps = 0
    while reps < max_reps:
        orc.quantize(xs, **kw)
        orc.quantize(ws, **kw)
        elems += (xs.shape[0] + ws.shape[0]) * K
        reps += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    return elems * BYTES_PER_ELEM_PREP / dt / 1e9, elems, dt, reps


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    rows = 64
    sample = oracle_sample(rows, rows)
    for _ in range(args.warmup):
        cpu_oracle_rate(sample, 0.0, 1)
    t0 = time.perf_counter()
    elems = 0
    for _ in range(args.steps):
        _, e, _, _ = cpu_oracle_rate(sample, 0.0, 1)
        elems += e
    dt = time.perf_counter() - t0
    value = elems * BYTES_PER_ELEM_PREP / dt / 1e9
    sample_desc = (f"each step: the first {rows} rows of X and of W ({2 * rows * K} elements), oracle quantizer only; "
                   f"GB/s = elements x {BYTES_PER_ELEM_PREP} B, the GPU arm's bytes per element")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample_desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ GPU arm
def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from rht_bit_block_gb300 import inputs, ufp4
    ufp4.load()
    # a stream of its own: on non-default streams the library launches its
    # kernels as programmatic dependents of the previous kernel
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    x_np, w_np = inputs.large_sweep(M, K, N)
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    xs = [to_t(x_np).to(dev) for _ in range(ROTATE)]
    wsrc = [to_t(w_np).to(dev) for _ in range(ROTATE)]
    desc = ufp4.make_desc(grid="e1m2", block=(1, BLOCK), n=16, sign_seed=inputs.SIGN_SEED,
                          scale_fmt=ufp4.SCALE_UE8M0, out_mask=ufp4.OUT_ROWWISE)
    qx = ufp4.alloc_quantized(M, K, desc, dev)
    qw = ufp4.alloc_quantized(N, K, desc, dev)
    tx, tw = ufp4.qtensor(*qx, M, K), ufp4.qtensor(*qw, N, K)
    D = torch.empty((M, N), dtype=torch.float32, device=dev)
    wsb = torch.empty(ufp4.ufp4_gemm_workspace_size(M, N, K, desc), dtype=torch.uint8, device=dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)
    n_ev = args.steps
    e_q0, e_q1 = [ev() for _ in range(n_ev)], [ev() for _ in range(n_ev)]
    e_g1 = [ev() for _ in range(n_ev)]

    def step(i, timed):
        xi, wi = xs[i % ROTATE], wsrc[i % ROTATE]
        if timed:
            e_q0[i].record(stream)
        # X and W share the descriptor: one launch quantizes both and writes
        # the GEMM's prepared operands into the workspace
        ufp4.ufp4_rht_quantize_prepare(xi, wi, desc, tx, tw, wsb, stream.cuda_stream)
        if timed:
            e_q1[i].record(stream)
        ufp4.ufp4_gemm_prepared(tx, tw, desc, D, wsb, stream.cuda_stream)
        if timed:
            e_g1[i].record(stream)

    for i in range(args.warmup):
        step(i, False)
    barrier()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    barrier()
    t0 = time.perf_counter()
    start_all = ev()
    end_all = ev()
    start_all.record(stream)
    for i in range(args.steps):
        step(i, True)
    end_all.record(stream)
    barrier()
    wall = time.perf_counter() - t0
    clocks = sampler.stop()
    assert ufp4.ufp4_device_error() == 0, "a bounded device wait gave up"
    q_ms = [e_q0[i].elapsed_time(e_q1[i]) for i in range(args.steps)]
    g_ms = [e_q1[i].elapsed_time(e_g1[i]) for i in range(args.steps)]  # the tensor-core kernel
    k_ms = g_ms
    total_ms = start_all.elapsed_time(end_all)
    q_s = sum(q_ms) / 1e3
    g_s = sum(g_ms) / 1e3
    q_time, q_units = aggregate(q_s, QUANT_BYTES * args.steps, world, dev)
    g_time, g_units = aggregate(g_s, GEMM_FLOPS * args.steps, world, dev)
    k_time, _ = aggregate(sum(k_ms) / 1e3, 0.0, world, dev)
    step_time, _ = aggregate(total_ms / 1e3, 0.0, world, dev)
    value = q_units / q_time / 1e9
    gemm_tflops = g_units / g_time / 1e12
    kernel_tflops = g_units / k_time / 1e12

    # ------------------------------------------------------- e2e (host buffers)
    # Every step copies X and W in from pinned host memory, runs
    # ufp4_rht_quantize_prepare and ufp4_gemm_prepared, and copies the codes,
    # scales and Y out.  Steps are pipelined over three streams with two sets of device
    # and host buffers: the copy-in of step i + 1 and the copy-out of step i - 1
    # run while step i computes, so the two directions of the host link
    # overlap.  The timed region spans the first copy-in to the last copy-out.
    xh = to_t(x_np).pin_memory()
    whh = to_t(w_np).pin_memory()
    xin = [xs[0], xs[1 % ROTATE] if ROTATE > 1 else to_t(x_np).to(dev)]
    win = [wsrc[0], wsrc[1 % ROTATE] if ROTATE > 1 else to_t(w_np).to(dev)]
    qxs = [qx, ufp4.alloc_quantized(M, K, desc, dev)]
    qws = [qw, ufp4.alloc_quantized(N, K, desc, dev)]
    txs = [tx, ufp4.qtensor(*qxs[1], M, K)]
    tws = [tw, ufp4.qtensor(*qws[1], N, K)]
    Ds = [D, torch.empty((M, N), dtype=torch.float32, device=dev)]
    wss = [wsb, torch.empty_like(wsb)]
    codes_h = [[torch.empty_like(t, device="cpu").pin_memory() for t in (*qxs[k], *qws[k])] for k in range(2)]
    Dh = [torch.empty((M, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    e_in = [torch.cuda.Event() for _ in range(2)]    # copy-in of buffer set k done
    e_comp = [torch.cuda.Event() for _ in range(2)]  # compute on set k done (its inputs free)
    e_out = [torch.cuda.Event() for _ in range(2)]   # copy-out of set k done (its outputs free)
    # enough steps that the pipeline's fill (the first copy-in) and drain (the
    # last copy-out, about 3 ms) weigh little against the steady state
    e2e_steps = max(4, min(args.steps, 64))

    def e2e_pass(n_steps, t_start=None, t_end=None):
        for i in range(n_steps):
            k = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(e_comp[k])
                if i == 0 and t_start is not None:
                    t_start.record(s_in)
                xin[k].copy_(xh, non_blocking=True)
                win[k].copy_(whh, non_blocking=True)
                e_in[k].record(s_in)
            stream.wait_event(e_in[k])
            if i >= 2:
                stream.wait_event(e_out[k])
            ufp4.ufp4_rht_quantize_prepare(xin[k], win[k], desc, txs[k], tws[k], wss[k], stream.cuda_stream)
            ufp4.ufp4_gemm_prepared(txs[k], tws[k], desc, Ds[k], wss[k], stream.cuda_stream)
            e_comp[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_comp[k])
                for hbuf, dbuf in zip(codes_h[k], (*qxs[k], *qws[k])):
                    hbuf.copy_(dbuf, non_blocking=True)
                Dh[k].copy_(Ds[k], non_blocking=True)
                e_out[k].record(s_out)
        if t_end is not None:
            t_end.record(s_out)

    e2e_pass(2)
    barrier()
    a, b = ev(), ev()
    e2e_pass(e2e_steps, a, b)
    barrier()
    e2e_s, e2e_units = aggregate(a.elapsed_time(b) / 1e3, QUANT_BYTES * e2e_steps, world, dev)
    h2d = (xh.numel() + whh.numel()) * 2
    d2h = sum(t.numel() * t.element_size() for t in codes_h[0]) + Dh[0].numel() * 4

    pk = peaks()
    q_launch_ms = statistics.mean(q_ms)  # one batched quantizer launch per step (X and W)
    q_gbs = QUANT_BYTES / (q_launch_ms / 1e3) / 1e9
    fp8_peak = 2.0 * pk["bf16"]  # dense FP8 = 2 x bf16 (nominal ratio)
    gemm_frac = gemm_tflops / fp8_peak
    rl_q = {"bound": "hbm", "achieved": q_gbs, "peak": pk["hbm"], "unit": "GB/s", "frac": q_gbs / pk["hbm"],
            "traffic": recorded_traffic("quantize_rows_kernel<E1M2,RTNE,UE8M0,PREP>"),
            "kernel": "quantize_rows_kernel<E1M2,RTNE,UE8M0,PREP> (X and W in one launch, with their prepared "
                      "GEMM operands)", "bytes_per_elem": BYTES_PER_ELEM_PREP,
            "peak_src": pk["src"] + " hbm_gbs (burst)"}
    rl_g = {"bound": "tensor", "achieved": kernel_tflops, "peak": fp8_peak, "unit": "TFLOP/s",
            "frac": kernel_tflops / fp8_peak, "traffic": recorded_traffic("gemm_pair_kernel<FP8>"),
            "kernel": "gemm_pair_kernel<FP8> (CTA-pair tensor-core kernel)",
            "peak_src": pk["src"] + " bf16_tflops (burst) x2, the FP8/bf16 nominal ratio"}
    dominant = rl_g if statistics.mean(k_ms) >= statistics.mean(q_ms) else rl_q

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, elems, dt, reps = cpu_oracle_rate(oracle_sample(1024, 1024), args.cpu_seconds, 64)
        cpu = {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"first 1024 rows of X and of W ({2 * 1024 * K} elements) per rep, {reps} reps, {dt:.1f} s; "
                         f"row-wise quantization only, GB/s = elements x {BYTES_PER_ELEM_PREP} B as for value"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_time / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 (bf16 in, 4-bit codes out)", "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": L2_NOTE,
                       "parallelism": f"replicas x{world}"},
            "quant_frac_of_hbm": value / pk["hbm"],
            "gemm": {"value": gemm_tflops, "unit": "TFLOP/s", "frac": gemm_frac, "peak": fp8_peak,
                     "includes": "the tensor-core kernel; its FP8 operands are written by the quantizer launch "
                                 "(no separate prep pass)"},
            "roofline": dominant, "roofline_quantize": rl_q, "roofline_gemm": rl_g,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_units / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": LAUNCHES_PER_STEP * args.steps, "clocks": clocks, "wall_s_timed": wall,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------- suite mode
def run_suite(args, sections=("dense", "rowwise", "sweep", "rowcol", "diag", "gemm", "moe")):
    """Further measurements, one JSON line each (not the headline): the other
    workloads of the configuration list and the widened rows.  CUDA events on
    the launching stream, 3 warm-ups, median of the timed repetitions; inputs
    larger than L2 or rotated over 5 copies."""
    import torch
    from rht_bit_block_gb300 import inputs, ufp4
    ufp4.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    pk = peaks()
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)

    def timed(fn, reps=20, warm=3):
        for i in range(warm):
            fn(i)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i, (a, b) in enumerate(ev):
            a.record(stream)
            fn(i)
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    def emit(name, workload, value, unit, frac=None, peak=None, **extra):
        line = {"suite": name, "workload": workload, "value": value, "unit": unit}
        if frac is not None:
            line.update({"frac": frac, "peak": peak})
        line.update(extra)
        print(json.dumps(line), flush=True)

    def want(name):  # --suite-match: the sweep cells and GEMM lines to run
        return not args.suite_match or re.search(args.suite_match, name) is not None

    def scale_bytes(desc):
        per = 1 if desc.scale_fmt == ufp4.SCALE_UE8M0 else 4
        return per / (desc.block_rows * desc.block_cols)

    if "dense" in sections:
        # the Dense-1.5B-like FPROP step: X 8192 x 2048 and W 5632 x 2048 quantized
        # in one launch, then the GEMM 8192 x 5632 x 2048 (prep and kernel timed apart)
        xd_np, wd_np = inputs.dense_fprop()
        (m2, k2), n2 = xd_np.shape, wd_np.shape[0]
        xs2 = [to_t(xd_np).to(dev) for _ in range(5)]
        ws2 = [to_t(wd_np).to(dev) for _ in range(5)]
        desc = ufp4.make_desc(grid="e1m2", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED,
                              scale_fmt=ufp4.SCALE_UE8M0, out_mask=ufp4.OUT_ROWWISE)
        qx2, qw2 = ufp4.alloc_quantized(m2, k2, desc, dev), ufp4.alloc_quantized(n2, k2, desc, dev)
        tx2, tw2 = ufp4.qtensor(*qx2, m2, k2), ufp4.qtensor(*qw2, n2, k2)
        D2 = torch.empty((m2, n2), dtype=torch.float32, device=dev)
        wsb2 = torch.empty(ufp4.ufp4_gemm_workspace_size(m2, n2, k2, desc), dtype=torch.uint8, device=dev)
        qms = timed(lambda i: ufp4.ufp4_rht_quantize_batch([xs2[i % 5], ws2[i % 5]], desc, [tx2, tw2],
                                                           stream.cuda_stream))
        pms = timed(lambda i: ufp4.ufp4_gemm_prepare(tx2, tw2, desc, wsb2, stream.cuda_stream))
        kms = timed(lambda i: ufp4.ufp4_gemm_prepared(tx2, tw2, desc, D2, wsb2, stream.cuda_stream))
        qb = (m2 + n2) * k2 * BYTES_PER_ELEM
        emit("dense_step", f"Dense-1.5B-like FPROP operands X {m2}x{k2} + W {n2}x{k2}, e1m2 1x16 UE8M0 n=16 RTNE, "
             "one batched launch", qb / (qms / 1e3) / 1e9, "GB/s", qb / (qms / 1e3) / 1e9 / pk["hbm"], pk["hbm"],
             ms=qms)
        fms = timed(lambda i: ufp4.ufp4_rht_quantize_prepare(xs2[i % 5], ws2[i % 5], desc, tx2, tw2, wsb2,
                                                             stream.cuda_stream))
        fb = (m2 + n2) * k2 * BYTES_PER_ELEM_PREP
        emit("dense_step", f"Dense-1.5B-like FPROP operands, quantized and prepared for the GEMM in one launch "
             "(ufp4_rht_quantize_prepare; replaces the batched launch + the prep pass)", fb / (fms / 1e3) / 1e9, "GB/s",
             fb / (fms / 1e3) / 1e9 / pk["hbm"], pk["hbm"], ms=fms, unfused_ms=qms + pms)
        tf = 2.0 * m2 * n2 * k2 / (kms / 1e3) / 1e12
        emit("dense_step", f"Dense-1.5B-like FPROP GEMM {m2}x{n2}x{k2} e1m2 1x16 UE8M0 (tensor-core kernel; "
             "prep timed apart)", tf, "TFLOP/s", tf / (2 * pk["bf16"]), 2 * pk["bf16"], kernel_ms=kms, prep_ms=pms)
        del xs2, ws2, D2, wsb2

    if "rowwise" in sections:
        # 1. large-shape sweep operand, row-wise (X 16384 x 7168, > L2)
        x5, _ = inputs.large_sweep(k=7168, n=128)
        xs5 = [to_t(x5).to(dev) for _ in range(2)]
        rows, cols = x5.shape
        cases = [("e1m2", (1, 16), 16, ufp4.SCALE_UE8M0, ufp4.ROUND_RTNE), ("int4", (1, 16), 16, ufp4.SCALE_UE8M0, 0),
                 ("e2m1", (1, 16), 16, ufp4.SCALE_UE8M0, 0), ("e2m1r2", (1, 16), 16, ufp4.SCALE_UE8M0, 0),
                 ("e1m2", (1, 16), 16, ufp4.SCALE_FP32, 0), ("e1m2", (1, 32), 64, ufp4.SCALE_UE8M0, 0),
                 ("e1m2", (1, 16), 256, ufp4.SCALE_UE8M0, 0), ("e2m1", (32, 32), 16, ufp4.SCALE_UE8M0, 0),
                 ("e1m2", (1, 16), 16, ufp4.SCALE_UE8M0, ufp4.ROUND_SR),
                 ("mxfp8", (1, 32), 1, ufp4.SCALE_UE8M0, 0), ("mxfp8", (1, 32), 16, ufp4.SCALE_UE8M0, 0)]
        for grid, block, n, fmt, rnd in cases:
            desc = ufp4.make_desc(grid=grid, block=block, n=n, sign_seed=inputs.SIGN_SEED, scale_fmt=fmt, rounding=rnd,
                                  sr_seed=inputs.SR_SEED, out_mask=ufp4.OUT_ROWWISE)
            out = ufp4.alloc_quantized(rows, cols, desc, dev)
            q = ufp4.qtensor(*out, rows, cols)
            ms = timed(lambda i: ufp4.ufp4_rht_quantize(xs5[i % 2], desc, q, None, stream.cuda_stream))
            code_bytes = 1.0 if grid == "mxfp8" else 0.5
            gbs = rows * cols * (2 + code_bytes + scale_bytes(desc)) / (ms / 1e3) / 1e9
            emit("quantize_rowwise", f"X {rows}x{cols} {grid} {block[0]}x{block[1]} "
                 f"{('E8M0' if grid == 'mxfp8' else 'UE8M0') if fmt else 'fp32'} n={n} {'SR' if rnd else 'RTNE'}", gbs,
                 "GB/s", gbs / pk["hbm"], pk["hbm"],
                 ms=ms)
        # two-level scale: the tensor amax pre-pass reads x once more before the quantizer reads it
        desc = ufp4.make_desc(grid="e2m1", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED,
                              scale_fmt=ufp4.SCALE_E4M3, out_mask=ufp4.OUT_ROWWISE)
        out = ufp4.alloc_quantized(rows, cols, desc, dev)
        t_amax = torch.zeros(1, dtype=torch.float32, device=dev)
        q = ufp4.qtensor(*out, rows, cols, t_amax)
        ms = timed(lambda i: ufp4.ufp4_rht_quantize(xs5[i % 2], desc, q, None, stream.cuda_stream))
        gbs = rows * cols * (2 * 2 + 0.5 + 1 / 16) / (ms / 1e3) / 1e9
        emit("quantize_rowwise", f"X {rows}x{cols} e2m1 1x16 two-level (E4M3 x fp32) n=16 RTNE: tensor amax "
             "pre-pass + quantize, x read twice", gbs, "GB/s", gbs / pk["hbm"], pk["hbm"], ms=ms)
        del xs5

    if "sweep" in sections:
        # the large-shape quantizer sweep on X 16384 x 7168, row-wise: n in {16, 64,
        # 256} x grid {E1M2, INT4, E2M1} x block {1x16 fp32, 1x32 fp32, 32x32 UE8M0}
        # x {RTNE, SR}, 54 cells
        x5, _ = inputs.large_sweep(k=7168, n=128)
        xs5 = [to_t(x5).to(dev) for _ in range(2)]
        rows, cols = x5.shape
        for n in (16, 64, 256):
            for grid in ("e1m2", "int4", "e2m1"):
                for block, fmt in (((1, 16), ufp4.SCALE_FP32), ((1, 32), ufp4.SCALE_FP32),
                                   ((32, 32), ufp4.SCALE_UE8M0)):
                    for rnd in (ufp4.ROUND_RTNE, ufp4.ROUND_SR):
                        name = (f"X {rows}x{cols} {grid} {block[0]}x{block[1]} "
                                f"{'UE8M0' if fmt else 'fp32'} n={n} {'SR' if rnd else 'RTNE'}")
                        if not want(name):
                            continue
                        desc = ufp4.make_desc(grid=grid, block=block, n=n, sign_seed=inputs.SIGN_SEED, scale_fmt=fmt,
                                              rounding=rnd, sr_seed=inputs.SR_SEED, out_mask=ufp4.OUT_ROWWISE)
                        out = ufp4.alloc_quantized(rows, cols, desc, dev)
                        q = ufp4.qtensor(*out, rows, cols)
                        ms = timed(lambda i: ufp4.ufp4_rht_quantize(xs5[i % 2], desc, q, None, stream.cuda_stream))
                        gbs = rows * cols * (2 + 0.5 + scale_bytes(desc)) / (ms / 1e3) / 1e9
                        emit("quantize_sweep", name, gbs, "GB/s", gbs / pk["hbm"], pk["hbm"], ms=ms)
                        del out, q
        del xs5

    if "rowcol" in sections:
        # 2. dY stochastic-rounding path: row-wise and column-wise from one read
        dy, _ = inputs.dy_sr()
        dys = [to_t(dy).to(dev) for _ in range(5)]
        r3, c3 = dy.shape
        # then the same shape rounded to nearest (the X and W operands' row + column pass)
        for rnd, fmt in ((ufp4.ROUND_SR, ufp4.SCALE_FP32), (ufp4.ROUND_SR, ufp4.SCALE_UE8M0),
                         (ufp4.ROUND_RTNE, ufp4.SCALE_FP32), (ufp4.ROUND_RTNE, ufp4.SCALE_UE8M0)):
            desc = ufp4.make_desc(grid="e1m2", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=fmt,
                                  rounding=rnd, sr_seed=inputs.SR_SEED,
                                  out_mask=ufp4.OUT_ROWWISE | ufp4.OUT_COLWISE)
            ro = ufp4.alloc_quantized(r3, c3, desc, dev)
            co = ufp4.alloc_quantized(c3, r3, desc, dev)
            rq, cq = ufp4.qtensor(*ro, r3, c3), ufp4.qtensor(*co, c3, r3)
            ms = timed(lambda i: ufp4.ufp4_rht_quantize(dys[i % 5], desc, rq, cq, stream.cuda_stream))
            gbs = r3 * c3 * (2 + 2 * (0.5 + scale_bytes(desc))) / (ms / 1e3) / 1e9
            tag = "SR" if rnd == ufp4.ROUND_SR else "RTNE"
            emit("quantize_rowcol", f"dY {r3}x{c3} e1m2 1x16 {'UE8M0' if fmt else 'fp32'} n=16 {tag} row+col", gbs,
                 "GB/s", gbs / pk["hbm"], pk["hbm"], ms=ms)
        # 2-D 32 x 32 blocks, row-wise and column-wise from one read, on the large operand
        xl, _ = inputs.large_sweep(k=7168, n=128)
        xls = [to_t(xl).to(dev)]
        rl, cl = xl.shape
        for n2 in (1, 16):
            desc = ufp4.make_desc(grid="e1m2", block=(32, 32), n=n2, sign_seed=inputs.SIGN_SEED,
                                  scale_fmt=ufp4.SCALE_UE8M0, out_mask=ufp4.OUT_ROWWISE | ufp4.OUT_COLWISE)
            ro = ufp4.alloc_quantized(rl, cl, desc, dev)
            co = ufp4.alloc_quantized(cl, rl, desc, dev)
            rq, cq = ufp4.qtensor(*ro, rl, cl), ufp4.qtensor(*co, cl, rl)
            ms = timed(lambda i: ufp4.ufp4_rht_quantize(xls[0], desc, rq, cq, stream.cuda_stream))
            gbs = rl * cl * (2 + 2 * (0.5 + scale_bytes(desc))) / (ms / 1e3) / 1e9
            emit("quantize_rowcol", f"X {rl}x{cl} e1m2 32x32 UE8M0 n={n2} RTNE row+col", gbs, "GB/s",
                 gbs / pk["hbm"], pk["hbm"], ms=ms)

    if "diag" in sections:
        # 3. diagnostics on the dense FPROP X
        x2, _ = inputs.dense_fprop(n=128)
        x2s = [to_t(x2).to(dev) for _ in range(5)]
        r2, c2 = x2.shape
        desc = ufp4.make_desc(grid="e1m2", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED,
                              scale_fmt=ufp4.SCALE_UE8M0, out_mask=ufp4.OUT_ROWWISE)
        qout = [ufp4.alloc_quantized(r2, c2, desc, dev) for _ in range(5)]
        for i in range(5):
            ufp4.ufp4_rht_quantize(x2s[i], desc, ufp4.qtensor(*qout[i], r2, c2), None, stream.cuda_stream)
        st = torch.zeros(4, dtype=torch.float64, device=dev)
        ms = timed(lambda i: ufp4.ufp4_quant_error_stats(x2s[i % 5], desc, ufp4.qtensor(*qout[i % 5], r2, c2), st,
                                                         stream.cuda_stream))
        gbs = r2 * c2 * (2 + 0.5 + 1 / 16) / (ms / 1e3) / 1e9
        s = st.cpu().numpy()
        emit("diagnostics", f"quant_error_stats X {r2}x{c2} e1m2 1x16 UE8M0 n=16", gbs, "GB/s", gbs / pk["hbm"],
             pk["hbm"], ms=ms, sqnr_db=float(10 * np.log10(s[0] / s[1])), shrinkage=float(s[2] / s[0]))
        del x2s, qout

    if "gemm" in sections:
        # 4. GEMMs per grid on the dense FPROP shape (tensor-core kernel alone, prep timed apart)
        M, N, K = 8192, 5632, 2048
        g = torch.Generator().manual_seed(7)
        for grid, block, kind_peak in (("e1m2", (1, 16), 2.0), ("int4", (1, 32), 2.0), ("e2m1", (1, 16), 6.0),
                                       ("e2m1", (1, 32), 6.0), ("e2m1r2", (1, 16), 6.0)):
            if not want(f"{M}x{N}x{K} {grid} {block[0]}x{block[1]} UE8M0"):
                continue
            desc = ufp4.make_desc(grid=grid, block=block, scale_fmt=ufp4.SCALE_UE8M0)
            def operand(rows):
                c = torch.randint(0, 256, (rows, K // 2), generator=g, dtype=torch.uint8)
                c = c & 0x77 if grid != "int4" else c & 0x77  # valid codes in every grid, no -0 / -8
                sc = torch.randint(120, 132, (rows, K // block[1]), generator=g, dtype=torch.uint8)
                return c.to(dev), sc.to(dev)
            A, B = operand(M), operand(N)
            qa, qb = ufp4.qtensor(*A, M, K), ufp4.qtensor(*B, N, K)
            ws = torch.empty(ufp4.ufp4_gemm_workspace_size(M, N, K, desc), dtype=torch.uint8, device=dev)
            D = torch.empty((M, N), dtype=torch.float32, device=dev)
            pms = timed(lambda i: ufp4.ufp4_gemm_prepare(qa, qb, desc, ws, stream.cuda_stream))
            kms = timed(lambda i: ufp4.ufp4_gemm_prepared(qa, qb, desc, D, ws, stream.cuda_stream))
            tf = 2.0 * M * N * K / (kms / 1e3) / 1e12
            peak = kind_peak * pk["bf16"]
            emit("gemm", f"{M}x{N}x{K} {grid} {block[0]}x{block[1]} UE8M0", tf, "TFLOP/s", tf / peak, peak,
                 kernel_ms=kms, prep_ms=pms, peak_src=f"measured bf16 burst x{kind_peak:g} (nominal ratio)")
            del A, B, ws, D
        # two-level scales: UE4M3 block bytes on the native FP4 kind, g_A g_B in the epilogue
        if want(f"{M}x{N}x{K} e2m1 1x16 two-level (UE4M3 x fp32)"):
            desc = ufp4.make_desc(grid="e2m1", block=(1, 16), scale_fmt=ufp4.SCALE_E4M3)
            def two_level_operand(rows):
                c = torch.randint(0, 256, (rows, K // 2), generator=g, dtype=torch.uint8) & 0x77
                sc = torch.randint(0x30, 0x48, (rows, K // 16), generator=g, dtype=torch.uint8)  # E4M3 0.5 .. 4
                return c.to(dev), sc.to(dev), torch.full((1,), 100.0, dtype=torch.float32, device=dev)
            A, B = two_level_operand(M), two_level_operand(N)
            qa, qb = ufp4.qtensor(A[0], A[1], M, K, A[2]), ufp4.qtensor(B[0], B[1], N, K, B[2])
            ws = torch.empty(ufp4.ufp4_gemm_workspace_size(M, N, K, desc), dtype=torch.uint8, device=dev)
            D = torch.empty((M, N), dtype=torch.float32, device=dev)
            pms = timed(lambda i: ufp4.ufp4_gemm_prepare(qa, qb, desc, ws, stream.cuda_stream))
            kms = timed(lambda i: ufp4.ufp4_gemm_prepared(qa, qb, desc, D, ws, stream.cuda_stream))
            tf = 2.0 * M * N * K / (kms / 1e3) / 1e12
            emit("gemm", f"{M}x{N}x{K} e2m1 1x16 two-level (UE4M3 x fp32)", tf, "TFLOP/s", tf / (6 * pk["bf16"]),
                 6 * pk["bf16"], kernel_ms=kms, prep_ms=pms, peak_src="measured bf16 burst x6 (nominal ratio)")
            del A, B, ws, D
        # MXFP8 operands (E4M3 codes read in place by the FP8 kernel)
        if want(f"{M}x{N}x{K} mxfp8 1x32 E8M0"):
            desc = ufp4.make_desc(grid="mxfp8", block=(1, 32), scale_fmt=ufp4.SCALE_UE8M0)
            def e4m3_operand(rows):
                c = torch.randint(0, 0x7F, (rows, K), generator=g, dtype=torch.uint8)  # finite magnitudes
                c = c | (torch.randint(0, 2, (rows, K), generator=g, dtype=torch.uint8) << 7)
                sc = torch.randint(120, 132, (rows, K // 32), generator=g, dtype=torch.uint8)
                return c.to(dev), sc.to(dev)
            A, B = e4m3_operand(M), e4m3_operand(N)
            qa, qb = ufp4.qtensor(*A, M, K), ufp4.qtensor(*B, N, K)
            ws = torch.empty(ufp4.ufp4_gemm_workspace_size(M, N, K, desc), dtype=torch.uint8, device=dev)
            D = torch.empty((M, N), dtype=torch.float32, device=dev)
            pms = timed(lambda i: ufp4.ufp4_gemm_prepare(qa, qb, desc, ws, stream.cuda_stream))
            kms = timed(lambda i: ufp4.ufp4_gemm_prepared(qa, qb, desc, D, ws, stream.cuda_stream))
            tf = 2.0 * M * N * K / (kms / 1e3) / 1e12
            emit("gemm", f"{M}x{N}x{K} mxfp8 1x32 E8M0", tf, "TFLOP/s", tf / (2 * pk["bf16"]), 2 * pk["bf16"],
                 kernel_ms=kms, prep_ms=pms, peak_src="measured bf16 burst x2 (nominal ratio)")
            del A, B, ws, D
        # fp32 block scales (the two-scale path: bf16 partials rescaled on the CUDA cores)
        if want(f"{M}x{N}x{K} e1m2 1x16 fp32 scales (two-scale path)"):
            desc = ufp4.make_desc(grid="e1m2", block=(1, 16), scale_fmt=ufp4.SCALE_FP32)
            A = (torch.randint(0, 256, (M, K // 2), generator=g, dtype=torch.uint8).__and__(0x77).to(dev),
                 torch.rand((M, K // 16), generator=g).add(0.5).to(dev))
            B = (torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.uint8).__and__(0x77).to(dev),
                 torch.rand((N, K // 16), generator=g).add(0.5).to(dev))
            qa, qb = ufp4.qtensor(*A, M, K), ufp4.qtensor(*B, N, K)
            ws = torch.empty(ufp4.ufp4_gemm_workspace_size(M, N, K, desc), dtype=torch.uint8, device=dev)
            D = torch.empty((M, N), dtype=torch.float32, device=dev)
            pms = timed(lambda i: ufp4.ufp4_gemm_prepare(qa, qb, desc, ws, stream.cuda_stream))
            kms = timed(lambda i: ufp4.ufp4_gemm_prepared(qa, qb, desc, D, ws, stream.cuda_stream))
            tf = 2.0 * M * N * K / (kms / 1e3) / 1e12
            emit("gemm", f"{M}x{N}x{K} e1m2 1x16 fp32 scales (two-scale path)", tf, "TFLOP/s", tf / (2 * pk["bf16"]),
                 2 * pk["bf16"], kernel_ms=kms, prep_ms=pms, peak_src="measured bf16 burst x2 (FP8 peak, for comparison)")
            del A, B, ws, D
        # the large-sweep FPROP GEMMs: 16384 x 7168 x 7168 per grid, 1x16 and 32x32 UE8M0 operands
        M5, N5, K5 = 16384, 7168, 7168
        for grid, block, kind_peak in (("e1m2", (1, 16), 2.0), ("int4", (1, 16), 2.0), ("e2m1", (1, 16), 6.0),
                                       ("e1m2", (32, 32), 2.0), ("int4", (32, 32), 2.0), ("e2m1", (32, 32), 6.0)):
            if not want(f"{M5}x{N5}x{K5} {grid} {block[0]}x{block[1]} UE8M0"):
                continue
            desc = ufp4.make_desc(grid=grid, block=block, scale_fmt=ufp4.SCALE_UE8M0)
            def operand(rows):
                c = torch.randint(0, 256, (rows, K5 // 2), generator=g, dtype=torch.uint8).__and__(0x77).to(dev)
                srows = rows // block[0] if block[0] > 1 else rows
                sc = torch.randint(120, 132, (srows, K5 // block[1]), generator=g, dtype=torch.uint8).to(dev)
                return c, sc
            A, B = operand(M5), operand(N5)
            qa, qb = ufp4.qtensor(*A, M5, K5), ufp4.qtensor(*B, N5, K5)
            ws = torch.empty(ufp4.ufp4_gemm_workspace_size(M5, N5, K5, desc), dtype=torch.uint8, device=dev)
            D = torch.empty((M5, N5), dtype=torch.float32, device=dev)
            pms = timed(lambda i: ufp4.ufp4_gemm_prepare(qa, qb, desc, ws, stream.cuda_stream), reps=10)
            kms = timed(lambda i: ufp4.ufp4_gemm_prepared(qa, qb, desc, D, ws, stream.cuda_stream), reps=10)
            tf = 2.0 * M5 * N5 * K5 / (kms / 1e3) / 1e12
            peak = kind_peak * pk["bf16"]
            emit("gemm", f"{M5}x{N5}x{K5} {grid} {block[0]}x{block[1]} UE8M0", tf, "TFLOP/s", tf / peak, peak,
                 kernel_ms=kms, prep_ms=pms, peak_src=f"measured bf16 burst x{kind_peak:g} (nominal ratio)")
            del A, B, ws, D

    if "moe" in sections:
        # 5. MoE-7.9B-like expert FFN step: seeded top-2 routing of 16384 tokens
        # over 8 experts (hidden 2048, ffn 1408); grouped row+col quantization of
        # X (RTNE) and dY (SR), per-expert W_e row+col (RTNE), then the grouped
        # FPROP, DGRAD and WGRAD GEMMs (prep included)
        lists, x_all, w_all, dy_np = inputs.moe_step()
        experts, hidden, ffn = w_all.shape[0], w_all.shape[2], w_all.shape[1]
        counts = [len(l) for l in lists]
        off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
        total = int(off[-1])
        xs = to_t(np.ascontiguousarray(np.concatenate([x_all[l] for l in lists]))).to(dev)
        dys = to_t(dy_np).to(dev)
        w_stack = to_t(np.ascontiguousarray(w_all.reshape(experts * ffn, hidden))).to(dev)
        w_off = [e * ffn for e in range(experts + 1)]
        kw = dict(grid="e1m2", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=ufp4.SCALE_UE8M0, out_mask=3)
        x_desc = ufp4.make_desc(**kw)
        dy_desc = ufp4.make_desc(rounding=ufp4.ROUND_SR, sr_seed=inputs.SR_SEED, **kw)
        gdesc = ufp4.make_desc(grid="e1m2", block=(1, 16), scale_fmt=ufp4.SCALE_UE8M0)
        pads = [ufp4.ufp4_grouped_padded_rows(c, x_desc) for c in counts]
        poff = np.concatenate([[0], np.cumsum(pads)]).astype(np.int64)
        ptot = int(poff[-1])

        def grouped_bufs(cols):
            rc = torch.empty((total, cols // 2), dtype=torch.uint8, device=dev)
            rs = torch.empty((total, cols // 16), dtype=torch.uint8, device=dev)
            cc = torch.empty((cols * ptot // 2,), dtype=torch.uint8, device=dev)
            cs = torch.empty((cols * ptot // 16,), dtype=torch.uint8, device=dev)
            row_q = ufp4.qtensor(rc, rs, total, cols)
            col_q = ufp4.QTensor(cc.data_ptr(), cs.data_ptr(), cols, ptot, 0, 0)
            rows = [ufp4.qtensor(rc[off[g]:off[g + 1]], rs[off[g]:off[g + 1]], counts[g], cols) for g in range(experts)]
            colsq = [ufp4.qtensor(cc[cols * poff[g] // 2: cols * poff[g + 1] // 2].view(cols, pads[g] // 2),
                                  cs[cols * poff[g] // 16: cols * poff[g + 1] // 16].view(cols, pads[g] // 16),
                                  cols, pads[g]) for g in range(experts)]
            return (rc, rs, cc, cs), row_q, col_q, rows, colsq
        xb, xrq, xcq, xrow, xcol = grouped_bufs(hidden)
        yb, yrq, ycq, yrow, ycol = grouped_bufs(ffn)
        # W_e: one grouped call over the stacked experts (ffn is a multiple of the
        # grouped padding unit, so each expert's column-wise slab is its own W_e^T)
        assert ufp4.ufp4_grouped_padded_rows(ffn, x_desc) == ffn
        wrc = torch.empty((experts * ffn, hidden // 2), dtype=torch.uint8, device=dev)
        wrs = torch.empty((experts * ffn, hidden // 16), dtype=torch.uint8, device=dev)
        wcc = torch.empty((experts, hidden, ffn // 2), dtype=torch.uint8, device=dev)
        wcs = torch.empty((experts, hidden, ffn // 16), dtype=torch.uint8, device=dev)
        w_rq = ufp4.qtensor(wrc, wrs, experts * ffn, hidden)
        w_cq = ufp4.QTensor(wcc.data_ptr(), wcs.data_ptr(), hidden, experts * ffn, 0, 0)
        wrow = [ufp4.qtensor(wrc[e * ffn:(e + 1) * ffn], wrs[e * ffn:(e + 1) * ffn], ffn, hidden) for e in range(experts)]
        wcol = [ufp4.qtensor(wcc[e], wcs[e], hidden, ffn) for e in range(experts)]
        gemms = {"FPROP": (xrow, wrow, [(c, ffn) for c in counts]),
                 "DGRAD": (yrow, wcol, [(c, hidden) for c in counts]),
                 "WGRAD": (ycol, xcol, [(ffn, hidden)] * experts)}
        outs = {k: [torch.empty((m, n), dtype=torch.float32, device=dev) for m, n in v[2]] for k, v in gemms.items()}
        wsz = max(ufp4.ufp4_gemm_grouped_workspace_size(a, b, gdesc) for a, b, _ in gemms.values())
        gws = torch.empty(max(1, wsz), dtype=torch.uint8, device=dev)

        def quantize_all(i):
            ufp4.ufp4_rht_quantize_grouped(xs, off.tolist(), x_desc, xrq, xcq, stream.cuda_stream)
            ufp4.ufp4_rht_quantize_grouped(dys, off.tolist(), dy_desc, yrq, ycq, stream.cuda_stream)
            ufp4.ufp4_rht_quantize_grouped(w_stack, w_off, x_desc, w_rq, w_cq, stream.cuda_stream)

        def gemm_all(i):
            for k, (a, b, _) in gemms.items():
                ufp4.ufp4_gemm_grouped(a, b, gdesc, outs[k], gws, stream.cuda_stream)

        qms = timed(quantize_all, reps=10)
        gms = timed(gemm_all, reps=10)
        flops = 3 * 2.0 * total * ffn * hidden
        qbytes = (total * hidden + total * ffn + experts * ffn * hidden) * (2 + 2 * (0.5 + 1 / 16))
        emit("moe_step", f"MoE-7.9B-like step, {total} routed rows, 8 experts, hidden {hidden}, ffn {ffn}: "
             "grouped row+col quantize of X (RTNE), dY (SR) and W_e (RTNE)", qbytes / (qms / 1e3) / 1e9, "GB/s",
             qbytes / (qms / 1e3) / 1e9 / pk["hbm"], pk["hbm"], ms=qms)
        emit("moe_step", f"MoE-7.9B-like step: grouped FPROP + DGRAD + WGRAD GEMMs, e1m2 1x16 UE8M0, prep included",
             flops / (gms / 1e3) / 1e12, "TFLOP/s", flops / (gms / 1e3) / 1e12 / (2 * pk["bf16"]), 2 * pk["bf16"],
             ms=gms, step_ms=qms + gms)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--suite", action="store_true",
                    help="further measurements (other workloads, widened rows), one JSON line each")
    ap.add_argument("--suite-sections", default="dense,rowwise,sweep,rowcol,diag,gemm,moe",
                    help="comma-separated subset of the suite: dense, rowwise, sweep, rowcol, diag, gemm, moe")
    ap.add_argument("--suite-match", default=None,
                    help="sweep and gemm sections: run only the cells and lines whose workload name matches "
                         "this regular expression")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.suite:
        run_suite(args, tuple(args.suite_sections.split(",")))
        return
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
