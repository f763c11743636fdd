"""Benchmark of the quantized MoE gather matmul (gqmm_gather_qmm) on GB300.

Default workload: the MoE prefill microbenchmark shape of the mlx issue "[CUDA] gather_qmm
~24x slower than equal-FLOPs quantized_matmul on GB10" (section "Kernel microbenchmark"):
T=2048 tokens, A=8 active experts, H=2048, F=768, E=64, affine 4-bit weights with 64-wide
groups, x ~ N(0, 1) bf16, idx uniform (unsorted).  One step = one gqmm_gather_qmm call
(on-device route sort + work-list plan + grouped tcgen05 GEMM + scatter epilogue) on inputs
already resident in HBM.  Metric: effective TFLOP/s = 2*T*A*H*F / step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent replica of the
workload on its own GPU (the op has no cross-GPU exchange); value = total FLOPs of all ranks /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

# gate activation of the expert-MLP workloads (the activation's cost is a few microseconds of
# elementwise work next to the projections; every activation is parity-tested)
MLP_ACTIVATION = "silu"
# GEMM launches (projections) per step, each timed by the library's kernel timer
GEMM_LAUNCHES_PER_STEP = {"gather": 1, "mlp": 2, "nn": 1}

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_bytes(w: wl.Workload, idx: np.ndarray | None) -> int:
    """Packed codes + scales/biases of the experts actually hit, x, y and idx, each once.  For
    the expert MLP: both projections' weights, x and y (the gate/up output and the gated
    hidden rows are intermediates, not counted: a kernel that kept them on chip moves none)."""
    hit = w.E if idx is None else len(np.unique(idx))

    def qbytes(rows, K):  # one expert's packed codes + bf16 scale and bias per group
        return rows * (K // 2 + 4 * (K // w.group_size))

    if w.kind == "mlp":
        weights = hit * (qbytes(2 * w.F, w.H) + qbytes(w.H, w.F))
    elif w.kind == "nn":  # W[e] is [K = H, N = F], quantized along F
        weights = hit * qbytes(w.H, w.F)
    else:
        weights = hit * qbytes(w.F, w.H)
    return int(weights + w.n * w.H * 2 + w.n * w.out_cols * 2 + (0 if idx is None else w.n * 4))


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"gqmm_clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------------------------
# CPU oracle legs (the only places this script runs the oracle)
# ----------------------------------------------------------------------------------------------

def oracle_inputs(w: wl.Workload, inp):
    """The oracle's quantized weights for the workload: (wq, scales, biases), or for the
    expert MLP ((gate/up), (down))."""
    import oracle

    if w.kind == "mlp":
        return (oracle.quantize(inp["w_gu"], group_size=w.group_size),
                oracle.quantize(inp["w_dn"], group_size=w.group_size))
    return oracle.quantize(inp["w"], group_size=w.group_size)


def oracle_rows(w: wl.Workload, x_cpu, qw, idx, rows):
    """The oracle on the listed flat rows; returns its thread count."""
    import oracle

    if w.kind == "mlp":
        oracle.moe_mlp(x_cpu, qw[0], qw[1], idx, w.E, group_size=w.group_size, rows=rows)
    elif w.kind == "nn":
        oracle.gather_qmm_nn(x_cpu, *qw, idx, w.E, group_size=w.group_size, rows=rows)
        return 1  # numpy row products, one thread
    else:
        oracle.gather_qmm(x_cpu, *qw, idx, w.E, group_size=w.group_size, rows=rows)
    return oracle.gather_qmm.last_threads


def oracle_rate(w: wl.Workload, x_cpu, qw, idx, target_s: float, max_rows: int | None = None):
    """Times the oracle on a bounded sample of rows; returns (TFLOP/s, rows, seconds, threads)."""
    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(w.n, size=min(w.n, 32), replace=False))
    t0 = time.perf_counter()
    oracle_rows(w, x_cpu, qw, idx, probe)
    dt = time.perf_counter() - t0
    rows = int(max(1, min(w.n, len(probe) * target_s / max(dt, 1e-6))))
    if max_rows:
        rows = min(rows, max_rows)
    sample = np.sort(rng.choice(w.n, size=rows, replace=False))
    t0 = time.perf_counter()
    threads = oracle_rows(w, x_cpu, qw, idx, sample)
    dt = time.perf_counter() - t0
    flops = w.flops / w.n * rows
    return flops / dt / 1e12, rows, dt, threads


def metric_name(w: wl.Workload) -> str:
    if w.kind == "mlp":
        return "moe_mlp TFLOPs (6*T*A*H*I/time)"
    if w.kind == "nn":
        return "gather_qmm_nn TFLOPs (2*T*A*K*N/time)"
    return "gather_qmm TFLOPs (2*T*A*H*F/time)"


def workload_config(w: wl.Workload) -> dict:
    c = {"workload": w.name, "T": w.T, "A": w.A, "H": w.H}
    c.update({"I": w.F} if w.kind == "mlp" else {"K": w.H, "N": w.F} if w.kind == "nn" else {"F": w.F})
    c.update({"E": w.E, "group_size": w.group_size, "bits": 4, "routing": w.routing})
    if w.kind == "mlp":
        c["op"] = "gqmm_moe_mlp: gate/up projection, act(gate) * up, down projection"
        c["activation"] = MLP_ACTIVATION
    return c


def run_reference(args, w: wl.Workload, world: int, rank: int):
    """The oracle, as it stands, on the host cores: each step computes a bounded sample of rows."""
    if rank != 0:
        return
    inp = wl.make_inputs(w)
    qw = oracle_inputs(w, inp)
    idx = inp["idx"]
    budget_s = 90.0
    rng = np.random.default_rng(1)
    probe = np.sort(rng.choice(w.n, size=min(w.n, 16), replace=False))
    t0 = time.perf_counter()
    oracle_rows(w, inp["x"], qw, idx, probe)
    per_row = (time.perf_counter() - t0) / len(probe)
    rows_per_step = int(max(1, min(w.n, budget_s / (args.steps + args.warmup) / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        oracle_rows(w, inp["x"], qw, idx, np.sort(rng.choice(w.n, rows_per_step, replace=False)))
    t0 = time.perf_counter()
    threads = 1
    for _ in range(args.steps):
        threads = oracle_rows(w, inp["x"], qw, idx, np.sort(rng.choice(w.n, rows_per_step, replace=False)))
    dt = time.perf_counter() - t0
    flops = w.flops / w.n * rows_per_step * args.steps
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": metric_name(w), "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{rows_per_step} random rows of the workload per step (of {w.n})"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------

def run_gpu(args, w: wl.Workload, world: int, rank: int, local: int):
    import quantized_moe_expert_device_gb300 as g

    lib = g.load_library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    inp = wl.make_inputs(w)
    idx_np = inp["idx"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    # Rotate enough distinct copies of every input that the working set exceeds 3x L2.
    per_copy = algorithmic_bytes(w, idx_np)
    copies = int(max(2, min(16, np.ceil(3 * l2 / max(per_copy, 1)))))
    if w.kind == "mlp":
        weights0 = []
        for key in ("w_gu", "w_dn"):
            w_dev = inp[key].to(dev)
            weights0 += list(g.gqmm_quantize(w_dev, group_size=w.group_size))
            del w_dev
        fn, ws_new = lib.gqmm_moe_mlp, (lambda: g.new_mlp_workspace(w.n, w.H, w.F, w.E, dev))
        sizes = (w.T, w.A, w.H, w.F, w.E, w.group_size, 4, g.ACTIVATIONS[MLP_ACTIVATION])
    else:
        w_dev = inp["w"].to(dev)
        weights0 = list(g.gqmm_quantize(w_dev, group_size=w.group_size))
        del w_dev
        if w.kind == "nn":  # no workspace: rows are independent, no route sort
            fn, ws_new = lib.gqmm_gather_qmm_nn, (lambda: None)
            sizes = (w.T, w.A, w.H, w.F, w.E, w.group_size, 4, 0)
        else:
            fn, ws_new = lib.gqmm_gather_qmm, (lambda: g.new_workspace(w.n, w.F, w.E, dev))
            sizes = (w.T, w.A, w.H, w.F, w.E, w.group_size, 4)
    x0 = inp["x"].to(dev)
    idx0 = None if idx_np is None else torch.from_numpy(np.ascontiguousarray(idx_np).view(np.int32)).to(dev)
    sets = []
    for c in range(copies):
        s = dict(x=x0.clone(), w=[t.clone() for t in weights0], idx=None if idx0 is None else idx0.clone(),
                 y=torch.empty(w.T, w.A, w.out_cols, dtype=torch.bfloat16, device=dev), ws=ws_new())
        sets.append(s)
    del x0, weights0, idx0
    torch.cuda.synchronize(dev)

    sptr = ctypes.c_void_p(stream.cuda_stream)
    fn_name = fn.__name__

    def argv(s, sorted_flag=0):
        P = ctypes.c_void_p
        if w.kind == "nn":
            return ((P(s["x"].data_ptr()),) + tuple(P(t.data_ptr()) for t in s["w"])
                    + (None if s["idx"] is None else P(s["idx"].data_ptr()),) + sizes + (P(s["y"].data_ptr()), sptr))
        return ((P(s["x"].data_ptr()),) + tuple(P(t.data_ptr()) for t in s["w"])
                + (None if s["idx"] is None else P(s["idx"].data_ptr()),) + sizes
                + (sorted_flag, 0, P(s["y"].data_ptr()), P(s["ws"].data_ptr()), s["ws"].numel(), sptr))

    calls = [argv(s) for s in sets]

    def step(i):
        rc = fn(*calls[i % copies])
        if rc != 0:
            raise RuntimeError(f"{fn_name} failed: {rc} {lib.gqmm_last_error().decode()}")

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    timer_slots = args.steps * GEMM_LAUNCHES_PER_STEP[w.kind]
    g.kernel_timer(timer_slots)  # events are created here, before the timed region
    g.kernel_timer(0)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    # Timed pass 1, the metric: K steps with nothing between the library's kernels (its own
    # kernel timer would put events between the route step and the GEMM, which stops the
    # GEMM's prologue from overlapping the route step).
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = g.launch_count()
    variants0 = {v: g.dispatch_count(v) for v in _VARIANT_KERNEL}
    t_host0 = time.perf_counter()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    t_host_enqueue = time.perf_counter() - t_host0
    torch.cuda.synchronize(dev)
    barrier(world)
    ms_total = ev0.elapsed_time(ev1)
    launches = g.launch_count() - launches0
    ran = [v for v in _VARIANT_KERNEL if g.dispatch_count(v) > variants0[v]]
    kernel = _VARIANT_KERNEL[ran[0]] if ran else "gemm_tc_kernel"
    # Hot pass (context only, not the metric): the same call repeated on one input set, so
    # inputs that fit in L2 stay there between steps.
    hot_steps = min(args.steps, 200)
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        fn(*calls[0])
    h0.record(stream)
    for _ in range(hot_steps):
        fn(*calls[0])
    h1.record(stream)
    torch.cuda.synchronize(dev)
    hot_ms = max_over_ranks(h0.elapsed_time(h1), world) / hot_steps
    # Timed pass 2, the roofline: the same K steps with CUDA events around every GEMM launch
    # on the call's stream (the library's kernel timer).
    g.kernel_timer(timer_slots)
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    n_timed, gemm_ms_total = g.kernel_timer_read()
    g.kernel_timer(0)
    if n_timed != timer_slots:
        raise RuntimeError(f"kernel timer recorded {n_timed} GEMM launches, expected {timer_slots}")
    status = 0
    for s in sets:
        if s["ws"] is not None:
            status |= g.gqmm_device_status(s["ws"])
    if status:
        raise RuntimeError(f"device status after timed region: {status:#x}")

    ms_max = max_over_ranks(ms_total, world)
    ms_per_step = ms_max / args.steps
    flops = float(w.flops)
    value = flops * world * args.steps / (ms_max * 1e-3) / 1e12

    peaks, peaks_src = load_peaks()
    alg_bytes = algorithmic_bytes(w, idx_np)
    # GEMM launches per step: 1 for gather_qmm, 2 for the expert MLP (its gate/up and down
    # projections); the roofline takes the step's FLOPs (bytes) over their summed durations.
    gemm_launches_per_step = n_timed / max(args.steps, 1)
    gemm_ms = gemm_ms_total / max(args.steps, 1)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if flops / alg_bytes >= ridge else "hbm"
    peak_source = f"{peaks_src} ({'bf16_tflops' if bound == 'tensor' else 'hbm_gbs'})"
    if w.kind == "nn":
        # CUDA-core kernel: the float32 FMA pipes (128 lanes per SM, 2 FLOP per FMA) at the
        # maximum SM clock; it issues two FMAs (dequantize, accumulate) per multiply-add of the
        # metric, so half of this peak is its ceiling
        bound = "alu"
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        sm_max = (clocks or {}).get("sm_max_mhz") or 2070
        peak = sms * 128 * 2 * sm_max * 1e6 / 1e12
        achieved = flops / (gemm_ms * 1e-3) / 1e12
        unit = "TFLOP/s"
        peak_source = f"derived: {sms} SMs x 128 FP32 lanes x 2 FLOP x {sm_max} MHz"
    elif bound == "tensor":
        achieved = flops / (gemm_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        unit = "TFLOP/s"
    else:
        achieved = alg_bytes / (gemm_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    t_roof_s = max(flops / (peaks["bf16_tflops"] * 1e12), alg_bytes / (peaks["hbm_gbs"] * 1e9))

    # ---- end to end: host-resident inputs, pinned, copied in and out every step ----
    # Every step copies its own inputs in from pinned host memory and its own result back.
    # Steps that move at least 1 MB run as a pipelined serving loop over two device buffer sets
    # and three streams: step i's inputs are copied in while step i-1 computes and step i-2's
    # result is copied out; a set is refilled only once the step that used it has finished with
    # its inputs and its result has left the device.  Smaller steps run everything on the call's
    # stream, where cross-stream events would cost more than the overlap saves.
    e2e_steps = max(3, min(args.steps, 200))
    x_h = inp["x"].pin_memory()
    idx_h = None if idx_np is None else torch.from_numpy(np.ascontiguousarray(idx_np).view(np.int32)).pin_memory()
    y_h = [torch.empty(w.T, w.A, w.out_cols, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = x_h.numel() * 2 + (0 if idx_h is None else idx_h.numel() * 4)
    d2h = y_h[0].numel() * 2
    h2d_s = torch.cuda.Stream(dev)
    d2h_s = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    pipelined = h2d + d2h >= (1 << 20)

    def e2e_step(i):
        b = i & 1
        s = sets[b]
        if not pipelined:
            s["x"].copy_(x_h, non_blocking=True)
            if idx_h is not None:
                s["idx"].copy_(idx_h, non_blocking=True)
            rc = fn(*calls[b])
            if rc != 0:
                raise RuntimeError(f"{fn_name} failed: {rc} {lib.gqmm_last_error().decode()}")
            y_h[b].copy_(s["y"], non_blocking=True)
            return
        with torch.cuda.stream(h2d_s):
            if i >= 2:
                h2d_s.wait_event(ev_done[b])  # step i - 2 is done with this set's inputs
            s["x"].copy_(x_h, non_blocking=True)
            if idx_h is not None:
                s["idx"].copy_(idx_h, non_blocking=True)
            ev_in[b].record(h2d_s)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])  # step i - 2's result has left this set's y
        rc = fn(*calls[b])
        if rc != 0:
            raise RuntimeError(f"{fn_name} failed: {rc} {lib.gqmm_last_error().decode()}")
        ev_done[b].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_done[b])
            y_h[b].copy_(s["y"], non_blocking=True)
            ev_out[b].record(d2h_s)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_s.wait_event(e0)
    d2h_s.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i + 4)
    stream.wait_event(ev_out[0])
    stream.wait_event(ev_out[1])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
    e2e_value = flops * world / (e2e_ms * 1e-3) / 1e12

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        qw = oracle_inputs(w, inp)
        rate, rows, secs, threads = oracle_rate(w, inp["x"], qw, idx_np, target_s=12.0)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} random rows of the workload ({w.flops / w.n * rows / 1e9:.2f} GFLOP, {secs:.1f} s)"}

    if rank != 0:
        return
    line = {
        "metric": metric_name(w),
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {**workload_config(w), "sorted_indices": False, "rows_per_expert": w.n / w.E,
                   "l2": f"inputs rotate over {copies} copies ({copies * per_copy / 1e6:.0f} MB > L2 {l2 / 1e6:.0f} MB)",
                   "gpu": torch.cuda.get_device_name(dev), "seeds": {"x": wl.SEED_X, "w": wl.SEED_W, "idx": wl.SEED_IDX},
                   "parallelism": f"replicas x{world}",
                   "hot": {"ms_per_step": hot_ms, "value": flops * world / (hot_ms * 1e-3) / 1e12,
                           "note": "one input set repeated (L2-warm where it fits); context, not the metric"}},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "traffic": measured_traffic(kernel, w.name), "kernel": kernel, "kernel_ms": gemm_ms,
                     "kernel_launches_per_step": gemm_launches_per_step,
                     "kernel_timing": "second timed pass of the same steps, CUDA events around each GEMM launch;"
                                      " kernel_ms = their summed duration per step",
                     "peak_source": peak_source},
        "op_roofline": {"t_min_us": t_roof_s * 1e6, "frac": t_roof_s / (ms_per_step * 1e-3),
                        "algorithmic_bytes": alg_bytes, "flops": flops},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "mode": "pipelined over 2 buffer sets and 3 streams" if pipelined else "serial on the call's stream"},
        "gpu_launches": launches,
        "clocks": clocks,
        "host_enqueue_ms_per_step": t_host_enqueue / args.steps * 1e3,
    }
    print(json.dumps(line), flush=True)


_CSRC = "quantized_moe_expert_device_gb300/csrc/"
# The sources each GEMM-step kernel is built from (a traffic record is stale once they change).
KERNEL_SOURCES = {
    "gemm_tc_kernel": (_CSRC + "gemm_tc.cu", _CSRC + "gqmm_internal.cuh"),
    "gemv_fma_kernel": (_CSRC + "gemv.cu", _CSRC + "gqmm_internal.cuh"),
    "gemv_mma_kernel": (_CSRC + "gemv_mma.cu", _CSRC + "gqmm_internal.cuh"),
    "gemm_nn_kernel": (_CSRC + "gemm_nn.cu", _CSRC + "gqmm_internal.cuh"),
}
# dispatch-count variant -> the kernel it launches for the GEMM step
_VARIANT_KERNEL = {"gemv": "gemv_fma_kernel", "gemv_mma": "gemv_mma_kernel", "gemm_narrow": "gemm_tc_kernel",
                   "gemm_tc": "gemm_tc_kernel", "nn": "gemm_nn_kernel"}


def kernel_source_sha(kernel):
    import hashlib

    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(kernel, workload):
    """DRAM bytes (read + write) of `kernel` from the committed ncu capture of this workload, per
    launch, or per step where a step launches it more than once (the expert MLP's two
    projections), matching the roofline's `achieved`; None when there is none or the kernel's
    sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")
    if kernel not in KERNEL_SOURCES or not os.path.exists(path):
        return None
    with open(path) as f:
        prof = json.load(f)
    if prof.get("source_sha256") != kernel_source_sha(kernel):
        return None
    return prof.get("dram_bytes_per_step", prof.get("dram_bytes_per_launch"))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="prefill_e64", choices=sorted(wl.workloads()))
    ap.add_argument("--impl", default="gqmm", choices=["gqmm", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    w = wl.workloads()[args.workload]
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, w, world, rank)
    else:
        run_gpu(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
