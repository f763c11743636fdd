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

    def qbytes(rows, K):  # one expert's packed codes + its scales (and biases)
        if w.mode == "mxfp4":
            return rows * (K // 2 + K // 32)
        if w.mode == "nvfp4":
            return rows * (K // 2 + K // 16) + 4  # + the expert's float32 scale
        if w.mode == "mxfp8":
            return rows * (K + K // 32)
        return rows * (K * w.bits // 8 + 4 * (K // w.group_size))  # bf16 scale and bias per group

    if w.kind == "mlp":
        weights = hit * (qbytes(2 * w.F, w.H) + qbytes(w.H, w.F))
    elif w.kind == "nn":  # W[e] is [K = H, N = F], quantized along F
        weights = hit * qbytes(w.H, w.F)
    else:
        weights = hit * qbytes(w.F, w.H)
    return int(weights + w.n * w.H * 2 + w.n * w.out_cols * 2 + (0 if idx is None else w.n * 4))


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs.  With timestamps, each
    sample carries nvidia-smi's own time, so summary(t0, t1) can take the samples of one window
    of host time (time.time())."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int, timestamps: bool = False):
        self.dev = device_index
        self.proc = None
        self.timestamps = timestamps
        self.samples = []  # (time or None, sm MHz, max sm MHz, set of active reasons)
        self.path = os.path.join(tempfile.gettempdir(), f"gqmm_clocks_bench_{os.getpid()}_{id(self)}.csv")

    def start(self):
        query = ("timestamp," if self.timestamps else "") + self.QUERY
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={query}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    @staticmethod
    def _stamp(text):
        import datetime

        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                ts = None
                if self.timestamps:
                    if not parts:
                        continue
                    ts = self._stamp(parts[0])
                    parts = parts[1:]
                if len(parts) < 9:
                    continue
                try:
                    sm, smax = float(parts[1]), float(parts[2])
                except ValueError:
                    continue
                active = {nm for nm, v in zip(self.REASONS, parts[5:9]) if v.lower() == "active"}
                self.samples.append((ts, sm, smax, active))
        try:
            os.remove(self.path)
        except OSError:
            pass
        return self.summary()

    def summary(self, t0=None, t1=None):
        sel = [s_ for s_ in self.samples if t0 is None or (s_[0] is not None and t0 <= s_[0] <= t1)]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for s_ in sel:
            reasons |= s_[3]
        return {"sm_mhz": float(np.median([s_[1] for s_ in sel])), "sm_max_mhz": max(s_[2] for s_ in sel),
                "reasons": sorted(reasons), "samples": len(sel)}


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
    if w.mode != "affine":
        return oracle.quantize_fp(inp["w"], w.mode)
    return oracle.quantize(inp["w"], group_size=w.group_size, bits=w.bits)


def oracle_rows(w: wl.Workload, x_cpu, qw, idx, rows):
    """The oracle on the listed flat rows; returns its thread count."""
    import oracle

    if w.kind == "mlp":
        oracle.moe_mlp(x_cpu, qw[0], qw[1], idx, w.E, group_size=w.group_size, rows=rows)
    elif w.kind == "nn":
        oracle.gather_qmm_nn(x_cpu, *qw, idx, w.E, group_size=w.group_size, rows=rows)
        return 1  # numpy row products, one thread
    elif w.mode != "affine":
        oracle.gather_qmm_fp(x_cpu, *qw, idx, w.E, w.mode, rows=rows)
        return oracle.nthreads_default()
    else:
        oracle.gather_qmm(x_cpu, *qw, idx, w.E, group_size=w.group_size, bits=w.bits, rows=rows)
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
    c.update({"E": w.E, "group_size": w.group_size, "bits": w.bits, "routing": w.routing})
    if w.mode != "affine":
        c.update({"mode": w.mode, "bits": 8 if w.mode == "mxfp8" else 4})
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

# Workloads timed after the headline, each on its own rotated inputs, into the line's per_config
# block: the equal-FLOPs dense control, the rows-per-expert sweep, the Mixtral-like expert shape,
# dense and MoE decode at 1-8 rows, the other group sizes, the expert MLP and transpose=False.
PER_CONFIG = ["prefill_dense", "prefill_e64_g32", "prefill_e64_g128", "prefill_e64_b2", "prefill_e64_b3",
              "prefill_e64_b8", "prefill_e64_mxfp4", "prefill_e64_nvfp4", "prefill_e64_mxfp8",
              "sweep_r4", "sweep_r8", "sweep_r16", "sweep_r32", "sweep_r64", "sweep_r128", "mixtral",
              "decode_dense_m1", "decode_dense_m2", "decode_dense_m4", "decode_dense_m8",
              "decode_moe_m1", "decode_moe_m2", "decode_moe_m4", "decode_moe_m8",
              "mlp_e64", "mlp_decode_m8", "nn_e4", "nn_e64"]
ROTATE_L2_MULTIPLE = 4        # distinct input copies cover at least this many times the L2 size
MAX_COPIES = 96               # ... within this many copies
MAX_CLONE_BYTES = 24 << 30    # ... and this many bytes of copies
STRIPS = 5                    # the timed steps are split into this many strips (median reported)


def _weights_on_device(g, w: wl.Workload, inp, dev):
    """The workload's weights quantized on the GPU: [wq, scales, biases] (both projections for the
    expert MLP), or [wq, scales, tensor scales or None] for a floating-point mode."""
    out = []
    for key in (("w_gu", "w_dn") if w.kind == "mlp" else ("w",)):
        w_dev = inp[key].to(dev)
        if w.mode != "affine":
            out += list(g.gqmm_quantize_fp(w_dev, w.mode))
        else:
            out += list(g.gqmm_quantize(w_dev, group_size=w.group_size, bits=w.bits))
        del w_dev
    return out


class Prepared:
    """Device-resident inputs of one workload, rotated over enough copies that one pass over them
    reads at least ROTATE_L2_MULTIPLE x L2 of distinct bytes, and the C-ABI call of each copy."""

    def __init__(self, g, lib, w: wl.Workload, dev, stream, cache):
        self.w, self.g, self.lib = w, g, lib
        self.inp = wl.make_inputs(w, cache=cache)
        idx_np = self.inp["idx"]
        self.idx_np = idx_np
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.per_copy = algorithmic_bytes(w, idx_np)
        weights0 = _weights_on_device(g, w, self.inp, dev)
        clone_bytes = (sum(t.numel() * t.element_size() for t in weights0 if t is not None)
                       + w.n * (w.H + w.out_cols) * 2 + w.n * 4)
        want = int(np.ceil(ROTATE_L2_MULTIPLE * self.l2 / max(self.per_copy, 1)))
        self.copies = int(max(2, min(want, MAX_COPIES, MAX_CLONE_BYTES // max(clone_bytes, 1))))
        if w.kind == "mlp":
            fn, ws_new = lib.gqmm_moe_mlp, (lambda: g.new_mlp_workspace(w.n, w.H, w.F, w.E, dev))
            sizes = (w.T, w.A, w.H, w.F, w.E, w.group_size, 4, g.ACTIVATIONS[MLP_ACTIVATION])
        elif w.kind == "nn":  # W[e] is [K = H, N = F]; the workspace is sized for N output columns
            fn, ws_new = lib.gqmm_gather_qmm_nn, (lambda: g.new_workspace(w.n, w.F, w.E, dev))
            sizes = (w.T, w.A, w.H, w.F, w.E, w.group_size, 4)
        else:
            ws_new = lambda: g.new_workspace(w.n, w.F, w.E, dev)  # noqa: E731
            if w.mode != "affine":
                fn, sizes = lib.gqmm_gather_qmm_fp, (w.T, w.A, w.H, w.F, w.E, g.MODES[w.mode])
            else:
                fn, sizes = lib.gqmm_gather_qmm, (w.T, w.A, w.H, w.F, w.E, w.group_size, w.bits)
        x0 = self.inp["x"].to(dev)
        idx0 = None if idx_np is None else torch.from_numpy(np.ascontiguousarray(idx_np).view(np.int32)).to(dev)
        self.sets = []
        for c in range(self.copies):
            last = c == self.copies - 1  # the last copy takes the originals instead of cloning them
            self.sets.append(dict(
                x=x0 if last else x0.clone(),
                w=weights0 if last else [None if t is None else t.clone() for t in weights0],
                idx=None if idx0 is None else (idx0 if last else idx0.clone()),
                y=torch.empty(w.T, w.A, w.out_cols, dtype=torch.bfloat16, device=dev), ws=ws_new()))
        torch.cuda.synchronize(dev)
        self.fn, self.fn_name = fn, fn.__name__
        P = ctypes.c_void_p

        def argv(st, sptr):
            head = (P(st["x"].data_ptr()),) + tuple(None if t is None else P(t.data_ptr()) for t in st["w"]) + (
                None if st["idx"] is None else P(st["idx"].data_ptr()),) + sizes
            return head + (0, 0, P(st["y"].data_ptr()), P(st["ws"].data_ptr()), st["ws"].numel(), sptr)

        self._argv = argv
        self.calls = self.calls_on(stream)

    def calls_on(self, stream):
        """The C-ABI arguments of every input copy, for a call on `stream`."""
        sptr = ctypes.c_void_p(stream.cuda_stream)
        return [self._argv(st, sptr) for st in self.sets]

    def step(self, i):
        rc = self.fn(*self.calls[i % self.copies])
        if rc != 0:
            raise RuntimeError(f"{self.fn_name} failed: {rc} {self.lib.gqmm_last_error().decode()}")

    def status(self):
        st = 0
        for s_ in self.sets:
            if s_["ws"] is not None:
                st |= self.g.gqmm_device_status(s_["ws"])
        return st

    def l2_note(self):
        return (f"inputs rotate over {self.copies} copies ({self.copies * self.per_copy / 1e6:.0f} MB of algorithmic "
                f"bytes; L2 {self.l2 / 1e6:.0f} MB)")


def timed_strips(prep: Prepared, steps: int, stream, world: int):
    """The metric's timed region: `steps` calls with nothing between the library's kernels, split
    into STRIPS strips with CUDA events on the call's stream at the strip boundaries.  Returns
    (total ms, [ms per step of each strip])."""
    bounds = [round(k * steps / STRIPS) for k in range(STRIPS + 1)]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(STRIPS + 1)]
    barrier(world)
    torch.cuda.synchronize()
    evs[0].record(stream)
    for k in range(STRIPS):
        for i in range(bounds[k], bounds[k + 1]):
            prep.step(i)
        evs[k + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    strips = [evs[k].elapsed_time(evs[k + 1]) / max(bounds[k + 1] - bounds[k], 1) for k in range(STRIPS)]
    return evs[0].elapsed_time(evs[STRIPS]), strips


MIN_GRAPH_CALLS = 20  # calls per captured strip


def graph_strips(prep: Prepared, steps: int, world: int, stream):
    """The metric's timed region: `steps` calls captured as CUDA graphs of at least
    MIN_GRAPH_CALLS back-to-back calls (up to STRIPS strips, each its own graph over the next
    input copies), replayed once untimed and then once each between CUDA events on the stream.
    Graph replay takes the host's per-call launch cost out of the device timeline, as a serving
    loop that replays captured decode steps does.  Returns (total ms, [ms per step of each
    strip], library launches per step)."""
    g = prep.g
    n_strips = max(1, min(STRIPS, steps // MIN_GRAPH_CALLS))
    bounds = [round(k * steps / n_strips) for k in range(n_strips + 1)]
    graphs = []
    launches0 = g.launch_count()
    for k in range(n_strips):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="relaxed"):
            calls = prep.calls_on(torch.cuda.current_stream())
            for i in range(bounds[k], bounds[k + 1]):
                rc = prep.fn(*calls[i % prep.copies])
                if rc != 0:
                    raise RuntimeError(f"{prep.fn_name} failed in capture: {rc} {prep.lib.gqmm_last_error().decode()}")
        graphs.append(graph)
    launches = (g.launch_count() - launches0) / max(steps, 1)
    for graph in graphs:
        graph.replay()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_strips + 1)]
    barrier(world)
    torch.cuda.synchronize()
    evs[0].record(stream)
    for k in range(n_strips):
        graphs[k].replay()
        evs[k + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    strips = [evs[k].elapsed_time(evs[k + 1]) / max(bounds[k + 1] - bounds[k], 1) for k in range(n_strips)]
    del graphs
    return evs[0].elapsed_time(evs[n_strips]), strips, launches


def kernel_pass(prep: Prepared, steps: int, world: int):
    """The same steps again with CUDA events around every GEMM launch on the call's stream (the
    library's kernel timer; those events would stop the GEMM's prologue from overlapping the route
    step, hence a separate pass).  Returns (GEMM ms per step, GEMM launches per step)."""
    g = prep.g
    slots = steps * GEMM_LAUNCHES_PER_STEP[prep.w.kind]
    g.kernel_timer(slots)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        prep.step(i)
    torch.cuda.synchronize()
    barrier(world)
    n_timed, ms_total = g.kernel_timer_read()
    g.kernel_timer(0)
    if n_timed != slots:
        raise RuntimeError(f"kernel timer recorded {n_timed} GEMM launches, expected {slots}")
    return ms_total / max(steps, 1), n_timed / max(steps, 1)


def kernel_time(prep: Prepared, steps: int, world: int, step_ms: float, launches_per_step: float):
    """(ms per step of the GEMM kernel(s), their launches per step, how it was timed).  When the
    step is those launches alone (dense or in-kernel-planned decode), the graph-replayed step time
    is their time; otherwise a separate pass of plain launches puts CUDA events around each GEMM
    launch (the library's kernel timer)."""
    per_step = GEMM_LAUNCHES_PER_STEP[prep.w.kind]
    if launches_per_step <= per_step:
        return step_ms, float(per_step), "the step is the kernel alone: graph replay, events at strip boundaries"
    gemm_ms, n = kernel_pass(prep, steps, world)
    return gemm_ms, n, ("a separate pass of plain launches, CUDA events around each GEMM launch;"
                        " kernel_ms = their summed duration per step")


def roofline_entry(w: wl.Workload, alg_bytes: int, gemm_ms: float, peaks, peaks_src, sm_max, sms, kernel):
    flops = float(w.flops)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if flops / alg_bytes >= ridge else "hbm"
    peak_source = f"{peaks_src} ({'bf16_tflops' if bound == 'tensor' else 'hbm_gbs'})"
    if bound == "tensor":
        achieved, peak, unit = flops / (gemm_ms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = alg_bytes / (gemm_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": measured_traffic(kernel, w.name), "kernel": kernel, "kernel_ms": gemm_ms,
            "peak_source": peak_source}


def op_roofline_entry(w: wl.Workload, alg_bytes: int, ms_per_step: float, peaks):
    flops = float(w.flops)
    t_roof_s = max(flops / (peaks["bf16_tflops"] * 1e12), alg_bytes / (peaks["hbm_gbs"] * 1e9))
    return {"t_min_us": t_roof_s * 1e6, "frac": t_roof_s / (ms_per_step * 1e-3), "algorithmic_bytes": alg_bytes,
            "flops": flops}


def _kernel_of(g, variants0):
    ran = [v for v in _VARIANT_KERNEL if g.dispatch_count(v) > variants0[v]]
    return _VARIANT_KERNEL[ran[0]] if ran else "gemm_tc_kernel"


def measure_config(g, lib, w: wl.Workload, dev, stream, world, cache, peaks, peaks_src, sms, target_s: float,
                   max_steps: int):
    """One per_config entry: the headline's method (rotated inputs, strips, kernel-timer pass) on
    another workload, with the step count chosen so its timed region lasts about target_s."""
    prep = Prepared(g, lib, w, dev, stream, cache)
    for i in range(max(3, min(prep.copies, 20))):
        prep.step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(10):
        prep.step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    est_ms = e0.elapsed_time(e1) / 10
    steps = int(min(max_steps, max(4 * STRIPS, target_s * 1e3 / max(est_ms, 1e-4))))
    variants0 = {v: g.dispatch_count(v) for v in _VARIANT_KERNEL}
    t0 = time.time()
    ms_total, strips, launches = graph_strips(prep, steps, world, stream)
    t1 = time.time()
    kernel = _kernel_of(g, variants0)
    gemm_ms, gemm_launches, timing = kernel_time(prep, steps, world, ms_total / steps, launches)
    status = prep.status()
    if status:
        raise RuntimeError(f"{w.name}: device status after the timed region: {status:#x}")
    ms_max = max_over_ranks(ms_total, world)
    ms_per_step = ms_max / steps
    alg = algorithmic_bytes(w, prep.idx_np)
    entry = {
        "workload": w.name, "metric": metric_name(w), "config": workload_config(w),
        "value": float(w.flops) * world / (ms_per_step * 1e-3) / 1e12, "unit": "TFLOP/s",
        "ms_per_step": ms_per_step, "steps": steps,
        "strips": {"n": len(strips), "median_ms_per_step": float(np.median(strips)), "ms_per_step": strips},
        "hbm_gbs": alg / (ms_per_step * 1e-3) / 1e9,
        "roofline": dict(roofline_entry(w, alg, gemm_ms, peaks, peaks_src, 2070, sms, kernel),
                         kernel_launches_per_step=gemm_launches, kernel_timing=timing),
        "op_roofline": op_roofline_entry(w, alg, ms_per_step, peaks),
        "gpu_launches_per_step": launches, "l2": prep.l2_note(), "window": (t0, t1),
    }
    del prep
    torch.cuda.empty_cache()
    return entry


def run_gpu(args, w: wl.Workload, world: int, rank: int, local: int):
    import quantized_moe_expert_device_gb300 as g

    lib = g.load_library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cache = {}
    prep = Prepared(g, lib, w, dev, stream, cache)
    inp, idx_np = prep.inp, prep.idx_np

    for i in range(args.warmup):
        prep.step(i)
    torch.cuda.synchronize(dev)
    g.kernel_timer(args.steps * GEMM_LAUNCHES_PER_STEP[w.kind])  # events are created here, before the timed region
    g.kernel_timer(0)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    # Timed pass 1, the metric: K steps captured as CUDA graphs, replayed in strips.
    variants0 = {v: g.dispatch_count(v) for v in _VARIANT_KERNEL}
    ms_total, strips, launches_per_step = graph_strips(prep, args.steps, world, stream)
    launches = int(round(launches_per_step * args.steps))
    kernel = _kernel_of(g, variants0)
    # Context: the same K steps as plain stream launches from the host (per-call host cost included).
    t_host0 = time.perf_counter()
    plain_ms, _ = timed_strips(prep, args.steps, stream, world)
    t_host_enqueue = time.perf_counter() - t_host0
    # Hot pass (context only, not the metric): the same call repeated on one input set, so
    # inputs that fit in L2 stay there between steps.
    hot_steps = min(args.steps, 200)
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        prep.fn(*prep.calls[0])
    h0.record(stream)
    for _ in range(hot_steps):
        prep.fn(*prep.calls[0])
    h1.record(stream)
    torch.cuda.synchronize(dev)
    hot_ms = max_over_ranks(h0.elapsed_time(h1), world) / hot_steps
    # The roofline: the GEMM kernel's own time per step.
    gemm_ms, gemm_launches_per_step, kernel_timing = kernel_time(prep, args.steps, world, ms_total / args.steps,
                                                                 launches_per_step)
    clocks = sampler.stop()
    status = prep.status()
    if status:
        raise RuntimeError(f"device status after timed region: {status:#x}")

    ms_max = max_over_ranks(ms_total, world)
    ms_per_step = ms_max / args.steps
    flops = float(w.flops)
    value = flops * world * args.steps / (ms_max * 1e-3) / 1e12
    peaks, peaks_src = load_peaks()
    alg_bytes = algorithmic_bytes(w, idx_np)
    sm_max = (clocks or {}).get("sm_max_mhz") or 2070
    roof = dict(roofline_entry(w, alg_bytes, gemm_ms, peaks, peaks_src, sm_max, sms, kernel),
                kernel_launches_per_step=gemm_launches_per_step, kernel_timing=kernel_timing)

    # ---- end to end: host-resident inputs, pinned, copied in and out every step ----
    # Every step copies its own inputs in from pinned host memory and its own result back.
    # Steps that move at least 1 MB run as a pipelined serving loop over two device buffer sets
    # and three streams: step i's inputs are copied in while step i-1 computes and step i-2's
    # result is copied out; a set is refilled only once the step that used it has finished with
    # its inputs and its result has left the device.  Smaller steps run everything on the call's
    # stream, where cross-stream events would cost more than the overlap saves.
    sets, calls, fn = prep.sets, prep.calls, prep.fn
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

    def call(b):
        rc = fn(*calls[b])
        if rc != 0:
            raise RuntimeError(f"{prep.fn_name} failed: {rc} {lib.gqmm_last_error().decode()}")

    def e2e_step(i):
        b = i & 1
        s = sets[b]
        if not pipelined:
            s["x"].copy_(x_h, non_blocking=True)
            if idx_h is not None:
                s["idx"].copy_(idx_h, non_blocking=True)
            call(b)
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
        call(b)
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
    l2_note = prep.l2_note()
    del prep, sets, calls
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp, idx_np)

    per_config = None
    if not args.no_per_config:
        names = [n for n in (args.per_config.split(",") if args.per_config else PER_CONFIG) if n and n != w.name]
        sampler = ClockSampler(local, timestamps=True)
        sampler.start()
        time.sleep(0.3)
        per_config = []
        for name in names:
            per_config.append(measure_config(g, lib, wl.workloads()[name], dev, stream, world, cache, peaks, peaks_src,
                                             sms, target_s=args.config_seconds, max_steps=max(args.steps, 20000)))
        sampler.stop()
        for e in per_config:
            e["clocks"] = sampler.summary(*e.pop("window"))

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
                   "l2": l2_note, "gpu": torch.cuda.get_device_name(dev),
                   "seeds": {"x": wl.SEED_X, "w": wl.SEED_W, "idx": wl.SEED_IDX},
                   "parallelism": f"replicas x{world}",
                   "strips": {"n": len(strips), "median_ms_per_step": float(np.median(strips)), "ms_per_step": strips,
                              "note": "the timed steps as CUDA graphs of >= 20 back-to-back calls, replayed with"
                                      " CUDA events at the strip boundaries; value and ms_per_step cover all of them"},
                   "stream_launches": {"ms_per_step": plain_ms / args.steps,
                                       "value": flops * world / (plain_ms / args.steps * 1e-3) / 1e12,
                                       "note": "the same steps as plain calls from the host, one at a time"},
                   "hot": {"ms_per_step": hot_ms, "value": flops * world / (hot_ms * 1e-3) / 1e12,
                           "note": "one input set repeated (L2-warm where it fits); context, not the metric"}},
        "roofline": roof,
        "op_roofline": op_roofline_entry(w, alg_bytes, ms_per_step, peaks),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "mode": "pipelined over 2 buffer sets and 3 streams" if pipelined else "serial on the call's stream"},
        "gpu_launches": launches,
        "clocks": clocks,
        "host_enqueue_ms_per_step": t_host_enqueue / args.steps * 1e3,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform

    return platform.processor() or platform.machine()


def cpu_baseline(w: wl.Workload, inp, idx_np):
    """The oracle, as it stands, on the host cores: the headline workload on a bounded row sample
    (all cores), its dequantize and gather steps timed apart, and single-threaded rates on the
    tiny correctness case and on one-row dense and MoE decode."""
    import oracle

    qw = oracle_inputs(w, inp)
    rate, rows, secs, threads = oracle_rate(w, inp["x"], qw, idx_np, target_s=12.0)
    out = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": f"{rows} random rows of the workload ({w.flops / w.n * rows / 1e9:.2f} GFLOP, {secs:.1f} s)",
           "cpu_model": cpu_model()}
    if w.kind == "gather":
        # the two steps of the oracle apart: dequantizing every hit expert's weights (float64),
        # and the dot products of the sampled rows against them (numpy matmul, float64)
        hit = np.unique(idx_np) if idx_np is not None else np.arange(w.E)
        t0 = time.perf_counter()
        deq = [oracle.dequantize(qw[0][e], qw[1][e], qw[2][e], w.group_size) for e in hit[:8]]
        t_deq = (time.perf_counter() - t0) / len(deq) * len(hit)
        out["dequant_s_per_step"] = t_deq
        out["dequant_note"] = f"dequantize of the {len(hit)} hit experts, timed on {len(deq)} and scaled"
        del deq
    single = {}
    for name in ("tiny", "decode_dense_m1", "decode_moe_m1"):
        sw = wl.workloads()[name]
        sin = wl.make_inputs(sw)
        sq = oracle.quantize(sin["w"])
        t0 = time.perf_counter()
        oracle.gather_qmm(sin["x"], *sq, sin["idx"], sw.E, nthreads=1)
        dt = time.perf_counter() - t0
        single[name] = {"value": sw.flops / dt / 1e12, "unit": "TFLOP/s", "s_per_call": dt, "threads": 1}
    out["single_thread"] = single
    return out


_CSRC = "quantized_moe_expert_device_gb300/csrc/"
# The sources each GEMM-step kernel is built from (a traffic record is stale once they change).
KERNEL_SOURCES = {
    "gemm_tc_kernel": (_CSRC + "gemm_tc.cu", _CSRC + "formats.cuh", _CSRC + "gqmm_internal.cuh"),
    "gemv_fma_kernel": (_CSRC + "gemv.cu", _CSRC + "gqmm_internal.cuh"),
    "gemv_mma_kernel": (_CSRC + "gemv_mma.cu", _CSRC + "gqmm_internal.cuh"),
}
# dispatch-count variant -> the kernel it launches for the GEMM step
_VARIANT_KERNEL = {"gemv": "gemv_fma_kernel", "gemv_mma": "gemv_mma_kernel", "gemm_narrow": "gemm_tc_kernel",
                   "gemm_tc": "gemm_tc_kernel"}


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
    ap.add_argument("--no-per-config", action="store_true", help="time the headline workload only")
    ap.add_argument("--per-config", default="", help="comma-separated workloads for the per_config block")
    ap.add_argument("--config-seconds", type=float, default=0.25, help="timed seconds per per_config workload")
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
