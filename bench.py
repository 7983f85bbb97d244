"""Benchmark of the FP8 scaled linear layer hot path on one GB300.

Workload (the headline configuration): one FP8 linear, M = N = K = 4096,
TE-style delayed scaling, X ~ N(0,1) and G ~ N(0,1e-3) drawn fresh for every
step (20 seeded sets, 1.25 GiB together, rotated so the inputs of a step are
never L2-resident), W ~ N(0,0.02) fixed, 16-step weight amax history, X and G
scales lagged one call.  One step = the whole hot path, one native call
(fp8_linear_step_delayed), seven kernel launches:
    state step (refresh every 16th) -> amax reset ->
    quantise X and W (delayed, q only; emits amax_x, amax_w), one launch ->
    fprop GEMM ; beside it, on the library's second stream: record amax_w +
    lag-update the x scale ; quantise+transpose G (emits amax_g), quantise X
    again, transposed, with the updated x scale, and transpose Wq's bytes into
    Wqᵀ, one launch ; lag-update the g scale -> dgrad and wgrad GEMMs in one
    launch.
Metric: GEMM TFLOP/s of the whole step (3 x 2*4096^3 FLOP per step divided by
the step time), plus per-kernel achieved TFLOP/s and GB/s (CUDA events at the
kernel boundaries of further steps run after the timed region), the roofline
of the dgrad+wgrad launch, end-to-end figures with host copies, SM clocks
sampled during the timed region, and the CPU oracle's time on a bounded
sample.  On one GPU the line
also carries `workloads`: configuration 1's latency (quantise X, W + fprop at
64x256x256, in one launch and in three), the MLP block, the packed THD batch and the block recipe
(whole-step TFLOP/s and each one's dominant kernel), and the quantisers at
2^30 elements.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    python bench.py --workload mlp|thd|block|sweep|config1   (one configuration)

With N > 1 (torchrun), every rank runs an independent replica on its own
GPU (weak scaling; the path has no exchange on one GPU) and rank 0 reports
the aggregate with the max time over ranks.  --impl reference times the CPU
oracle (the slow, obviously correct restatement) on a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import shutil
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "FP8 linear fwd+bwd TFLOP/s & quantize GB/s vs GB300 FP8/HBM peak"
CFG = synth.CONFIG2
M, N, K = CFG["M"], CFG["N"], CFG["K"]
N_SETS = CFG["steps"]
GEMM_FLOP = 2.0 * M * N * K
STEP_FLOP = 3 * GEMM_FLOP
# algorithmic bytes of the quantisers per step (bf16 in, e4m3 out)
# forward launch: X -> Xq (3 B/el) and W -> Wq, Wqᵀ (4 B/el); backward launch:
# G -> Gq, Gqᵀ (4 B/el) and X -> Xqᵀ (3 B/el)
# algorithmic bytes of the step's two quantiser launches: forward X -> xq and
# W -> wq (bf16 read, e4m3 written); backward G -> gq, gqt and X -> xqt, plus
# wqt as the byte transpose of wq (read and written once)
QBYTES = {"quant_fwd": 3 * M * K + 3 * N * K, "quant_bwd": 4 * M * N + 3 * M * K + 2 * N * K}
FP8_PER_BF16 = 2.0  # nominal dense FP8 : BF16 tensor rate on Blackwell (4.5 : 2.25 PFLOP/s)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], src="measured")
    return dict(hbm=6800.0, bf16=1900.0, src="fallback")


def profile_traffic(name: str):
    """Per-launch DRAM bytes recorded in the committed ncu summary, or None."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", open(p).read())
    return float(m.group(1)) if m else None


REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
# NVML clock-event reason bits (nvmlClocksEventReason*) of those four
NVML_REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                    "hw_thermal_slowdown": 0x40}


def clock_summary(rows, source):
    """rows: (sm_mhz, max_sm_mhz, set of reason names) per sample."""
    if not rows:
        return None
    reasons = sorted({r for _, _, rs in rows for r in rs})
    return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
            "reasons": reasons, "samples": len(rows), "source": source}


class ClockSampler:
    """SM clock and throttle reasons sampled while the timed region runs.

    Reads NVML (the driver's management library, as nvidia-smi does) from a
    thread about every millisecond, so that short timed regions still get
    samples; falls back to nvidia-smi at 50 ms when NVML cannot be loaded.
    Read-only: no clock or other setting is changed."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_s: float = 0.001):
        self.index = index
        self.period = period_s
        self.proc = None
        self.lines = []
        self.rows = []
        self.nvml = None
        self.stop = threading.Event()
        self.t = None

    def _nvml_open(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            lib.nvmlShutdown()
            return False
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        if reasons_fn is None:
            lib.nvmlShutdown()
            return False
        self.nvml = (lib, h, reasons_fn)
        return True

    def _nvml_loop(self):
        import ctypes
        lib, h, reasons_fn = self.nvml
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and  # NVML_CLOCK_SM
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                    reasons_fn(h, ctypes.byref(rs)) == 0):
                names = {n for n, b in NVML_REASON_BITS.items() if rs.value & b}
                self.rows.append((float(clk.value), float(mx.value), names))
            time.sleep(self.period)

    def __enter__(self):
        if self._nvml_open():
            self.t = threading.Thread(target=self._nvml_loop, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.rows and time.time() - t0 < 5:
                time.sleep(0.001)
            return self
        exe = shutil.which("nvidia-smi")
        if exe:
            self.proc = subprocess.Popen(
                [exe, f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()  # the first sample marks the sampler as running
            while not self.lines and time.time() - t0 < 10 and self.proc.poll() is None:
                time.sleep(0.01)
        return self

    def mark(self):
        """Index of the next sample: samples from here on fall in the region."""
        return len(self.rows) if self.nvml else len(self.lines)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.nvml:
            self.stop.set()
            self.t.join(timeout=2)
            self.nvml[0].nvmlShutdown()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, start: int = 0):
        if self.nvml:
            return clock_summary(list(self.rows[start:]), "nvml")
        rows = []
        for ln in self.lines[start:]:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                names = {REASON_NAMES[i] for i, v in enumerate(parts[2:])
                         if v.lower() in ("active", "1")}
                rows.append((float(parts[0]), float(parts[1]), names))
            except ValueError:
                continue
        return clock_summary(rows, "nvidia-smi")


# --------------------------------------------------------------- GPU arm ---

# the step's event segments; dgrad and wgrad run as one launch (between the
# sixth and seventh events), the last segment is empty
SEGMENTS = ["quant_fwd", "gemm_fprop", "meta_fwd", "quant_bwd", "meta_bwd", "gemm_dgrad_wgrad",
            "empty"]


class Step:
    """One delayed-scaling training step = one native call
    (fp8_linear_step_delayed), with optional per-segment events."""

    def __init__(self, fp8, torch, dev, x_sets, g_sets, w):
        self.fp8, self.torch = fp8, torch
        self.x_sets, self.g_sets, self.w = x_sets, g_sets, w
        self.io = fp8.LinearStep(M, N, K, device=dev)
        self.meta = fp8.Fp8Meta(16, device=dev)
        self.count = [0]
        self.launches = 0
        self.events = None  # per-step event lists of the timed region
        self.pool = []      # events created (and recorded once) ahead of it

    def prepare_events(self, steps, every):
        """Create the timed region's events up front so the region itself
        only passes their handles to the native call; steps without events
        get None."""
        self.pool = []
        for i in range(steps):
            if i % every != 0:
                self.pool.append(None)
                continue
            ev = [self.torch.cuda.Event(enable_timing=True) for _ in range(len(SEGMENTS) + 1)]
            for e in ev:
                e.record()
            self.pool.append(ev)
        self.pool.reverse()
        self.events = []

    def run(self, t, x=None, g=None):
        x = self.x_sets[t % len(self.x_sets)] if x is None else x
        g = self.g_sets[t % len(self.g_sets)] if g is None else g
        self.io.set_inputs(x, self.w, g)
        ev = None
        if self.events is not None and self.pool:
            ev = self.pool.pop()
            if ev is not None:
                self.events.append(ev)
        self.fp8.fp8_linear_step_delayed(self.meta, self.count, self.io, events=ev)
        # kernels: the amax reset, 2 quantiser launches, fprop, one
        # dgrad/wgrad launch, 2 state updates (+1 refresh every 16 steps)
        self.launches += 7 + (1 if self.count[0] % 16 == 0 else 0)


def kernel_times(steps_events):
    """Average ms per launch of each segment over the timed steps."""
    acc = {k: [] for k in SEGMENTS}
    for ev in steps_events:
        for i, name in enumerate(SEGMENTS):
            acc[name].append(ev[i].elapsed_time(ev[i + 1]))
    return {k: sum(v) / len(v) for k, v in acc.items()}


def max_over_ranks(values, device=None):
    """Element-wise maximum of each rank's floats over all ranks, so the job
    is timed by its slowest replica; the values unchanged when no process
    group of more than one rank is up."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def headline_config(world: int) -> dict:
    """The headline workload's config, the same dict on both arms."""
    return {"workload": "one FP8 linear fwd+dgrad+wgrad, delayed scaling, M=N=K=4096, "
                        "16-step amax history, fresh X/G per step",
            "M": M, "N": N, "K": K, "recipe": "delayed", "input_sets": N_SETS,
            "l2": "inputs rotate over 20 X/G sets (1.25 GiB) > 129 MB L2",
            "parallelism": f"replicas x{world}"}


def whole_job_tflops(ms_step: float, world: int) -> float:
    """Every rank runs one full 4096^3 step per step (replicas, weak
    scaling): the job's FLOPs over the slowest rank's step time."""
    return STEP_FLOP * world / (ms_step * 1e-3) / 1e12


def gpu_arm(args, rank, world):
    import torch
    import scaled_linear_layers_gb300 as fp8

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def to_dev(h):
        return torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)

    seed = CFG["seed"] + rank
    w = to_dev(synth.normal_bf16((N, K), CFG["w_sigma"], seed, "w"))
    x_host = [synth.normal_bf16((M, K), CFG["x_sigma"], seed, "x", t) for t in range(N_SETS)]
    g_host = [synth.normal_bf16((M, N), CFG["g_sigma"], seed, "g", t) for t in range(N_SETS)]
    x_sets = [to_dev(h) for h in x_host]
    g_sets = [to_dev(h) for h in g_host]
    step = Step(fp8, torch, dev, x_sets, g_sets, w)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for t in range(args.warmup):
        step.run(t)
    fp8.fp8_check_device_status()
    barrier()

    # --- device-resident timed region: the API's step as a caller runs it
    # (nothing recorded inside it; an event between two kernels stops their
    # programmatic overlap and puts a step's kernels on one stream, which cost
    # the region about 2 % when every 10th step carried events)
    torch.cuda.synchronize()
    step.launches = 0
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        first = clk.mark()
        t_start.record()
        for t in range(args.warmup, args.warmup + args.steps):
            step.run(t)
        t_end.record()
        barrier()
        clocks = clk.summary(first)
    launches = step.launches
    ms_total = t_start.elapsed_time(t_end)
    fp8.fp8_check_device_status()

    # --- per-kernel segments: the same steps continued live right after the
    # timed region, as many again, with CUDA events at every kernel boundary
    # of every event_every-th step (the others run as the timed ones do, so
    # the event steps see the loop's steady power state)
    segs = None
    n_ev = 0
    if not args.no_kernel_events:
        every = max(1, args.event_every)
        n_seg = max(args.steps, 20 * every)
        step.prepare_events(n_seg, every)
        torch.cuda.synchronize()
        t0 = args.warmup + args.steps
        for t in range(t0, t0 + n_seg):
            step.run(t)
        torch.cuda.synchronize()
        n_ev = len(step.events)
        segs = kernel_times(step.events)
        step.events = None
        fp8.fp8_check_device_status()

    # --- end-to-end: every step copies its X and G in from pinned host memory
    # and reads its result back.  The result read is the step's metric, the
    # three amax values it measured (the quantities the scaling recipe
    # produces each step), as a training loop reads its loss; a second pass
    # reads Y, dX and dW back in full (96 MB a step) and is reported beside
    # it.  Three streams (H2D, compute, D2H) with double-buffered device
    # inputs and outputs let step t's copies overlap steps t-1 / t+1's
    # kernels; the meta state is shared, so the numerics are those of the
    # device-resident loop.  (Three buffers measured slower: 0.68 against
    # 0.58 ms a step with the full read; the host link is the limit.)
    n_host, NB = 4, 2
    xp = [torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).pin_memory() for h in x_host[:n_host]]
    gp = [torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).pin_memory() for h in g_host[:n_host]]
    x_buf = [torch.empty((M, K), dtype=torch.bfloat16, device=dev) for _ in range(NB)]
    g_buf = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(NB)]
    ios = [step.io] + [fp8.LinearStep(M, N, K, device=dev) for _ in range(NB - 1)]
    h2d = x_buf[0].numel() * 2 + g_buf[0].numel() * 2
    e2e_steps = max(3, min(args.steps, 200))
    s_comp = torch.cuda.current_stream()

    def e2e_pass(full: bool):
        """ms per step of e2e_steps steps, and the D2H bytes per step."""
        if full:
            outs = [[torch.empty((M, N), dtype=torch.bfloat16).pin_memory(),
                     torch.empty((M, K), dtype=torch.bfloat16).pin_memory(),
                     torch.empty((N, K), dtype=torch.bfloat16).pin_memory()] for _ in range(NB)]
            srcs = [[io.y, io.dx, io.dw] for io in ios]
        else:
            outs = [[torch.empty(3, dtype=torch.float32).pin_memory()] for _ in range(NB)]
            srcs = [[io.amax] for io in ios]
        d2h = sum(o.numel() * o.element_size() for o in outs[0])
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(NB)]
        ev_used = [torch.cuda.Event() for _ in range(NB)]   # compute done with inputs of slot
        ev_comp = [torch.cuda.Event() for _ in range(NB)]   # outputs of slot written
        ev_read = [torch.cuda.Event() for _ in range(NB)]   # outputs of slot copied out
        for e in ev_used + ev_read:
            e.record(s_comp)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_comp)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        for t in range(e2e_steps):
            b = t % NB
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_used[b])
                x_buf[b].copy_(xp[t % n_host], non_blocking=True)
                g_buf[b].copy_(gp[t % n_host], non_blocking=True)
                ev_in[b].record(s_in)
            s_comp.wait_event(ev_in[b])
            s_comp.wait_event(ev_read[b])
            step.io = ios[b]
            step.run(t, x_buf[b], g_buf[b])
            ev_used[b].record(s_comp)
            ev_comp[b].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                for o, src in zip(outs[b], srcs[b]):
                    o.copy_(src, non_blocking=True)
                ev_read[b].record(s_out)
        s_comp.wait_stream(s_in)
        s_comp.wait_stream(s_out)
        e1.record(s_comp)
        barrier()
        step.io = ios[0]
        return e0.elapsed_time(e1) / e2e_steps, d2h

    ms_e2e_step, d2h = e2e_pass(False)
    ms_e2e_full, d2h_full = e2e_pass(True)

    ms_step = ms_total / args.steps
    ms_step, ms_e2e_step, ms_e2e_full = max_over_ranks([ms_step, ms_e2e_step, ms_e2e_full], dev)
    if rank != 0:
        return None

    peaks = load_peaks()
    fp8_peak = peaks["bf16"] * FP8_PER_BF16
    kernels = {}
    gemm_tflops = None
    if segs is not None:
        # the roofline kernel: the launch carrying dgrad and wgrad (two of the
        # step's three GEMMs)
        gemm_tflops = 2 * GEMM_FLOP / (segs["gemm_dgrad_wgrad"] * 1e-3) / 1e12
        for k, n in (("gemm_fprop", 1), ("gemm_dgrad_wgrad", 2)):
            kernels[k] = {"us": round(segs[k] * 1e3, 2),
                          "tflops": round(n * GEMM_FLOP / (segs[k] * 1e-3) / 1e12, 1)}
        for k, b in QBYTES.items():
            gbs = b / (segs[k] * 1e-3) / 1e9
            kernels[k] = {"us": round(segs[k] * 1e3, 2), "gbs": round(gbs, 1),
                          "frac_hbm": round(gbs / peaks["hbm"], 3),
                          "frac_hbm_nominal_8tbs": round(gbs / 8000.0, 3)}
        for k in ("meta_fwd", "meta_bwd"):
            kernels[k] = {"us": round(segs[k] * 1e3, 2)}
    value = whole_job_tflops(ms_step, world)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 operands, fp32 accumulate, bf16 out",
        "data": "synthetic (seeded normal inputs of the configuration's shapes)",
        "config": headline_config(world),
        "roofline": {"bound": "tensor",
                     "achieved": None if gemm_tflops is None else round(gemm_tflops, 1),
                     "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": None if gemm_tflops is None else round(gemm_tflops / fp8_peak, 3),
                     "traffic": profile_traffic("gemm_fp8_pair_dgrad_wgrad_4096.md"),
                     "kernel": "gemm_f8_pair_kernel<256> carrying dgrad and wgrad (2-SM tcgen05, "
                               "one launch, 2 x 2*4096^3 FLOP)",
                     "peak_source": f"{peaks['src']} bf16 burst {peaks['bf16']} TFLOP/s x 2 (fp8:bf16 nominal)"},
        "kernels": kernels,
        "e2e": {"value": round(whole_job_tflops(ms_e2e_step, world), 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e_step, 4),
                "result_read": "the step's three amax values (its per-step metric)"},
        "e2e_full_outputs": {"value": round(whole_job_tflops(ms_e2e_full, world), 2),
                             "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                             "d2h_bytes_per_step": d2h_full,
                             "ms_per_step": round(ms_e2e_full, 4),
                             "result_read": "Y, dX and dW in full"},
        "gpu_launches": launches,
        "kernel_timing": None if segs is None else
        f"CUDA events at the kernel boundaries of {n_ev} steps (every {max(1, args.event_every)}-th "
        "of a second loop run right after the timed region; an event between two kernels stops "
        "their programmatic overlap, so these steps are not part of the timed region)",
        "clocks": clocks,
    }
    return line


# ---------------------------------------------------------- oracle (CPU) ---

PANEL = 16  # GEMM rows the oracle computes per GEMM for the GPU line's baseline


_SAMPLE_INPUTS = {}


def oracle_sample_step(step_idx: int, w_h, state_meta, rows_q: int = M, panel: int = PANEL):
    """One step of the oracle on a bounded sample: the quantisers on the first
    rows_q rows of X, W and G (the state machine runs on those rows' amaxes)
    and each GEMM on a panel x rows_q block of its output or contraction (the
    sampled operands).  Returns the seconds spent and the seconds
    extrapolated to the full 4096^3 step: quantiser time x 4096/rows_q, GEMM
    time x (4096/panel) x (4096/rows_q)."""
    import oracle
    from oracle import state as ost
    key = (step_idx % N_SETS, rows_q)
    if key not in _SAMPLE_INPUTS:   # the leading rows_q rows of the step's X and G
        _SAMPLE_INPUTS[key] = (
            synth.normal_bf16((rows_q, K), CFG["x_sigma"], CFG["seed"], "x", step_idx % N_SETS),
            synth.normal_bf16((rows_q, N), CFG["g_sigma"], CFG["seed"], "g", step_idx % N_SETS))
    x, g = _SAMPLE_INPUTS[key]
    w = np.ascontiguousarray(w_h[:rows_q])
    st, meta = state_meta
    t0 = time.perf_counter()
    st.step()
    xq, amax_x = oracle.quantize(x, meta.x_scale_inv)
    wq, amax_w = oracle.quantize(w, meta.scale_inv)
    tg0 = time.perf_counter()
    oracle.gemm(xq[:panel], wq, meta.x_scale, meta.scale)            # Y panel
    tg = time.perf_counter() - tg0
    meta.record(amax_w)
    meta.note_x(amax_x)
    gq, amax_g = oracle.quantize(g, meta.g_scale_inv)
    xq2, _ = oracle.quantize(x, meta.x_scale_inv)
    tg0 = time.perf_counter()
    oracle.gemm(np.ascontiguousarray(gq[:panel, :rows_q]), oracle.transpose_u8(wq),
                meta.g_scale, meta.scale)                             # dX panel
    oracle.gemm(np.ascontiguousarray(oracle.transpose_u8(gq)[:panel]), oracle.transpose_u8(xq2),
                meta.g_scale, meta.x_scale)                           # dW panel
    tg += time.perf_counter() - tg0
    meta.note_g(amax_g)
    spent = time.perf_counter() - t0
    full = (spent - tg) * (M / rows_q) + tg * (M / panel) * (M / rows_q)
    return spent, full


def reference_sample_size(total_steps: int, budget_s: float = 90.0):
    """Rows of each tensor the oracle quantises and GEMM panel rows per step,
    sized so total_steps steps take about budget_s seconds of one core: about
    2 ms per sampled row for the four quantisers and 12 us per (panel row x
    sampled row) for the three GEMMs."""
    per_step = budget_s / max(1, total_steps)
    rows = 16
    while rows * 2 <= M and rows * 2 * 2e-3 <= 0.5 * per_step:
        rows *= 2
    panel = int(max(1, min(64, 0.4 * per_step / (rows * 12e-6))))
    return rows, panel


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    import oracle
    from oracle import state as ost
    oracle.build()
    rows_q, panel = reference_sample_size(args.steps + args.warmup)
    w_h = synth.normal_bf16((N, K), CFG["w_sigma"], CFG["seed"], "w")
    st = ost.StepCounter(16)
    meta = st.new_weight()
    for t in range(args.warmup):
        oracle_sample_step(t, w_h, (st, meta), rows_q, panel)
    spent_total, full_total = 0.0, 0.0
    for t in range(args.warmup, args.warmup + args.steps):
        s, f = oracle_sample_step(t, w_h, (st, meta), rows_q, panel)
        spent_total += s
        full_total += f
    ms_step = full_total / args.steps * 1e3
    value = STEP_FLOP / (ms_step * 1e-3) / 1e12
    sample = (f"per step: the 4 quantisers on {rows_q} of 4096 rows of X, W and G, each GEMM "
              f"on a {panel} x {rows_q} block of its output or contraction; quantiser time "
              f"scaled by 4096/{rows_q}, GEMM time by (4096/{panel})(4096/{rows_q})")
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 GEMM on decoded e4m3, fp32 scales", "data": "synthetic",
        "config": headline_config(world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "cpu_seconds": round(spent_total, 2)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def cpu_baseline_for_gpu_line(steps: int = 2):
    """The oracle timed on this host for the GPU line's cpu_baseline field
    (rank 0, one GPU only): a bounded sample of 2 steps (~10-30 s)."""
    import oracle
    from oracle import state as ost
    oracle.build()
    w_h = synth.normal_bf16((N, K), CFG["w_sigma"], CFG["seed"], "w")
    st = ost.StepCounter(16)
    meta = st.new_weight()
    spent_total, full_total = 0.0, 0.0
    for t in range(steps):
        s, f = oracle_sample_step(t, w_h, (st, meta))
        spent_total += s
        full_total += f
    ms_step = full_total / steps * 1e3
    return {"value": round(STEP_FLOP / (ms_step * 1e-3) / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{steps} steps; per step the 4 quantisers over full 4096x4096 tensors and "
                      f"each GEMM on a {PANEL}-row panel, GEMM time extrapolated to M=4096",
            "cpu_seconds": round(spent_total, 2), "ms_per_step_extrapolated": round(ms_step, 1)}



# ------------------------------------------------- the other workloads ---
# `--workload mlp|thd|block|sweep|config1` measures one remaining
# configuration as a line of its own; the default run also carries all of
# them, briefly, in its line's `workloads` object.  Inputs are drawn on the
# device from a seeded torch generator with the configurations' shapes and
# distributions (configuration 1 uses the host generator of the tests);
# parity of the same paths on host-generated inputs is in
# tests/test_gpu_configs.py.

def _timed(torch, fn, steps, warmup):
    for t in range(warmup):
        fn(t)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(steps):
        fn(warmup + t)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps  # ms per step


def _segments(torch, calls, reps):
    """Mean ms of each (name, fn) segment over reps runs of the sequence, with
    an event between consecutive segments (which stops their overlap)."""
    acc = {n: [] for n, _ in calls}
    for _ in range(reps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
        ev[0].record()
        for i, (_, fn) in enumerate(calls):
            fn()
            ev[i + 1].record()
        torch.cuda.synchronize()
        for i, (n, _) in enumerate(calls):
            acc[n].append(ev[i].elapsed_time(ev[i + 1]))
    return {n: statistics.mean(v) for n, v in acc.items()}


def _seeded_normal(torch, shape, sigma, seed, dev, outliers=None):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * sigma
    if outliers is not None:
        p, factor = outliers
        hit = torch.rand(shape, generator=g, device=dev) < p
        x = torch.where(hit, x * factor, x)
    return x.to(torch.bfloat16)


class _DynLinear:
    """fwd + dgrad + wgrad of one projection under current scaling as one
    native call (fp8_linear_step_dynamic): every operand through the
    single-launch dynamic quantiser (q and qt), fprop, then dgrad and wgrad."""

    def __init__(self, fp8, torch, dev, M, N, K, x, w, g):
        self.fp8, self.M, self.N, self.K = fp8, M, N, K
        self.x, self.w, self.g = x, w, g
        self.step = fp8.LinearStep(M, N, K, device=dev)
        self.step.set_inputs(x, w, g)
        self.state = fp8.DynamicStepState(device=dev)

    def run(self):
        self.fp8.fp8_linear_step_dynamic(self.state, self.step)

    def calls(self):
        """The step's launches as the public single calls it is made of (same
        kernels, same workspaces), in segments: X and W quantised, fprop, G
        quantised, dgrad and wgrad in one launch."""
        fp8, io, sc = self.fp8, self.step, self.state.scales
        M, N, K = self.M, self.N, self.K
        n = fp8.fp8_quantize_fused_workspace_bytes() // 4
        ws = [self.state.workspace[i * n:(i + 1) * n] for i in range(3)]

        def quant_xw():
            fp8.fp8_quantize_fused_dynamic(self.x, sc[0:1], sc[1:2], io.xq, io.xqt, io.amax[0:1],
                                           ws[0])
            fp8.fp8_quantize_fused_dynamic(self.w, sc[2:3], sc[3:4], io.wq, io.wqt, io.amax[1:2],
                                           ws[1])
        return [
            ("quant_x_w", quant_xw),
            ("fprop", lambda: fp8.fp8_linear_fprop(io.xq, sc[0:1], io.wq, sc[2:3], M, N, K,
                                                   fp8.DYNAMIC, None, io.y)),
            ("quant_g", lambda: fp8.fp8_quantize_fused_dynamic(self.g, sc[4:5], sc[5:6], io.gq,
                                                               io.gqt, io.amax[2:3], ws[2])),
            ("dgrad_wgrad", lambda: fp8.fp8_linear_dgrad_wgrad(io.gq, io.gqt, sc[4:5], io.wqt,
                                                               sc[2:3], io.xqt, sc[0:1], M, N, K,
                                                               fp8.DYNAMIC, io.dx, io.dw)),
        ]


def _gemm_line(metric_name, value_tflops, ms, flop, workload, extra, peaks):
    fp8_peak = peaks["bf16"] * FP8_PER_BF16
    return {"metric": metric_name, "value": round(value_tflops, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "flop_per_step": flop, "higher_is_better": True,
            "frac_of_fp8_peak": round(value_tflops / fp8_peak, 3),
            "fp8_peak": round(fp8_peak, 1), "data": "synthetic (seeded, on device)",
            "config": {"workload": workload, **extra}}


def _dominant(kernels, peaks):
    """The kernel (segment) with the largest time, with its roofline fraction."""
    name = max(kernels, key=lambda k: kernels[k]["us"])
    d = dict(kernels[name], kernel=name)
    if "tflops" in d:
        d["frac_of_fp8_peak"] = round(d["tflops"] / (peaks["bf16"] * FP8_PER_BF16), 3)
    if "gbs" in d:
        d["frac_hbm"] = round(d["gbs"] / peaks["hbm"], 3)
    return d


def _dyn_kernels(torch, projs, reps):
    """Per-segment µs and TFLOP/s of dynamic-scaling projections, summed over
    the projections of one step."""
    tot = {}
    flops = {"fprop": 0.0, "dgrad_wgrad": 0.0}
    for p in projs:
        seg = _segments(torch, p.calls(), reps)
        for k, v in seg.items():
            tot[k] = tot.get(k, 0.0) + v
        flops["fprop"] += 2.0 * p.M * p.N * p.K
        flops["dgrad_wgrad"] += 4.0 * p.M * p.N * p.K
    out = {}
    for k, ms in tot.items():
        out[k] = {"us": round(ms * 1e3, 1)}
        if k in flops:
            out[k]["tflops"] = round(flops[k] / (ms * 1e-3) / 1e12, 1)
    return out


def workload_mlp(args, steps=None, warmup=None):
    import torch
    import scaled_linear_layers_gb300 as fp8
    c = synth.CONFIG3
    dev = torch.device("cuda", 0)
    M, H, F = c["M"], c["hidden"], c["ffn"]
    projs = []
    for i, (K, N) in enumerate(((H, 2 * F), (F, H))):
        x = _seeded_normal(torch, (M, K), c["x_sigma"], 10 * i + 1, dev)
        w = _seeded_normal(torch, (N, K), c["w_sigma"], 10 * i + 2, dev)
        g = _seeded_normal(torch, (M, N), c["g_sigma"], 10 * i + 3, dev)
        projs.append(_DynLinear(fp8, torch, dev, M, N, K, x, w, g))
    flop = sum(6.0 * p.M * p.N * p.K for p in projs)
    ms = _timed(torch, lambda t: [p.run() for p in projs], steps or args.steps,
                warmup or args.warmup)
    kernels = _dyn_kernels(torch, projs, 3)
    fp8.fp8_check_device_status()
    peaks = load_peaks()
    line = _gemm_line(METRIC, flop / (ms * 1e-3) / 1e12, ms, flop,
                      "transformer MLP block, tokens 16384, hidden 4096, FFN 14336 (gate/up "
                      "4096->28672, down 14336->4096), dynamic scaling, fwd+dgrad+wgrad",
                      {"M": M, "hidden": H, "ffn": F, "recipe": "dynamic"}, peaks)
    line["kernels"] = kernels
    line["dominant_kernel"] = _dominant(kernels, peaks)
    return line


def workload_thd(args, steps=None, warmup=None):
    import torch
    import scaled_linear_layers_gb300 as fp8
    c = synth.CONFIG4
    dev = torch.device("cuda", 0)
    lengths = synth.thd_lengths(c["seed"], c["n_seq"], c["lo"], c["hi"])
    T = int(lengths.sum())
    Tp = fp8.fp8_padded_rows(T, c["multiple"])
    K, N = c["K"], c["N"]
    x = _seeded_normal(torch, (T, K), c["x_sigma"], 41, dev)
    w = _seeded_normal(torch, (N, K), c["w_sigma"], 42, dev)
    g = _seeded_normal(torch, (Tp, N), c["g_sigma"], 43, dev)
    g[T:] = 0
    xp = torch.empty((Tp, K), dtype=torch.bfloat16, device=dev)
    lin = _DynLinear(fp8, torch, dev, Tp, N, K, xp, w, g)

    def step(t):
        fp8.fp8_pad_tokens(x, c["multiple"], xp)
        lin.run()
    flop = 6.0 * Tp * N * K
    ms = _timed(torch, step, steps or args.steps, warmup or args.warmup)
    pad = _segments(torch, [("pad", lambda: fp8.fp8_pad_tokens(x, c["multiple"], xp))], 3)
    kernels = _dyn_kernels(torch, [lin], 3)
    kernels["pad"] = {"us": round(pad["pad"] * 1e3, 1),
                      "gbs": round(4.0 * T * K / (pad["pad"] * 1e-3) / 1e9, 1)}
    fp8.fp8_check_device_status()
    peaks = load_peaks()
    line = _gemm_line(METRIC, flop / (ms * 1e-3) / 1e12, ms, flop,
                      "packed THD batch, 64 sequences of 128..4096 tokens, zero-padded to a "
                      "multiple of 16, linear 4096->4096, dynamic scaling, pad + fwd+dgrad+wgrad",
                      {"tokens": T, "padded_tokens": Tp, "K": K, "N": N, "recipe": "dynamic"},
                      peaks)
    line["kernels"] = kernels
    line["dominant_kernel"] = _dominant(kernels, peaks)
    return line


def workload_block(args, steps=None, warmup=None):
    import torch
    import scaled_linear_layers_gb300 as fp8
    c = synth.CONFIG5
    dev = torch.device("cuda", 0)
    M, K, N = c["M"], c["K"], c["N"]
    if getattr(args, "block_shape", None):  # a smaller case of the same recipe (profiling)
        M, N, K = (int(v) for v in args.block_shape.split(","))
    out = (c["p"], c["factor"])
    x = _seeded_normal(torch, (M, K), c["sigma"], 51, dev, out)
    w = _seeded_normal(torch, (N, K), c["sigma"], 52, dev, out)
    g = _seeded_normal(torch, (M, N), c["sigma"], 53, dev, out)
    u8 = dict(dtype=torch.uint8, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    xq, xqt, wq, wqt, gq, gqt = (torch.empty((M, K), **u8), torch.empty((K, M), **u8),
                                 torch.empty((N, K), **u8), torch.empty((K, N), **u8),
                                 torch.empty((M, N), **u8), torch.empty((N, M), **u8))
    xs, xsi, xst, xsit = (torch.empty((M, K // 128), **f32), torch.empty((M, K // 128), **f32),
                          torch.empty((M // 128, K), **f32), torch.empty((M // 128, K), **f32))
    ws, wsi = torch.empty((N // 128, K // 128), **f32), torch.empty((N // 128, K // 128), **f32)
    gs, gsi, gst, gsit = (torch.empty((M, N // 128), **f32), torch.empty((M, N // 128), **f32),
                          torch.empty((M // 128, N), **f32), torch.empty((M // 128, N), **f32))
    y, dx, dw = (torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                 torch.empty((M, K), dtype=torch.bfloat16, device=dev),
                 torch.empty((N, K), dtype=torch.bfloat16, device=dev))

    def quant():
        fp8.fp8_quantize_transpose(x, fp8.BLOCK, xs, xsi, xq, xqt, xst, xsit)
        fp8.fp8_quantize_transpose(w, fp8.BLOCK_2D, ws, wsi, wq, wqt)
        fp8.fp8_quantize_transpose(g, fp8.BLOCK, gs, gsi, gq, gqt, gst, gsit)
    calls = [
        ("quant_block_x_w_g", quant),
        ("fprop", lambda: fp8.fp8_linear_fprop(xq, xs, wq, ws, M, N, K, fp8.BLOCK, None, y)),
        ("dgrad", lambda: fp8.fp8_linear_dgrad(gq, gs, wqt, ws, M, N, K, fp8.BLOCK, dx)),
        ("wgrad", lambda: fp8.fp8_linear_wgrad(gqt, gst, xqt, xst, M, N, K, fp8.BLOCK, dw)),
    ]
    flop = 6.0 * M * N * K
    ms = _timed(torch, lambda t: [fn() for _, fn in calls], steps or args.steps,
                warmup or args.warmup)
    seg = _segments(torch, calls, 3)
    fp8.fp8_check_device_status()
    peaks = load_peaks()
    line = _gemm_line(METRIC, flop / (ms * 1e-3) / 1e12, ms, flop,
                      "block-scaled recipe (1x128 activation/gradient tiles, 128x128 weight "
                      f"tiles), M={M}, N={N}, K={K}, 1% outliers x50, fwd+dgrad+wgrad",
                      {"M": M, "N": N, "K": K, "recipe": "block"}, peaks)
    gflop = 2.0 * M * N * K
    qbytes = 4 * M * K + 4 * N * K + 4 * M * N + 16 * (M * K + M * N) // 128 + 8 * (N * K) // (128 * 128)
    line["kernels"] = {k: {"us": round(seg[k] * 1e3, 1),
                           "tflops": round(gflop / (seg[k] * 1e-3) / 1e12, 1)}
                       for k in ("fprop", "dgrad", "wgrad")}
    qs = seg["quant_block_x_w_g"]
    line["kernels"]["quant_block_x_w_g"] = {"us": round(qs * 1e3, 1),
                                            "gbs": round(qbytes / (qs * 1e-3) / 1e9, 1)}
    line["dominant_kernel"] = _dominant(line["kernels"], peaks)
    return line


def _graph_time(torch, fn, reps=20):
    """Seconds per call of fn, replayed from a CUDA graph of `reps` calls (no
    host gaps); plain stream launches where a launch form cannot be captured."""
    try:
        g = torch.cuda.CUDAGraph()
        fn(0)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for i in range(reps):
                fn(i)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e-3, "graph"
    except Exception:  # a launch form the capture does not take: time it plainly
        torch.cuda.synchronize()
        return _timed(torch, fn, reps, 3) * 1e-3, "stream"


def workload_sweep(args, lgs=range(20, 31, 2), multi=True, only=None):
    """Quantise-only sweep, n = 2^20 .. 2^30 bf16 elements ([n/4096, 4096]),
    each kernel replayed from a CUDA graph of 20 launches (no host gaps)."""
    import torch
    import scaled_linear_layers_gb300 as fp8
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    rows_out = []
    for lg in lgs:
        n = 1 << lg
        R, C = n // 4096, 4096
        nbuf = 2 if n >= (1 << 26) else 8
        xs = [_seeded_normal(torch, (R, C), 1.0, 60 + i, dev) for i in range(nbuf)]
        q = torch.empty((R, C), dtype=torch.uint8, device=dev)
        qt = torch.empty((C, R), dtype=torch.uint8, device=dev)
        sc = torch.ones(8, dtype=torch.float32, device=dev)
        bs = torch.empty((R, C // 128), dtype=torch.float32, device=dev)
        bsi = torch.empty((R, C // 128), dtype=torch.float32, device=dev)
        ws = torch.zeros(fp8.fp8_quantize_fused_workspace_bytes() // 4, dtype=torch.int32, device=dev)
        dbias = torch.empty(C, dtype=torch.bfloat16, device=dev)
        dws = torch.empty(fp8.fp8_dbias_workspace_bytes(R, C) // 4, dtype=torch.float32, device=dev)
        s, si, a = sc[0:1], sc[1:2], sc[2:3]
        si.fill_(100.0)
        cases = {
            "amax": (2, lambda i: fp8.fp8_amax(xs[i % nbuf], a)),
            "quantize_delayed": (3, lambda i: fp8.fp8_quantize(xs[i % nbuf], fp8.DELAYED, None, si, q, a)),
            "quantize_dynamic_2pass": (5, lambda i: fp8.fp8_quantize(xs[i % nbuf], fp8.DYNAMIC, s, sc[3:4], q, a)),
            "quantize_dynamic_fused": (3, lambda i: fp8.fp8_quantize_fused_dynamic(xs[i % nbuf], s, sc[3:4], q, None, a, ws)),
            "cast_transpose_delayed": (4, lambda i: fp8.fp8_quantize_transpose(xs[i % nbuf], fp8.DELAYED, None, si, q, qt, amax_out=a)),
            # the same plus the bias gradient (column sums) in the same read
            "cast_transpose_dbias": (4, lambda i: fp8.fp8_quantize_transpose_dbias(xs[i % nbuf], fp8.DELAYED, None, si, q, qt, dbias, dws, amax_out=a)),
            "block_1x128": (3, lambda i: fp8.fp8_quantize(xs[i % nbuf], fp8.BLOCK, bs, bsi, q, None)),
        }
        row = {"n": n}
        for name, (bpe, fn) in cases.items():
            if only is not None and name not in only:
                continue
            t, mode = _graph_time(torch, fn)
            gbs = bpe * n / t / 1e9
            row[name] = {"us": round(t * 1e6, 2), "gbs": round(gbs, 1),
                         "frac_hbm": round(gbs / peaks["hbm"], 3),
                         "frac_hbm_nominal_8tbs": round(gbs / 8000.0, 3), "timing": mode}
        rows_out.append(row)
        del xs
        torch.cuda.empty_cache()
    line = {"metric": "quantize GB/s (algorithmic bytes) vs HBM",
            "value": max(r["cast_transpose_delayed"]["gbs"] for r in rows_out
                         if "cast_transpose_delayed" in r),
            "unit": "GB/s", "higher_is_better": True, "data": "synthetic (seeded, on device)",
            "config": {"workload": "quantise-only sweep, 2^20..2^30 bf16 elements, [n/4096, 4096]"},
            "hbm_peak_measured": peaks["hbm"], "sweep": rows_out}
    if not multi:
        return line
    # many weights in one pass: the MLP block's two weights (gate/up
    # [28672, 4096], down [4096, 14336]) plus 64 [1024, 1024] weights
    ws_multi = [_seeded_normal(torch, (28672, 4096), 0.02, 70, dev),
                _seeded_normal(torch, (4096, 14336), 0.02, 71, dev)] + \
        [_seeded_normal(torch, (1024, 1024), 0.02, 72 + i, dev) for i in range(64)]
    nm = len(ws_multi)
    am, sm, sim = (torch.empty(nm, dtype=torch.float32, device=dev) for _ in range(3))
    ms = _timed(torch, lambda t: fp8.fp8_multi_amax_scales(ws_multi, am, sm, sim), 20, 3)
    nbytes = 2 * sum(w.numel() for w in ws_multi)
    line["multi_amax_scales"] = {"tensors": nm, "bytes": nbytes, "us": round(ms * 1e3, 2),
                                 "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                                 "frac_hbm": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm"], 3)}
    del ws_multi
    fp8.fp8_check_device_status()
    return line


def workload_config1(args, iters=1000):
    """Configuration 1, the latency case: X [64,256] ~N(0,1), W [256,256]
    ~N(0,0.02), seed 0, current scaling, fprop.  Two paths through the public
    API: one launch (fp8_linear_fprop_dynamic_small: amaxes, scales, casts and
    the GEMM in one CTA) and three launches (the single-launch dynamic
    quantiser on X and on W, then fp8_linear_fprop).  For each, the median µs
    per iteration over `iters` iterations bracketed by events (eager: host
    launch overhead included) and the µs per iteration of a CUDA graph of the
    iteration's launches replayed back to back (device time).  A bf16
    torch.matmul (cuBLAS) of the same shape is timed the same way as context:
    the pages report FP8 slower than bf16 on small matmuls."""
    import torch
    import scaled_linear_layers_gb300 as fp8
    c = synth.CONFIG1
    dev = torch.device("cuda", 0)
    Mc, Kc, Nc = c["M"], c["K"], c["N"]

    def to_dev(h):
        return torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)
    x = to_dev(synth.normal_bf16((Mc, Kc), c["x_sigma"], c["seed"], "x"))
    w = to_dev(synth.normal_bf16((Nc, Kc), c["w_sigma"], c["seed"], "w"))
    f32 = dict(dtype=torch.float32, device=dev)
    sc = torch.empty(6, **f32)
    sc1 = torch.empty(4, **f32)
    xq = torch.empty((Mc, Kc), dtype=torch.uint8, device=dev)
    wq = torch.empty((Nc, Kc), dtype=torch.uint8, device=dev)
    y = torch.empty((Mc, Nc), dtype=torch.bfloat16, device=dev)
    y1 = torch.empty((Mc, Nc), dtype=torch.bfloat16, device=dev)
    n = fp8.fp8_quantize_fused_workspace_bytes() // 4
    wsp = torch.zeros(2 * n, dtype=torch.int32, device=dev)

    def run3(_=0):
        fp8.fp8_quantize_fused_dynamic(x, sc[0:1], sc[1:2], xq, None, sc[4:5], wsp[:n])
        fp8.fp8_quantize_fused_dynamic(w, sc[2:3], sc[3:4], wq, None, sc[5:6], wsp[n:])
        fp8.fp8_linear_fprop(xq, sc[0:1], wq, sc[2:3], Mc, Nc, Kc, fp8.DYNAMIC, None, y)

    def run1(_=0):
        fp8.fp8_linear_fprop_dynamic_small(x, w, sc1, y1)

    def median_us(fn):
        for _ in range(20):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(iters)]
        for a, b in ev:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3
    eager1 = median_us(run1)
    t1, mode1 = _graph_time(torch, run1, reps=100)
    eager3 = median_us(run3)
    t3, mode3 = _graph_time(torch, run3, reps=100)
    fp8.fp8_check_device_status()
    same = bool(torch.equal(y, y1))
    bf16 = median_us(lambda: torch.matmul(x, w.t()))
    yb = torch.empty((Mc, Nc), dtype=torch.bfloat16, device=dev)
    tb, _ = _graph_time(torch, lambda _=0: torch.matmul(x, w.t(), out=yb), reps=100)
    flop = 2.0 * Mc * Nc * Kc
    return {"metric": "latency of current-scaling fprop (quantise X, W + GEMM)",
            "value": round(eager1, 2), "unit": "us", "higher_is_better": False,
            "config": {"workload": "single FP8 linear fprop, dynamic tensorwise scaling, "
                                   "X [64,256], W [256,256], seed 0", "M": Mc, "N": Nc, "K": Kc},
            "iterations": iters,
            "one_launch": {"median_us_eager": round(eager1, 2),
                           "us_per_iteration_graph": round(t1 * 1e6, 2), "graph_timing": mode1,
                           "tflops_graph": round(flop / t1 / 1e12, 3)},
            "three_launches": {"median_us_eager": round(eager3, 2),
                               "us_per_iteration_graph": round(t3 * 1e6, 2),
                               "graph_timing": mode3},
            "same_output_bits": same,
            "bf16_torch_matmul_median_us": round(bf16, 2),
            "bf16_torch_matmul_us_per_iteration_graph": round(tb * 1e6, 2),
            "note": "latency-bound: roofline fractions are not meaningful at this size"}


def workloads_summary(args):
    """Every configuration besides the headline one, briefly, for the default
    line (rank 0, one GPU): configuration 1's latency, the MLP block, the
    packed THD batch and the block recipe (whole-step TFLOP/s and the
    dominant kernel), and the 2^30-element quantisers."""
    import torch
    out = {}
    for key, fn in (("config1_fprop_64x256x256", lambda: workload_config1(args)),
                    ("config3_mlp_16384x4096x14336", lambda: workload_mlp(args, 5, 3)),
                    ("config4_thd_64seq_4096", lambda: workload_thd(args, 5, 3)),
                    ("config5_block_32768x8192x8192", lambda: workload_block(args, 5, 3)),
                    ("quantize_2^30", lambda: workload_sweep(
                        args, lgs=[30], multi=False,
                        only=("amax", "quantize_delayed", "cast_transpose_delayed",
                              "block_1x128")))):
        with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
            first = clk.mark()
            line = fn()
            clocks = clk.summary(first)
        for k in ("metric", "higher_is_better", "data", "fp8_peak", "hbm_peak_measured"):
            line.pop(k, None)
        line["clocks"] = clocks
        out[key] = line
        torch.cuda.empty_cache()
    if "quantize_2^30" in out:
        q = out["quantize_2^30"]
        q["sweep"] = q["sweep"][0]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kernel-events", action="store_true",
                    help="time the step without per-kernel events (no per-kernel breakdown)")
    ap.add_argument("--event-every", type=int, default=10,
                    help="the per-kernel segments come from every n-th step of a second loop "
                         "(as long as the timed one, at least 20 n steps) run after the timed "
                         "region, with events at every kernel boundary: an event between two "
                         "kernels stops the second from overlapping the first")
    ap.add_argument("--workload", default="linear4096",
                    choices=["linear4096", "mlp", "thd", "block", "sweep", "config1"])
    ap.add_argument("--no-workloads", action="store_true",
                    help="leave the other configurations out of the default line")
    ap.add_argument("--block-shape", default=None, metavar="M,N,K",
                    help="--workload block on another shape (multiples of 128), e.g. for a "
                         "profiler capture of a small case")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.workload != "linear4096":
        if rank != 0:
            return
        fn = {"mlp": workload_mlp, "thd": workload_thd, "block": workload_block,
              "sweep": workload_sweep, "config1": workload_config1}[args.workload]
        print(json.dumps(fn(args)), flush=True)
        return
    if args.impl == "reference":
        line = reference_arm(args, rank, world)
    else:
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            # before the first CUDA call, so no process state is shared with it
            cpu = cpu_baseline_for_gpu_line()
        line = gpu_arm(args, rank, world)
        if line is not None:
            line["cpu_baseline"] = cpu
            if world == 1 and not args.no_workloads:
                line["workloads"] = workloads_summary(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
