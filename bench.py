#!/usr/bin/env python
"""Benchmark of the MACaQ W4A4 (MXFP4) linear layer on B300.

One step = the whole online hot path on one batch: the activation transform
(balance, 32-channel block Hadamard, MXFP4 encode; one CUDA kernel) followed by
the block-scaled MXFP4 GEMM (one tcgen05 kernel) -- up to 6 token rows one
kernel does both (``macaq_linear``: the transform inside the few-rows GEMM) --
i.e. ``macaq_linear`` on the
prefill MLP down-projection M=8192 tokens, K=25600, N=5120 (the largest
single-GPU configuration; ``--config`` picks another workload).  Weights are
prepared once, outside the timed region (balance from a 512-row calibration
batch, fold, quantise).

Reported (one JSON line on rank 0):
  value          W4A4 linear TFLOP/s (2*M*N*K per step / device time), whole job
  roofline       the GEMM kernel against the dense MXFP4 tensor peak (measured
                 bf16 peak x the nominal fp4/bf16 ratio 13.5/2.25)
  act_quant      the transform kernel's GB/s against measured HBM bandwidth
  e2e            the same metric through the C ABI with pinned host buffers,
                 host->device of X and device->host of Y inside the timing
                 every step; the copies of neighbouring steps overlap the
                 compute (two copy streams, rotating buffer slots); the fully
                 serialised figure is reported beside it
  cpu_baseline   the CPU oracle on a bounded row sample of the same workload
  per_config     the same device timing (value, GEMM roofline, transform GB/s)
                 for the prefill attention projection (N=5120 and fused QKV
                 N=7168), decode M=1/8/16 and the routed MoE layer

Timing: W warm-up steps, then exactly K steps between a barrier and a device
synchronise, CUDA events on the launching stream around every kernel; inputs
rotate over enough copies that each step's working set was evicted from L2
(126 MB) by the steps in between.  Multi-GPU: one independent replica per rank
(rows are independent; no collective on the data path), max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FP4_OVER_BF16 = 13.5 / 2.25      # nominal dense fp4 : bf16 tensor throughput on B300
L2_BYTES = 126 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class _NvmlCtypes:
    """Minimal NVML binding through ctypes (the driver's libnvidia-ml)."""

    def __init__(self, bus_id):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        rc = 1
        if bus_id:
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(0), ctypes.byref(self.h))
        if rc != 0:
            raise RuntimeError("no NVML device handle")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_clock(self):
        c = self.ct.c_uint()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(c))  # NVML_CLOCK_SM
        return c.value

    def max_sm_clock(self):
        c = self.ct.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.ct.byref(c))
        return c.value

    def mem_clock(self):
        c = self.ct.c_uint()
        self.lib.nvmlDeviceGetClockInfo(self.h, 2, self.ct.byref(c))  # NVML_CLOCK_MEM
        return c.value

    def max_mem_clock(self):
        c = self.ct.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 2, self.ct.byref(c))
        return c.value

    def reasons(self):
        r = self.ct.c_ulonglong()
        self._reasons(self.h, self.ct.byref(r))
        return r.value


class ClockSampler:
    """Samples SM and memory clocks and clock-event (throttle) reasons through NVML
    while running (read-only queries: no setting of the GPU is changed)."""

    REASONS = {
        0x0000000000000001: "gpu_idle", 0x0000000000000002: "applications_clocks_setting",
        0x0000000000000004: "sw_power_cap", 0x0000000000000008: "hw_slowdown",
        0x0000000000000010: "sync_boost", 0x0000000000000020: "sw_thermal_slowdown",
        0x0000000000000040: "hw_thermal_slowdown", 0x0000000000000080: "hw_power_brake_slowdown",
        0x0000000000000100: "display_clock_setting",
    }

    def __init__(self, bus_id: str | None, period_s: float = 0.001):
        self.samples = []
        self.mem_samples = []
        self.reasons = set()
        self.period = period_s
        self.ok = False
        self.err = ""
        try:
            self.nv = _NvmlCtypes(bus_id)
            self.max_mhz = self.nv.max_sm_clock()
            self.max_mem_mhz = self.nv.max_mem_clock()
            self.ok = True
        except Exception as e:  # noqa: BLE001 - clocks are then reported as unavailable
            self.err = str(e)
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.sm_clock())
                self.mem_samples.append(self.nv.mem_clock())
                r = self.nv.reasons()
                for bit, name in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:  # noqa: BLE001
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self._t is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": self.err}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons - {"gpu_idle"}),
                "mem_mhz": statistics.median(self.mem_samples) if self.mem_samples else None,
                "mem_max_mhz": self.max_mem_mhz, "samples": len(self.samples)}


def pci_bus_id(dev) -> str | None:
    try:
        import torch
        p = torch.cuda.get_device_properties(dev)
        return "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except Exception:  # noqa: BLE001
        return None


# ----------------------------------------------------------------- oracle leg

def oracle_linear_rate(d, rows: int, target_s: float):
    """Time the CPU oracle (transform + MXFP4 of sampled rows, fp64 GEMM against
    the prepared weight) and return (TFLOP/s, rows used, seconds, threads)."""
    import numpy as np
    import torch

    import oracle

    wl = d["workload"]
    s, inv = oracle.balance_scales(d["X_calib"], d["W"])
    cw, sw = oracle.quantize(d["W"], s)
    deq_w = oracle.dequant(cw, sw)          # weight preparation: outside the timing

    def run(n):
        X = d["X"][:n] if "X" in d else d["GU"][:n].contiguous()
        t0 = time.perf_counter()
        if "X" not in d:            # gated input: the SwiGLU step first
            X = oracle.silu_mul(X)
        ca, sa = oracle.quantize(X, inv)
        Y = oracle.gemm_ref(oracle.dequant(ca, sa), deq_w)
        torch.from_numpy(Y).to(torch.bfloat16)
        return time.perf_counter() - t0

    run(min(rows, 4))
    n = max(1, min(rows, 16))
    dt = run(n)
    while dt < target_s * 0.5 and n < min(rows, wl.M):
        n = min(wl.M, max(n + 1, int(n * min(8.0, target_s / max(dt, 1e-3)))))
        dt = run(n)
    flops = 2.0 * n * wl.N * wl.K
    threads = max(oracle.num_threads(), os.cpu_count() or 1)
    return flops / dt / 1e12, n, dt, threads


def reference_arm_moe(args, rank: int, world: int):
    """--impl reference on the MoE workload: each step runs the oracle's gate+up
    projection (transform, MXFP4, fp64 GEMM) on the rows routed to one expert."""
    if rank != 0:
        return 0
    import workloads
    import oracle

    config = config or args.config
    d = workloads.make_moe(workloads.MOE if config == "moe" else workloads.MOE_SMALL)
    wl = d["workload"]
    r, cr = d["routing"], d["calib_routing"]
    off, coff = r["offsets"].numpy(), cr["offsets"].numpy()
    prepared = {}

    def prep(e):
        if e not in prepared:
            xc = d["X_calib"][cr["row_src"][coff[e]:coff[e + 1]].long()]
            s, inv = oracle.balance_scales(xc, d["W_gu"][e])
            cw, sw = oracle.quantize(d["W_gu"][e], s)
            prepared[e] = (inv, oracle.dequant(cw, sw))
        return prepared[e]

    n_steps = args.warmup + args.steps
    for i in range(n_steps):
        prep(i % wl.E)            # weight preparation: outside the timing

    def step(i):
        e = i % wl.E
        inv, deq_w = prep(e)
        X = d["X"][r["row_src"][off[e]:off[e + 1]].long()]
        ca, sa = oracle.quantize(X, inv)
        oracle.gemm_ref(oracle.dequant(ca, sa), deq_w)
        return 2.0 * X.shape[0] * 2 * wl.F * wl.K

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    flops = sum(step(args.warmup + i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    threads = max(oracle.num_threads(), os.cpu_count() or 1)
    sample = "gate+up projection of the rows routed to one expert per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (fp32 transform)", "data": "synthetic",
        "config": moe_workload_config(wl),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def reference_arm(args, rank: int, world: int):
    """--impl reference: the CPU oracle as it stands, rank 0 only."""
    if args.config.startswith("moe"):
        return reference_arm_moe(args, rank, world)
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401
    import workloads
    import oracle

    d = workloads.make_dense(args.config)
    wl = d["workload"]
    s, inv = oracle.balance_scales(d["X_calib"], d["W"])
    cw, sw = oracle.quantize(d["W"], s)
    deq_w = oracle.dequant(cw, sw)
    # size one step (a row sample) so the whole run takes about two minutes
    t0 = time.perf_counter()
    ca, sa = oracle.quantize(d["X"][:8], inv)
    oracle.gemm_ref(oracle.dequant(ca, sa), deq_w)
    per_row = (time.perf_counter() - t0) / 8
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(wl.M, budget / max(per_row, 1e-6))))

    def step(i):
        r0 = (i * rows) % max(1, wl.M - rows + 1)
        ca, sa = oracle.quantize(d["X"][r0:r0 + rows], inv)
        oracle.gemm_ref(oracle.dequant(ca, sa), deq_w)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * wl.N * wl.K * args.steps
    value = flops / dt / 1e12
    threads = max(oracle.num_threads(), os.cpu_count() or 1)
    sample = f"{rows} of {wl.M} rows per step (full N={wl.N}, K={wl.K})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (fp32 transform)", "data": "synthetic",
        "config": dict(workload_config(wl), hadamard_block=32),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


METRIC = "W4A4 linear TFLOPS + act-quant GB/s, as fraction of B300 FP4/HBM roofline"


def workload_config(wl):
    return {"workload": f"{wl.name}: M={wl.M} tokens, K={wl.K}, N={wl.N}, bf16 in/out, "
                        f"MXFP4 W4A4",
            "M": wl.M, "K": wl.K, "N": wl.N, "calib_rows": wl.calib_rows,
            "l2": "inputs rotate over copies larger than L2 between steps"}


def gemm_kernel_name(M: int) -> str:
    """The GEMM kernel macaq_w4a4_gemm launches for M token rows."""
    return "gemm_mxf4_skinny_kernel" if M <= 64 else "gemm_mxf4_pair_kernel"


FUSED_LINEAR_MAX_ROWS = 6    # macaq_linear: one launch, the transform inside the few-rows GEMM
FUSED_LINEAR_KERNEL = "gemm_mxf4_skinny_kernel<16, 5, true>"


# ------------------------------------------------------------------- GPU arm

def gpu_arm(args, rank: int, world: int, config: str | None = None, light: bool = False):
    """The dense layer's line (rank 0; None elsewhere).  light: device timing
    only (no end-to-end leg, no CPU baseline), for the per-configuration table."""
    import torch
    import torch.distributed as dist

    import workloads
    import w4a4_mxfp4_quantized_02_b300 as mq

    config = config or args.config
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    mq.lib()
    peaks = load_peaks()
    fused = args.fused_swiglu and not light
    if fused and (workloads.DENSE[config].act != "swiglu" or args.hadamard_block != 32):
        raise SystemExit("--fused-swiglu needs a SwiGLU-input workload (down) and --hadamard-block 32")
    d = workloads.make_dense_gated(config) if fused else workloads.make_dense(config)
    wl = d["workload"]
    M, N, K = wl.M, wl.N, wl.K
    stream = torch.cuda.current_stream()
    xcols = 2 * K if fused else K   # the step's input: the gate|up matrix when fused

    # offline preparation (not timed): calibration, fold, weight quantisation
    Xc = d["X_calib"].to(dev)
    W = d["W"].to(dev)
    s, inv = mq.macaq_balance_scales(Xc, W)
    hb = args.hadamard_block
    w_codes, w_scales = mq.macaq_quant_weight_hb(W, s, hb)
    del W, Xc

    # up to 6 token rows (Hadamard block 32) the layer is one launch
    # (macaq_linear: the transform inside the few-rows GEMM)
    one_launch = not fused and hb == 32 and M <= FUSED_LINEAR_MAX_ROWS
    ws_bytes = mq.macaq_linear_workspace_bytes(M, K)
    step_bytes = M * xcols * 2 + ws_bytes * 2 + w_codes.numel() + w_scales.numel() + M * N * 2
    nsets = max(2, math.ceil(2.5 * L2_BYTES / step_bytes) + 1)
    X0 = (d["GU"] if fused else d["X"]).to(dev)
    sets = []
    for i in range(nsets):
        sets.append({
            "X": X0.clone() if i else X0,
            "wc": w_codes.clone() if i else w_codes,
            "ws": w_scales.clone() if i else w_scales,
            "Y": torch.empty(M, N, dtype=torch.bfloat16, device=dev),
            "a_codes": torch.empty(M, K // 2, dtype=torch.uint8, device=dev),
            "a_scales": torch.empty(mq.macaq_scale_bytes(M, K), dtype=torch.uint8, device=dev),
            "lws": torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev),
        })

    def linear_part(i):
        b = sets[i % nsets]
        mq.macaq_linear(b["X"], inv, b["wc"], b["ws"], N, Y=b["Y"], workspace=b["lws"])

    def quant_part(i):
        b = sets[i % nsets]
        if fused:
            mq.macaq_quant_act_silu(b["X"], inv, b["a_codes"], b["a_scales"])
        else:
            mq.macaq_quant_act_hb(b["X"], inv, hb, b["a_codes"], b["a_scales"])

    def gemm_part(i):
        b = sets[i % nsets]
        mq.macaq_w4a4_gemm(b["a_codes"], b["a_scales"], b["wc"], b["ws"], M, N, K, Y=b["Y"])

    # per-kernel timing (the eager kernel-group batches) needs the kernels as
    # separate calls; the other steps are the layer as a user calls it
    # (macaq_linear, Hadamard block 32: its GEMM may load its first weight
    # stages while its own transform still runs)
    parts = [linear_part] if one_launch else [quant_part, gemm_part]
    layer_call = not fused and hb == 32

    def step(i):
        if layer_call:
            linear_part(i)
            return
        for part in parts:
            part(i)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    status = mq.macaq_check_device_error()
    if status != 0:
        raise RuntimeError(f"device error during warm-up: {mq.macaq_status_string(status)}")
    chunk = nsets * max(1, math.ceil(8 / nsets))
    graph = None if args.no_graphs else capture_graph(lambda: [step(i) for i in range(chunk)])
    plan = StepPlan(args.steps, args.kernel_events_every, chunk if graph is not None else 0)
    batches = KernelBatches(plan.eager_steps, min(nsets, 4), len(parts))
    batches.calibrate(parts, stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(pci_bus_id(dev))
    with sampler:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        h0 = time.perf_counter()
        batches.run(parts, stream, graph, plan.replays)
        host_enqueue_s = time.perf_counter() - h0
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end) - batches.padding_ms()
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    if one_launch:
        (gemm_avg,) = batches.per_launch_ms()
        quant_avg = None
    else:
        quant_avg, gemm_avg = batches.per_launch_ms()
    status = mq.macaq_check_device_error()
    if status != 0:
        raise RuntimeError(f"device error in the timed region: {mq.macaq_status_string(status)}")

    flops = 2.0 * M * N * K
    value = flops * args.steps * world / (elapsed_ms * 1e-3) / 1e12
    gemm_tflops = flops / (gemm_avg * 1e-3) / 1e12
    quant_bytes = M * xcols * 2 + M * K // 2 + M * K // 32
    quant_gbs = None if quant_avg is None else quant_bytes / (quant_avg * 1e-3) / 1e9
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16

    e2e_value = e2e_ms = e2e_serial_ms = None
    nslot = min(3, nsets)
    if not light:
        # end to end through the C ABI: pinned host X in, pinned host Y out
        def layer(b):
            if fused:
                mq.macaq_quant_act_silu(b["X"], inv, b["a_codes"], b["a_scales"])
                mq.macaq_w4a4_gemm(b["a_codes"], b["a_scales"], b["wc"], b["ws"], M, N, K, Y=b["Y"])
            elif hb == 32:
                mq.macaq_linear(b["X"], inv, b["wc"], b["ws"], N, Y=b["Y"])
            else:
                mq.macaq_quant_act_hb(b["X"], inv, hb, b["a_codes"], b["a_scales"])
                mq.macaq_w4a4_gemm(b["a_codes"], b["a_scales"], b["wc"], b["ws"], M, N, K, Y=b["Y"])

        e2e_steps = max(3, min(args.steps, 50))
        Xh = (d["GU"] if fused else d["X"]).pin_memory()
        Yh = [torch.empty(M, N, dtype=torch.bfloat16).pin_memory() for _ in range(nslot)]
        b = sets[0]
        for _ in range(2):
            b["X"].copy_(Xh, non_blocking=True)
            layer(b)
            Yh[0].copy_(b["Y"], non_blocking=True)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            b["X"].copy_(Xh, non_blocking=True)
            layer(b)
            Yh[0].copy_(b["Y"], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_serial_ms = e0.elapsed_time(e1) / e2e_steps
        e2e_ms = e2e_pipelined(stream, e2e_steps, nslot,
                               lambda k: sets[k]["X"].copy_(Xh, non_blocking=True),
                               lambda k: layer(sets[k]),
                               lambda k: Yh[k].copy_(sets[k]["Y"], non_blocking=True))
        e2e_value = flops * world / (e2e_ms * 1e-3) / 1e12

    gemm_kernel = FUSED_LINEAR_KERNEL if one_launch else gemm_kernel_name(M)
    traffic = recorded_traffic(gemm_kernel, wl.name)

    if rank != 0:
        return None
    cpu = None
    if world == 1 and not args.no_cpu_baseline and not light:
        try:
            rate, rows, dt, threads = oracle_linear_rate(d, wl.M, args.cpu_seconds)
            cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": f"{rows} of {wl.M} rows (full N={N}, K={K}), {dt:.1f} s; "
                             "weight prepared outside the timing"}
        except Exception as e:  # noqa: BLE001 - reported, not fatal
            cpu = {"value": None, "unit": "TFLOP/s", "cores": None, "kind": "oracle",
                   "sample": f"failed: {e}"}

    # the GEMM's bound: FP4 tensor throughput above the ridge intensity, HBM
    # bytes below it (decode: the weight bytes)
    # (one launch: the kernel reads X in bf16 instead of the transformed codes)
    x_bytes = M * K * 2 if one_launch else M * (K // 2 + K // 32)
    gemm_bytes = x_bytes + N * (K // 2 + K // 32) + M * N * 2
    timing = (f"CUDA events around kernel groups: {batches.describe()} of the {args.steps} timed steps")
    if flops / gemm_bytes >= fp4_peak * 1e12 / (peaks["hbm_gbs"] * 1e9):
        roofline = {"bound": "tensor", "kernel": gemm_kernel,
                    "achieved": gemm_tflops, "peak": fp4_peak, "unit": "TFLOP/s",
                    "frac": gemm_tflops / fp4_peak, "traffic": traffic,
                    "peak_note": f"{peaks['source']} bf16 burst {peaks['bf16_tflops']} x "
                                 f"{FP4_OVER_BF16:g} (nominal fp4/bf16)",
                    "avg_launch_us": gemm_avg * 1e3, "timing": timing}
    else:
        gbs = gemm_bytes / (gemm_avg * 1e-3) / 1e9
        roofline = {"bound": "hbm",
                    "kernel": gemm_kernel,
                    "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm_gbs"], "traffic": traffic, "bytes_per_launch": gemm_bytes,
                    "peak_note": f"{peaks['source']} HBM copy bandwidth",
                    "tflops": gemm_tflops, "avg_launch_us": gemm_avg * 1e3, "timing": timing}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4 (e2m1 codes, e8m0 block scales, fp32 accumulate; fp32 transform)",
        "data": "synthetic",
        "config": dict(workload_config(wl), hadamard_block=hb,
                       **({"input": "gate|up [M, 2K]; SiLU(gate) * up fused into the transform"}
                          if fused else {})),
        "roofline": roofline,
        "act_quant": {"kernel": f"inside {FUSED_LINEAR_KERNEL} (no launch of its own)", "achieved": None,
                      "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": None, "bytes_per_launch": 0,
                      "traffic": None, "avg_launch_us": None} if one_launch else
                     {"kernel": "quant_grouped_tma_kernel<.., true> (SwiGLU, one group)" if fused
                      else "quant_kernel (register-staged: a few rows)" if M <= 64 and hb == 32
                      else "quant_dense_tma_kernel", "achieved": quant_gbs,
                      "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": quant_gbs / peaks["hbm_gbs"], "bytes_per_launch": quant_bytes,
                      "traffic": None if fused or (M <= 64 and hb == 32) else recorded_traffic("quant_dense_tma_kernel", wl.name),
                      "avg_launch_us": quant_avg * 1e3},
        "cpu_baseline": cpu,
        "e2e": None if light else {
            "value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": M * xcols * 2,
            "d2h_bytes_per_step": M * N * 2, "ms_per_step": e2e_ms,
            "copies": f"overlapped across steps ({nslot} buffer slots, separate copy streams)",
            "serial_ms_per_step": e2e_serial_ms},
        "gpu_launches": len(parts) * args.steps,
        "host_enqueue_us_per_step": host_enqueue_s / args.steps * 1e6,
        "launch": plan.describe(),
        "eager_delay_ms": batches.padding_ms(),
        "eager_batch_host_us": batches.host_us, "eager_batch_device_us": batches.device_us,
        "clocks": sampler.summary(),
    }
    return line


# ------------------------------------------------------- W4A16 GPU arm

METRIC_W4A16 = "W4A16 linear TFLOP/s (bf16 GEMM on expanded MXFP4 weights)"


def oracle_w4a16_rate(d, inv, wd, target_s: float):
    """Time the CPU oracle of the W4A16 layer (bf16 transform of sampled rows,
    fp64 GEMM against the expanded weight) and return (TFLOP/s, rows, s, threads)."""
    import numpy as np
    import torch

    import oracle

    wl = d["workload"]
    w64 = (wd.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    def run(n):
        t0 = time.perf_counter()
        xt = oracle.transform_bf16(d["X"][:n], inv)
        a = (xt.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        torch.from_numpy(oracle.gemm_ref(a, w64)).to(torch.bfloat16)
        return time.perf_counter() - t0

    run(min(wl.M, 4))
    n = max(1, min(wl.M, 16))
    dt = run(n)
    while dt < target_s * 0.5 and n < wl.M:
        n = min(wl.M, max(n + 1, int(n * min(8.0, target_s / max(dt, 1e-3)))))
        dt = run(n)
    threads = max(oracle.num_threads(), os.cpu_count() or 1)
    return 2.0 * n * wl.N * wl.K / dt / 1e12, n, dt, threads


def gpu_arm_w4a16(args, rank: int, world: int):
    """The W4A16 fallback layer: the bf16 transform and the W4A16 GEMM, which
    reads the MXFP4 checkpoint and expands it to bf16 in shared memory (both
    this library's kernels)."""
    import torch
    import torch.distributed as dist

    import workloads
    import w4a4_mxfp4_quantized_02_b300 as mq

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    mq.lib()
    peaks = load_peaks()
    d = workloads.make_dense(args.config)
    wl = d["workload"]
    M, N, K = wl.M, wl.N, wl.K
    hb = args.hadamard_block
    stream = torch.cuda.current_stream()

    Xc = d["X_calib"].to(dev)
    W = d["W"].to(dev)
    s, inv = mq.macaq_balance_scales(Xc, W)
    w_codes, w_scales = mq.macaq_quant_weight_hb(W, s, hb)
    del W, Xc

    w_bytes = w_codes.numel() + w_scales.numel()
    step_bytes = M * K * 4 + w_bytes + M * N * 2
    nsets = max(2, math.ceil(2.5 * L2_BYTES / step_bytes) + 1)
    X0 = d["X"].to(dev)
    sets = [{"X": X0.clone() if i else X0, "wc": w_codes.clone() if i else w_codes,
             "ws": w_scales.clone() if i else w_scales,
             "Xt": torch.empty(M, K, dtype=torch.bfloat16, device=dev),
             "Y": torch.empty(M, N, dtype=torch.bfloat16, device=dev)} for i in range(nsets)]

    def transform_part(i):
        b = sets[i % nsets]
        mq.macaq_transform_act_bf16(b["X"], inv, hb, Xt=b["Xt"])

    def gemm_part(i):
        b = sets[i % nsets]
        mq.macaq_w4a16_gemm(b["Xt"], b["wc"], b["ws"], N, Y=b["Y"])

    def step(i):
        transform_part(i)
        gemm_part(i)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    chunk = nsets * max(1, math.ceil(8 / nsets))
    graph = None if args.no_graphs else capture_graph(lambda: [step(i) for i in range(chunk)])
    plan = StepPlan(args.steps, args.kernel_events_every, chunk if graph is not None else 0)
    batches = KernelBatches(plan.eager_steps, min(nsets, 4), 2)
    batches.calibrate([transform_part, gemm_part], stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(pci_bus_id(dev))
    with sampler:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        batches.run([transform_part, gemm_part], stream, graph, plan.replays)
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end) - batches.padding_ms()
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    q_ms, g_ms = batches.per_launch_ms()
    status = mq.macaq_check_device_error()
    if status != 0:
        raise RuntimeError(f"device error in the timed region: {mq.macaq_status_string(status)}")
    flops = 2.0 * M * N * K
    value = flops * args.steps * world / (elapsed_ms * 1e-3) / 1e12
    gemm_tflops = flops / (g_ms * 1e-3) / 1e12
    # algorithmic bytes: bf16 activations, the MXFP4 weight (codes and scales), bf16 Y
    gemm_bytes = M * K * 2 + N * (K // 2 + K // 32) + M * N * 2
    t_bytes = M * K * 4
    t_gbs = t_bytes / (q_ms * 1e-3) / 1e9

    # end to end through the C ABI (pinned host X in, Y out)
    work = torch.empty(mq.macaq_w4a16_linear_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
    Xh = d["X"].pin_memory()
    nslot = min(3, nsets)
    Yh = [torch.empty(M, N, dtype=torch.bfloat16).pin_memory() for _ in range(nslot)]
    e2e_steps = max(3, min(args.steps, 50))
    e2e_ms = e2e_pipelined(
        stream, e2e_steps, nslot,
        lambda k: sets[k]["X"].copy_(Xh, non_blocking=True),
        lambda k: mq.macaq_w4a16_linear(sets[k]["X"], inv, sets[0]["wc"], sets[0]["ws"], N, hb, Y=sets[k]["Y"],
                                        workspace=work),
        lambda k: Yh[k].copy_(sets[k]["Y"], non_blocking=True))

    if rank != 0:
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        try:
            import numpy as np

            import oracle
            s_ref, inv_ref = oracle.balance_scales(d["X_calib"], d["W"])
            cw, sw = oracle.quantize(d["W"], s_ref, hb=hb)
            wd = oracle.dequant_bf16(cw, sw)      # weight preparation: outside the timing
            rate, rows, dt, threads = oracle_w4a16_rate(d, inv_ref.astype(np.float32), wd, args.cpu_seconds)
            cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": f"{rows} of {M} rows (full N={N}, K={K}), {dt:.1f} s; "
                             "weight expansion outside the timing"}
        except Exception as e:  # noqa: BLE001 - reported, not fatal
            cpu = {"value": None, "unit": "TFLOP/s", "cores": None, "kind": "oracle",
                   "sample": f"failed: {e}"}
    bf16_peak = peaks["bf16_tflops"]
    timing = f"CUDA events around kernel groups: {batches.describe()} of the {args.steps} timed steps"
    if flops / gemm_bytes >= bf16_peak * 1e12 / (peaks["hbm_gbs"] * 1e9):
        roofline = {"bound": "tensor", "kernel": "gemm_w4a16_kernel",
                    "achieved": gemm_tflops, "peak": bf16_peak, "unit": "TFLOP/s",
                    "frac": gemm_tflops / bf16_peak, "traffic": recorded_traffic("gemm_w4a16_kernel", wl.name),
                    "peak_note": f"{peaks['source']} bf16 burst", "avg_launch_us": g_ms * 1e3,
                    "timing": timing}
    else:
        gbs = gemm_bytes / (g_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": "gemm_w4a16_kernel", "achieved": gbs,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                    "traffic": recorded_traffic("gemm_w4a16_kernel", wl.name), "bytes_per_launch": gemm_bytes,
                    "peak_note": f"{peaks['source']} HBM copy bandwidth", "tflops": gemm_tflops,
                    "avg_launch_us": g_ms * 1e3, "timing": timing}
    line = {
        "metric": METRIC_W4A16, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (fp32 transform rounded to bf16; MXFP4 weights expanded to bf16 on chip; fp32 accumulate)",
        "data": "synthetic",
        "config": dict(workload_config(wl), hadamard_block=hb, precision="w4a16"),
        "roofline": roofline,
        "act_transform": {"kernel": "quant_dense_tma_kernel (bf16 output)", "achieved": t_gbs,
                          "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": t_gbs / peaks["hbm_gbs"],
                          "bytes_per_launch": t_bytes, "avg_launch_us": q_ms * 1e3},
        "cpu_baseline": cpu,
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2,
                "ms_per_step": e2e_ms,
                "copies": f"overlapped across steps ({nslot} buffer slots, separate copy streams)"},
        "gpu_launches": 2 * args.steps,
        "launch": plan.describe(),
        "eager_delay_ms": batches.padding_ms(),
        "eager_batch_host_us": batches.host_us, "eager_batch_device_us": batches.device_us,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------- Flip Refinement GPU arm

METRIC_FLIP = "offline weight preparation with Flip Refinement: weight rows per second"
FP32_LANES_PER_SM = 128        # fp32 FMA lanes per SM (B300)


def oracle_flip_rate(d, rows: int, sweeps: int):
    """Time the CPU oracle: the Hessian of the calibration rows, then the
    transform, round to nearest and refinement of `rows` weight rows.
    Returns (rows/s with the Hessian's time charged pro rata, detail)."""
    import oracle

    wl = d["workload"]
    t0 = time.perf_counter()
    s, inv = oracle.balance_scales(d["X_calib"], d["W"])
    A = oracle.transform_f32(d["X_calib"], inv)
    H = oracle.flip_hessian(A)
    t_h = time.perf_counter() - t0
    t0 = time.perf_counter()
    W = d["W"][:rows].contiguous()
    wt = oracle.transform_f32(W, s)
    c, sc = oracle.quantize(W, s)
    oracle.flip_refine(wt, H, c, sc, sweeps)
    t_r = time.perf_counter() - t0
    rate = rows / (t_r + t_h * rows / wl.N)
    threads = max(oracle.num_threads(), os.cpu_count() or 1)
    return rate, t_h, t_r, threads


def gpu_arm_flip(args, rank: int, world: int):
    """One layer's offline preparation: balance scales, the fp32 transforms of
    the calibration rows and the weight, the Hessian, round-to-nearest MXFP4,
    and Flip Refinement of every weight row."""
    import torch

    import workloads
    import w4a4_mxfp4_quantized_02_b300 as mq

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    mq.lib()
    peaks = load_peaks()
    d = workloads.make_dense(args.config)
    wl = d["workload"]
    N, K, Mc = wl.N, wl.K, wl.calib_rows
    hb = args.hadamard_block
    sweeps = args.sweeps
    stream = torch.cuda.current_stream()
    Xc = d["X_calib"].to(dev)
    W = d["W"].to(dev)
    A = torch.empty(Mc, K, dtype=torch.float32, device=dev)
    Wt = torch.empty(N, K, dtype=torch.float32, device=dev)
    H = torch.empty(K, K, dtype=torch.float32, device=dev)
    codes = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(mq.macaq_scale_bytes(N, K), dtype=torch.uint8, device=dev)
    flips = torch.empty(N, dtype=torch.int32, device=dev)
    work = torch.empty(mq.macaq_flip_refine_workspace_bytes(N, K), dtype=torch.uint8, device=dev)
    stages = ["balance+transforms", "hessian", "rtn", "prepare", "sweeps"]

    def step(ev=None):
        rec = (lambda i: ev[i].record(stream)) if ev is not None else (lambda i: None)
        rec(0)
        s, inv = mq.macaq_balance_scales(Xc, W)
        mq.macaq_transform_f32(Xc, inv, hb, Y=A)
        mq.macaq_transform_f32(W, s, hb, Y=Wt)
        rec(1)
        mq.macaq_flip_hessian(A, args.damp, H=H)
        rec(2)
        mq.macaq_quant_weight_hb(W, s, hb, codes, scales)
        rec(3)
        mq.macaq_flip_prepare(Wt, H, codes, scales, work)
        rec(4)
        mq.macaq_flip_sweeps(H, N, K, codes, scales, work, sweeps, flips=flips)
        rec(5)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if mq.macaq_check_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    sampler = ClockSampler(pci_bus_id(dev))
    torch.cuda.synchronize()
    with sampler:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize()
    elapsed_ms = t0.elapsed_time(t1)
    if mq.macaq_check_device_error() != 0:
        raise RuntimeError("device error in the timed region")
    parts = {name: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j, name in enumerate(stages)}
    moves = flips.cpu().numpy()
    ms = elapsed_ms / args.steps

    cpu = None
    if not args.no_cpu_baseline:
        try:
            rate, t_h, t_r, threads = oracle_flip_rate(d, args.cpu_rows, sweeps)
            cpu = {"value": rate, "unit": "rows/s", "cores": threads, "kind": "oracle",
                   "sample": f"Hessian of {Mc} x {K} calibration rows ({t_h:.1f} s, charged pro rata) "
                             f"and {args.cpu_rows} of {N} weight rows refined ({t_r:.1f} s)"}
        except Exception as e:  # noqa: BLE001 - reported, not fatal
            cpu = {"value": None, "unit": "rows/s", "cores": None, "kind": "oracle", "sample": f"failed: {e}"}
    # the dominant kernel is the descent: per move it streams one row of H
    # (K fp32) into the row's g; per row it also reads g and writes codes
    total_moves = float(moves.sum())
    sweep_bytes = total_moves * K * 4 + N * K * 4 + N * K
    sweep_gbs = sweep_bytes / (parts["sweeps"] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": "flip_sweep_kernel", "achieved": sweep_gbs,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": sweep_gbs / peaks["hbm_gbs"],
                "traffic": None, "bytes_per_launch": sweep_bytes,
                "peak_note": f"{peaks['source']} HBM copy bandwidth (H of {K * K * 4 / 1e6:.0f} MB "
                             f"{'fits' if K * K * 4 < L2_BYTES else 'exceeds'} L2)",
                "avg_launch_us": parts["sweeps"] * 1e3}
    # the Hessian and g = R H are fp32 FMA chains on the CUDA cores (no tensor
    # path keeps the definition's order): their bound is the fp32 FMA rate
    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    clk = sampler.summary().get("sm_mhz") or 2032.0
    fp32_peak = 2.0 * sm * FP32_LANES_PER_SM * clk * 1e6 / 1e12
    fma_chains = {
        "kernel": "sgemm_seq_kernel", "unit": "TFLOP/s", "peak": fp32_peak, "bound": "alu",
        "peak_note": f"fp32 FMA: {sm} SMs x {FP32_LANES_PER_SM} lanes x 2 x {clk:.0f} MHz (derived)",
        "hessian": 2.0 * K * K * Mc / (parts["hessian"] * 1e-3) / 1e12,
        "prepare_g": 2.0 * N * K * K / (parts["prepare"] * 1e-3) / 1e12,
    }
    line = {
        "metric": METRIC_FLIP, "value": N / (ms * 1e-3), "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (fp32 transform, Hessian and descent; MXFP4 codes)", "data": "synthetic",
        "config": dict(workload_config(wl), hadamard_block=hb, sweeps=sweeps, damp=args.damp,
                       stage="flip refinement (offline)"),
        "stages_ms": parts,
        "moves_per_row": {"mean": float(moves.mean()), "max": int(moves.max()), "min": int(moves.min())},
        "roofline": roofline,
        "fma_chains": fma_chains,
        "cpu_baseline": cpu,
        "e2e": None,
        "gpu_launches": 8 * args.steps,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- MoE GPU arm

def moe_workload_config(wl, fused: bool = True):
    how = ("the gate+up GEMM epilogue writes the down input's MXFP4 (SiLU(gate)*up, transform)" if fused
           else "SiLU(gate)*up fused into the down input's transform")
    return {"workload": f"{wl.name}: {wl.T} tokens x top-{wl.topk} of {wl.E} experts = {wl.rows} rows; "
                        f"gate+up K={wl.K} N={2 * wl.F}, {how}, down K={wl.F} N={wl.K}, weighted "
                        f"top-{wl.topk} combine into the token outputs; bf16 in/out, MXFP4 W4A4",
            "T": wl.T, "E": wl.E, "topk": wl.topk, "K": wl.K, "F": wl.F, "rows": wl.rows,
            "l2": "weights (302 MB of codes) exceed L2; no input rotation needed"}


def oracle_moe_rate(d, target_s: float):
    """CPU oracle on the rows of a sample of experts (gate+up projection)."""
    import numpy as np  # noqa: F401
    import torch  # noqa: F401

    import oracle

    wl = d["workload"]
    r, cr = d["routing"], d["calib_routing"]
    off, coff = r["offsets"].numpy(), cr["offsets"].numpy()
    done_flops, dt, experts = 0.0, 0.0, 0
    for e in range(wl.E):
        xc = d["X_calib"][cr["row_src"][coff[e]:coff[e + 1]].long()]
        s, inv = oracle.balance_scales(xc, d["W_gu"][e])
        cw, sw = oracle.quantize(d["W_gu"][e], s)
        deq_w = oracle.dequant(cw, sw)           # weight preparation: outside the timing
        X = d["X"][r["row_src"][off[e]:off[e + 1]].long()]
        t0 = time.perf_counter()
        ca, sa = oracle.quantize(X, inv)
        oracle.gemm_ref(oracle.dequant(ca, sa), deq_w)
        dt += time.perf_counter() - t0
        done_flops += 2.0 * X.shape[0] * 2 * wl.F * wl.K
        experts += 1
        if dt > target_s:
            break
    threads = max(oracle.num_threads(), os.cpu_count() or 1)
    return done_flops / dt / 1e12, experts, dt, threads


def gpu_arm_moe(args, rank: int, world: int, config: str | None = None, light: bool = False):
    """The routed layer's line (rank 0; None elsewhere); light as gpu_arm."""
    import torch
    import torch.distributed as dist

    import workloads
    import w4a4_mxfp4_quantized_02_b300 as mq

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    mq.lib()
    peaks = load_peaks()
    config = config or args.config
    d = workloads.make_moe(workloads.MOE if config == "moe" else workloads.MOE_SMALL)
    wl = d["workload"]
    E, K, F, rows = wl.E, wl.K, wl.F, wl.rows
    stream = torch.cuda.current_stream()

    # offline preparation (not timed): per-expert calibration and weight quantisation
    r, cr = d["routing"], d["calib_routing"]
    coff = cr["offsets"].numpy()
    Xc = d["X_calib"].to(dev)
    Xdc = d["Xd_calib"].to(dev)
    c_rows = cr["row_src"].to(dev)
    W = d["W_gu"].to(dev)
    s_gu = torch.empty(E, K, dtype=torch.float32, device=dev)
    inv_gu = torch.empty_like(s_gu)
    for e in range(E):
        s_gu[e], inv_gu[e] = mq.macaq_balance_scales(Xc, W[e], xc_rows=c_rows[coff[e]:coff[e + 1]])
    fused = not args.moe_unfused
    if fused:
        # gate and up rows interleaved in chunks of 64 channels: the gate+up
        # GEMM's epilogue then writes the down input's MXFP4 directly
        Wil = mq.macaq_interleave_gate_up(W)
        wgu_codes, wgu_scales = mq.macaq_quant_weight_grouped(Wil, s_gu)
        del Wil
    else:
        wgu_codes, wgu_scales = mq.macaq_quant_weight_grouped(W, s_gu)
    del W
    W = d["W_down"].to(dev)
    s_dn = torch.empty(E, F, dtype=torch.float32, device=dev)
    inv_dn = torch.empty_like(s_dn)
    for e in range(E):
        s_dn[e], inv_dn[e] = mq.macaq_balance_scales(Xdc[coff[e]:coff[e + 1]], W[e])
    wdn_codes, wdn_scales = mq.macaq_quant_weight_grouped(W, s_dn)
    del W, Xc, Xdc

    X = d["X"].to(dev)
    row_src = r["row_src"].to(dev)
    ident = torch.arange(rows, dtype=torch.int32, device=dev)
    offs = r["offsets"].to(dev)
    P = mq.macaq_grouped_padded_rows(rows, E)
    a_gu = torch.empty(P, K // 2, dtype=torch.uint8, device=dev)
    as_gu = torch.empty(mq.macaq_scale_bytes(P, K), dtype=torch.uint8, device=dev)
    a_dn = torch.empty(P, F // 2, dtype=torch.uint8, device=dev)
    as_dn = torch.empty(mq.macaq_scale_bytes(P, F), dtype=torch.uint8, device=dev)
    Ygu = torch.empty(rows, 2 * F, dtype=torch.bfloat16, device=dev)
    Ydn = torch.empty(rows, K, dtype=torch.bfloat16, device=dev)
    tok_rows = r["tok_rows"].to(dev)
    tok_w = r["tok_weights"].to(dev)
    Ytok = torch.empty(wl.T, K, dtype=torch.bfloat16, device=dev)

    def k_quant_gu(i, Xin=None):
        mq.macaq_quant_act_grouped(X if Xin is None else Xin, row_src, offs, inv_gu, rows, E, a_gu, as_gu)

    def k_gemm_gu(i):
        if fused:
            # the epilogue forms h = SiLU(gate) * up and writes the down input's MXFP4
            mq.macaq_grouped_w4a4_gemm_swiglu(a_gu, as_gu, wgu_codes, wgu_scales, offs, rows, E, F, K, inv_dn,
                                              h_codes=a_dn, h_scales=as_dn)
        else:
            mq.macaq_grouped_w4a4_gemm(a_gu, as_gu, wgu_codes, wgu_scales, offs, rows, E, 2 * F, K, Y=Ygu)

    def k_quant_dn(i):
        # unfused route: the down input is SiLU(gate) * up of the bf16 gate+up
        # output, fused into its transform
        mq.macaq_quant_act_grouped_silu(Ygu, offs, inv_dn, rows, E, a_dn, as_dn)

    def k_gemm_dn(i):
        mq.macaq_grouped_w4a4_gemm(a_dn, as_dn, wdn_codes, wdn_scales, offs, rows, E, K, F, Y=Ydn)

    def k_combine(i, Yout=None):
        # the token outputs: each token's eight expert rows, weighted
        mq.macaq_moe_combine(Ydn, tok_rows, tok_w, out=Ytok if Yout is None else Yout)

    parts = [k_quant_gu, k_gemm_gu] + ([] if fused else [k_quant_dn]) + [k_gemm_dn, k_combine]

    def step(Xin=None, Yout=None):
        k_quant_gu(0, Xin)
        for part in parts[1:-1]:
            part(0)
        k_combine(0, Yout)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = mq.macaq_check_device_error()
    if status != 0:
        raise RuntimeError(f"device error during warm-up: {mq.macaq_status_string(status)}")
    chunk = 4
    graph = None if args.no_graphs else capture_graph(lambda: [step() for _ in range(chunk)])
    plan = StepPlan(args.steps, args.kernel_events_every, chunk if graph is not None else 0)
    # every step computes the same layer on the same tokens, so a batch of
    # steps may share the one set of intermediate buffers
    batches = KernelBatches(plan.eager_steps, 2, len(parts))
    batches.calibrate(parts, stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(pci_bus_id(dev))
    with sampler:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        h0 = time.perf_counter()
        batches.run(parts, stream, graph, plan.replays)
        host_enqueue_s = time.perf_counter() - h0
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end) - batches.padding_ms()
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    avg = batches.per_launch_ms()
    if fused:
        avg = avg[:2] + [None] + avg[2:]   # no separate down-input transform
    status = mq.macaq_check_device_error()
    if status != 0:
        raise RuntimeError(f"device error in the timed region: {mq.macaq_status_string(status)}")

    flops = wl.flops_gate_up + wl.flops_down
    value = flops * args.steps * world / (elapsed_ms * 1e-3) / 1e12
    # algorithmic bytes: codes + scales of A and W, bf16 Y (the grouped GEMMs are
    # bound by the weight bytes at this token count)
    def gemm_bytes(n, k, out_bytes):
        return rows * (k // 2 + k // 32) + E * n * (k // 2 + k // 32) + out_bytes
    # the fused gate+up GEMM writes the down input's codes and scales instead of bf16 g|u
    gu_out = rows * (F // 2 + F // 32) if fused else rows * 2 * F * 2
    gu_bytes, dn_bytes = gemm_bytes(2 * F, K, gu_out), gemm_bytes(K, F, rows * K * 2)
    # algorithmic bytes: each token row read once (its eight expert copies are
    # gathered from L2), every sorted row's codes and scales written once
    q_bytes = [wl.T * K * 2 + rows * (K // 2 + K // 32), rows * 2 * F * 2 + rows * (F // 2 + F // 32)]
    gu_gbs = gu_bytes / (avg[1] * 1e-3) / 1e9
    dn_gbs = dn_bytes / (avg[3] * 1e-3) / 1e9
    # combine: every expert row read once, every token row written once
    cb_bytes = rows * K * 2 + wl.T * K * 2 + wl.T * wl.topk * 8
    cb_gbs = cb_bytes / (avg[4] * 1e-3) / 1e9

    e2e_ms = e2e_serial_ms = None
    if not light:
        # end to end through the C ABI: pinned host tokens in, pinned host token outputs out
        e2e_steps = max(3, min(args.steps, 20))
        Xh = d["X"].pin_memory()
        Yh = [torch.empty(wl.T, K, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        for _ in range(2):
            X.copy_(Xh, non_blocking=True)
            step()
            Yh[0].copy_(Ytok, non_blocking=True)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            X.copy_(Xh, non_blocking=True)
            step()
            Yh[0].copy_(Ytok, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_serial_ms = e0.elapsed_time(e1) / e2e_steps
        Xs, Ys = [X, torch.empty_like(X)], [Ytok, torch.empty_like(Ytok)]
        e2e_ms = e2e_pipelined(stream, e2e_steps, 2,
                               lambda k: Xs[k].copy_(Xh, non_blocking=True),
                               lambda k: step(Xin=Xs[k], Yout=Ys[k]),
                               lambda k: Yh[k].copy_(Ys[k], non_blocking=True))

    if rank != 0:
        return None
    cpu = None
    if world == 1 and not args.no_cpu_baseline and not light:
        try:
            rate, experts, dt, threads = oracle_moe_rate(d, args.cpu_seconds)
            cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": f"gate+up projection of the rows of {experts} of {E} experts, {dt:.1f} s; "
                             "weight prepared outside the timing"}
        except Exception as e:  # noqa: BLE001 - reported, not fatal
            cpu = {"value": None, "unit": "TFLOP/s", "cores": None, "kind": "oracle",
                   "sample": f"failed: {e}"}
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4 (e2m1 codes, e8m0 block scales, fp32 accumulate; fp32 transform)",
        "data": "synthetic",
        "config": moe_workload_config(wl, fused),
        "roofline": {"bound": "hbm",
                     "kernel": ("gemm_mxf4_pair_kernel<6, true, 1> (grouped gate+up, MXFP4 h epilogue)" if fused
                                else "gemm_mxf4_pair_kernel<6, true> (grouped, gate+up)"),
                     "achieved": gu_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gu_gbs / peaks["hbm_gbs"],
                     "traffic": recorded_traffic("gemm_mxf4_pair_kernel", wl.name) if fused else None,
                     "bytes_per_launch": gu_bytes, "avg_launch_us": avg[1] * 1e3,
                     "tflops": wl.flops_gate_up / (avg[1] * 1e-3) / 1e12,
                     "timing": f"CUDA events around kernel groups: {batches.describe()} of the "
                               f"{args.steps} timed steps"},
        "down_gemm": {"achieved": dn_gbs, "unit": "GB/s", "frac": dn_gbs / peaks["hbm_gbs"],
                      "bytes_per_launch": dn_bytes, "avg_launch_us": avg[3] * 1e3,
                      "tflops": wl.flops_down / (avg[3] * 1e-3) / 1e12},
        "combine": {"kernel": "moe_combine_kernel", "achieved": cb_gbs, "unit": "GB/s",
                    "frac": cb_gbs / peaks["hbm_gbs"], "bytes_per_launch": cb_bytes,
                    "avg_launch_us": avg[4] * 1e3},
        "act_quant": ({"kernel": "quant_grouped_tma_kernel (token rows; the down input comes from the "
                                 "gate+up GEMM's epilogue)",
                       "achieved": q_bytes[0] / (avg[0] * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                       "unit": "GB/s", "frac": q_bytes[0] / (avg[0] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                       "bytes_per_launch": q_bytes[0], "avg_launch_us": avg[0] * 1e3} if fused else
                      {"kernel": "quant_grouped_tma_kernel (token rows; SwiGLU-fused for the down input)",
                       "achieved": [q_bytes[0] / (avg[0] * 1e-3) / 1e9, q_bytes[1] / (avg[2] * 1e-3) / 1e9],
                       "peak": peaks["hbm_gbs"], "unit": "GB/s (gate+up input, down input)",
                       "frac": [q_bytes[0] / (avg[0] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                q_bytes[1] / (avg[2] * 1e-3) / 1e9 / peaks["hbm_gbs"]],
                       "bytes_per_launch": q_bytes, "avg_launch_us": [avg[0] * 1e3, avg[2] * 1e3]}),
        "cpu_baseline": cpu,
        "e2e": None if light else {
            "value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": wl.T * K * 2, "d2h_bytes_per_step": wl.T * K * 2,
            "ms_per_step": e2e_ms,
            "copies": "overlapped across steps (2 buffer slots, separate copy streams)",
            "serial_ms_per_step": e2e_serial_ms},
        "gpu_launches": len(parts) * args.steps,
        "host_enqueue_us_per_step": host_enqueue_s / args.steps * 1e6,
        "launch": plan.describe(),
        "eager_delay_ms": batches.padding_ms(),
        "eager_batch_host_us": batches.host_us, "eager_batch_device_us": batches.device_us,
        "clocks": sampler.summary(),
    }
    return line


class StepPlan:
    """How the timed steps run.  About one step in `every` runs eagerly for
    per-kernel timing (KernelBatches).  With a captured graph of `chunk` steps,
    the other steps run as whole-graph replays (the host's launch cost then
    does not pace short steps); without one, every step runs eagerly."""

    def __init__(self, steps: int, every: int, chunk: int):
        every = max(1, every)
        n_events = (steps + every - 1) // every
        if chunk > 0:
            self.replays = (steps - n_events) // chunk
            first = self.replays * chunk
            self.eager_steps = list(range(first, steps))
            self.event_steps = list(self.eager_steps)
        else:
            self.replays = 0
            self.eager_steps = list(range(steps))
            self.event_steps = list(self.eager_steps)
        self.chunk = chunk

    def describe(self) -> str:
        if self.replays:
            return (f"{self.replays} replays of a CUDA graph of {self.chunk} steps, spread evenly in front "
                    f"of {len(self.eager_steps)} eager steps in kernel-by-kernel batches with CUDA events")
        return "eager launches in kernel-by-kernel batches with CUDA events"


def replay_schedule(replays: int, groups: int) -> list:
    """How many graph replays go in front of each of `groups` eager groups:
    all `replays`, spread as evenly as whole numbers allow (no group gets more
    than one more than another); with no groups, one entry holding them all."""
    if groups <= 0:
        return [replays]
    return [(k + 1) * replays // groups - k * replays // groups for k in range(groups)]


class KernelBatches:
    """The eager steps of the timed region, run in batches of `nb` whole steps
    kernel by kernel -- every step's first kernel, then every step's second,
    and so on -- with one CUDA event between kernel groups on the launching
    stream.  Consecutive launches of one kernel keep their programmatic launch
    overlap (as in a stack of layers), and an event's launch gap is paid once
    per group instead of once per launch.  Every step still runs all of its
    kernels on its own buffers; a batch never reuses a buffer set."""

    CYCLES_PER_US = 2000  # SM cycles per microsecond (about 2 GHz) for the delays

    def __init__(self, steps: list, nb: int, nparts: int):
        import torch

        nb = max(1, nb)
        self.groups = [steps[i:i + nb] for i in range(0, len(steps), nb)]
        self.nparts = nparts
        self.events = [[torch.cuda.Event(enable_timing=True) for _ in range(nparts + 1)]
                       for _ in self.groups]
        self.pad_cycles = 0
        self.pad_events = []
        self.host_us = self.device_us = None

    def calibrate(self, parts, stream):
        """Short kernels can finish before the host has enqueued the next one;
        the group's events then time the host, not the kernels.  Run the
        first group once (untimed) queued behind a device-side delay, compare
        the host's enqueue time with the group's device time, and when the
        host is not well ahead, precede every timed group by a delay of twice
        the host time, so that the whole group is queued before its first
        event.  The delays lie outside the groups' events and are subtracted
        from the timed region's device time (padding_ms)."""
        import torch

        if not self.groups:
            return
        group = self.groups[0]
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(20000 * self.CYCLES_PER_US)  # about 20 ms to enqueue behind
        e0.record(stream)
        h0 = time.perf_counter()
        for part in parts:
            for i in group:
                part(i)
        host_s = time.perf_counter() - h0
        e1.record(stream)
        torch.cuda.synchronize()
        self.host_us = host_s * 1e6
        self.device_us = e0.elapsed_time(e1) * 1e3
        # only where the device would otherwise run dry: a delay in front of
        # a group the host keeps queued anyway would only add idle time (and
        # idle time lets a power-capped GPU recover, flattering the kernels)
        if self.host_us > 0.8 * self.device_us:
            self.pad_cycles = int(2 * self.host_us * self.CYCLES_PER_US)

    def run(self, parts, stream, graph=None, replays: int = 0):
        """The timed steps: `replays` replays of `graph` (whole steps), spread
        evenly in front of the groups, so that each group is enqueued while the
        device still runs the replayed steps before it (real work, not idle
        time), then each group kernel by kernel between its events."""
        import torch

        schedule = replay_schedule(replays, len(self.groups))
        if not self.groups:
            for _ in range(schedule[0]):
                graph.replay()
        for k, (group, ev) in enumerate(zip(self.groups, self.events)):
            for _ in range(schedule[k]):
                graph.replay()
            if self.pad_cycles:
                pe = torch.cuda.Event(enable_timing=True)
                pe.record(stream)
                torch.cuda._sleep(self.pad_cycles)
                self.pad_events.append((pe, ev[0]))
            ev[0].record(stream)
            for j, part in enumerate(parts):
                for i in group:
                    part(i)
                ev[j + 1].record(stream)

    def padding_ms(self) -> float:
        """Device time of the delays before the groups (after a synchronize)."""
        return sum(a.elapsed_time(b) for a, b in self.pad_events)

    def per_launch_ms(self) -> list:
        """Average device time per launch of each kernel (after a synchronize)."""
        n = sum(len(g) for g in self.groups)
        return [sum(ev[j].elapsed_time(ev[j + 1]) for ev in self.events) / n for j in range(self.nparts)]

    def describe(self) -> str:
        sizes = sorted({len(g) for g in self.groups})
        out = f"{sum(len(g) for g in self.groups)} eager steps in kernel-by-kernel batches of {sizes}"
        if self.pad_cycles:
            out += (f"; the host enqueued a batch in {self.host_us:.0f} us against {self.device_us:.0f} us "
                    f"on the device, so each batch followed a device-side delay of about "
                    f"{2 * self.host_us:.0f} us (outside its events; subtracted from the region's time)")
        return out


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (one all-reduce; x itself when alone)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def e2e_pipelined(stream, steps: int, nslot: int, h2d, run, d2h) -> float:
    """End-to-end ms per step with the host copies overlapped across steps:
    step i copies its input in on one stream, runs on `stream`, copies its
    result out on a third, using buffer slot i % nslot (a slot is reused only
    after its previous result has left and its input been consumed).  Every
    step still moves its own input and result over PCIe inside the timing."""
    import torch

    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nslot)]
    ev_run = [torch.cuda.Event() for _ in range(nslot)]
    ev_out = [torch.cuda.Event() for _ in range(nslot)]

    def one(i):
        k = i % nslot
        with torch.cuda.stream(s_in):
            if i >= nslot:
                s_in.wait_event(ev_run[k])
            h2d(k)
            ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        if i >= nslot:
            stream.wait_event(ev_out[k])
        run(k)
        ev_run[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[k])
            d2h(k)
            ev_out[k].record(s_out)

    for i in range(nslot):
        one(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    s_in.wait_event(t0)
    for i in range(steps):
        one(i)
    for k in range(nslot):
        stream.wait_event(ev_out[k])
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def capture_graph(fn):
    """Capture fn (a run of whole steps: their kernels and the programmatic
    dependencies between them) into one CUDA graph and check one replay."""
    import torch
    import w4a4_mxfp4_quantized_02_b300 as mq
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        fn()
    g.replay()
    torch.cuda.synchronize()
    status = mq.macaq_check_device_error()
    if status != 0:
        raise RuntimeError(f"device error in a graph replay: {mq.macaq_status_string(status)}")
    return g


# The sources each kernel family is compiled from: a recorded DRAM traffic
# figure is used only while the hash of its kernel's sources is unchanged.
KERNEL_SOURCES = {
    "gemm_mxf4_pair_kernel": ("gemm.cu", "ptx.cuh", "mx_block.cuh", "internal.h"),
    "gemm_mxf4_skinny_kernel": ("gemm.cu", "gemm_skinny.cuh", "ptx.cuh", "internal.h"),
    FUSED_LINEAR_KERNEL: ("gemm.cu", "gemm_skinny.cuh", "ptx.cuh", "mx_block.cuh", "internal.h"),
    "gemm_w4a16_kernel": ("gemm.cu", "gemm_w4a16.cuh", "ptx.cuh", "internal.h"),
    "quant_dense_tma_kernel": ("quant.cu", "mx_block.cuh", "ptx.cuh", "internal.h"),
}


def kernel_source_sha(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "w4a4_mxfp4_quantized_02_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """dram__bytes_read.sum + dram__bytes_write.sum of one launch of `kernel`
    on `workload`, from the ncu record under profiles/, or None when there is
    none or the kernel's sources changed since it was taken."""
    prof = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(prof):
        return None
    with open(prof) as f:
        entries = json.load(f).get("entries", [])
    for e in entries:
        if (e.get("kernel") == kernel and e.get("workload") == workload
                and e.get("source_sha") == kernel_source_sha(kernel)):
            return e.get("dram_bytes_per_launch")
    return None


def mma_probe():
    """Tensor-pipe rate of kind::mxf4 MMAs (M=128, N, K=64) per SM."""
    import torch
    import w4a4_mxfp4_quantized_02_b300 as mq
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    iters = 4000
    print("| N | mode | cycles per 4 MMAs | PFLOP/s (all SMs, at the measured clock) | clock GHz |")
    print("|---|---|---|---|---|")
    names = {0: "MMAs only", 1: "+ 6 scale copies per 4 MMAs", 2: "+ copies + commit"}
    for mode in (0, 1, 2):
        for n in (64, 128, 192, 256):
            out = mq.macaq_debug_mma_rate(n | (mode << 16), iters, sms).cpu().double()
            cyc = out[0:2 * sms:2].median().item()
            ns = out[1:2 * sms:2].median().item()
            flops = sms * 4 * iters * 2 * 128 * n * 64
            print(f"| {n} | {names[mode]} | {cyc / iters:.1f} | {flops / ns / 1e6:.2f} | {cyc / ns:.3f} |")
    return 0


def read_probe():
    """Read bandwidth a library reaches on this GPU, beside the copy peak:
    torch's sum over a bf16 vector (reads only), torch's copy (reads and
    writes), and cuBLAS bf16 products shaped like decode (the weight streamed
    once).  Each timing is the median of 20 runs, L2 flushed before each."""
    import torch
    dev = torch.device("cuda:0")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def timed(fn, iters=20, warm=3):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        evs = []
        for _ in range(iters):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            evs.append((e0, e1))
        torch.cuda.synchronize()
        ts = sorted(a.elapsed_time(b) for a, b in evs)
        return ts[len(ts) // 2] * 1e-3

    print("| operation | bytes (MB) | time (us) | GB/s |")
    print("|---|---|---|---|")
    for mib in (64, 512, 2048):
        n = (mib << 20) // 2
        x = torch.empty(n, dtype=torch.bfloat16, device=dev).normal_()
        y = torch.empty_like(x)
        t = timed(lambda: x.sum(dtype=torch.float32))
        print(f"| torch sum, {mib} MiB bf16 (read) | {2 * n / 1e6:.1f} | {t * 1e6:.1f} | {2 * n / t / 1e9:.0f} |")
        t = timed(lambda: y.copy_(x))
        print(f"| torch copy, {mib} MiB bf16 (read + write) | {4 * n / 1e6:.1f} | {t * 1e6:.1f} | "
              f"{4 * n / t / 1e9:.0f} |")
        del x, y
    for (m, n, k) in ((16, 6400, 5120), (16, 25600, 5120), (16, 51200, 5120)):
        w = torch.empty(n, k, dtype=torch.bfloat16, device=dev).normal_()
        a = torch.empty(m, k, dtype=torch.bfloat16, device=dev).normal_()
        t = timed(lambda: a @ w.t())
        print(f"| cuBLAS bf16 [{m}, {k}] x [{n}, {k}]^T (weight read once) | {n * k * 2 / 1e6:.1f} | "
              f"{t * 1e6:.1f} | {n * k * 2 / t / 1e9:.0f} |")
        del w, a
    return 0


PER_CONFIG = ("attn", "attn_qkv", "decode_m1", "decode_m8", "decode_m16", "moe")


def _summary(line: dict) -> dict:
    """The device-timed part of a configuration's line."""
    keep_r = ("bound", "kernel", "achieved", "peak", "unit", "frac", "avg_launch_us", "tflops")
    keep_q = ("kernel", "achieved", "unit", "frac", "avg_launch_us", "bytes_per_launch")
    out = {"workload": line["config"]["workload"], "value": line["value"], "unit": line["unit"],
           "ms_per_step": line["ms_per_step"], "steps": line["steps"],
           "eager_delay_ms": line.get("eager_delay_ms", 0.0),
           "roofline": {k: v for k, v in line["roofline"].items() if k in keep_r},
           "act_quant": {k: v for k, v in line["act_quant"].items() if k in keep_q}}
    for k in ("down_gemm", "combine"):
        if k in line:
            out[k] = line[k]
    return out


def per_config_table(args, rank: int, world: int) -> dict:
    """Device timing of the other configurations (same steps and warm-up, no
    end-to-end leg and no CPU baseline), one after another on this GPU."""
    import torch

    table = {}
    for name in PER_CONFIG:
        if name.startswith("moe"):
            line = gpu_arm_moe(args, rank, world, config=name, light=True)
        else:
            line = gpu_arm(args, rank, world, config=name, light=True)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        if line is not None:
            table[name] = _summary(line)
    return table


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["macaq", "reference"], default="macaq")
    ap.add_argument("--config", default="down",
                    help="workload of the line: down (default: prefill MLP down-projection, the "
                         "largest single-GPU configuration), attn, attn_qkv, decode_m1/m8/m16, tiny, moe")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--moe-unfused", action="store_true",
                    help="moe: the gate+up GEMM writes bf16 gate|up and a separate kernel forms the down input")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the device-timed table of the other configurations")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--hadamard-block", type=int, choices=[32, 64], default=32,
                    help="Hadamard block of the transform (dense workloads)")
    ap.add_argument("--fused-swiglu", action="store_true",
                    help="down: feed the gate|up matrix and fuse SiLU(gate) * up into the transform")
    ap.add_argument("--precision", choices=["w4a4", "w4a16"], default="w4a4",
                    help="w4a16: the weight-only fallback (dense workloads)")
    ap.add_argument("--stage", choices=["layer", "flip"], default="layer",
                    help="flip: time the offline weight preparation with Flip Refinement")
    ap.add_argument("--sweeps", type=int, default=2, help="Flip Refinement passes")
    ap.add_argument("--damp", type=float, default=0.0, help="Flip Refinement diagonal damping")
    ap.add_argument("--cpu-rows", type=int, default=64, help="weight rows the oracle refines")
    ap.add_argument("--no-graphs", action="store_true",
                    help="launch every step eagerly instead of replaying a captured CUDA graph")
    ap.add_argument("--kernel-events-every", type=int, default=4,
                    help="bracket the kernels of every n-th timed step with CUDA events")
    ap.add_argument("--probe", choices=["mma", "read"], help="print a hardware probe table and exit")
    args = ap.parse_args()
    if args.probe == "mma":
        return mma_probe()
    if args.probe == "read":
        return read_probe()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        if args.stage == "flip":
            return gpu_arm_flip(args, rank, world)
        if args.precision == "w4a16":
            return gpu_arm_w4a16(args, rank, world)
        if args.config.startswith("moe"):
            line = gpu_arm_moe(args, rank, world)
        else:
            line = gpu_arm(args, rank, world)
            if (not args.no_per_config and args.config == "down" and args.hadamard_block == 32
                    and not args.fused_swiglu):
                table = per_config_table(args, rank, world)
                if line is not None:
                    line["per_config"] = table
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
