"""Benchmark of the SageBwd hot path on GB300: one step = quantise + forward + backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--causal]

Workload: the headline configuration, B=2 H=16 N=8192 d=128 fp16, non-causal (``--causal`` for
the causal variant), synthetic seeded inputs (Q, K, V ~ N(0,1), dO ~ N(0,1e-4)); each rank under
torchrun processes its own batch (weak scaling, no data-path collective).

Metric: effective TOPS = 14 B H N^2 d / step time (the 6 integer GEMMs and the 16-bit dP GEMM
of forward + backward; halved when causal).  One JSON line on rank 0 carries the device-timed
value, the end-to-end value through the public API with host buffers (``e2e``), the roofline of
the dominant call, the clocks seen during the timed region, the number of library kernels
launched, and the CPU oracle timed on a bounded sample (``cpu_baseline``).

``--impl reference`` times the CPU oracle alone (the reference arm: the method has no published
GPU implementation to run), each step a bounded sample of the same workload.  ``--qat`` times the
Attn-QAT step instead of SageBwd's, with the Attn-QAT oracle as its CPU baseline.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HOST_CORES = len(os.sched_getaffinity(0))
if "reference" in sys.argv:
    # the reference arm times the oracle on every host core this process may use: set the BLAS
    # thread count before numpy loads
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = str(HOST_CORES)

import workloads  # noqa: E402

METRIC = "fwd+bwd effective TOPS (N=8192,d=128) and % of INT8/FP16 tensor-core roofline"
UNIT = "TOPS"
KERNELS_PER_STEP = 4    # quantise pass (it also writes the fp16 operand copies), fwd, bwd prologue, bwd
# The rate of the legacy warp-level integer MMA (mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32),
# the only INT8 tensor-core instruction sm_103a has (ptxas rejects tcgen05 kind::i8 there), as
# measured on GB300 by a probe kernel when the integer GEMMs' instruction was chosen.  It stands in
# for the "INT8 peak" of the literal roofline reading.
INT8_MMA_SYNC_TOPS = 152.0
BURST_REGION_MS = 1000.0  # a timed region shorter than this compares with the burst peak
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "bwd_traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "bit_trainable_attention_sage_gb300", "csrc", f)
                  for f in ("sage_bwd.cu", "sage_device.cuh", "sage_internal.h")]


# ------------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU under torchrun; nothing on the data path)
# ------------------------------------------------------------------------------------------
def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Largest value over all ranks (the slowest rank sets the job time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config_of(w: workloads.Workload) -> dict:
    """The ``config`` object both arms report for a workload."""
    return {"workload": f"{w.name} {w.tag}", "B": w.B, "H": w.H, "N": w.N, "d": w.d,
            "causal": w.causal, "smooth_k": True, "smooth_q": w.smooth_q, "per_rank": "own batch",
            "l2": f"inputs larger than L2 (Q,K,V,dO = {8 * w.B * w.H * w.N * w.d // 2**20} MiB per step)"}


def step_roofline(w: workloads.Workload, step_ms: float, p16_tflops: float) -> dict:
    """The step's combined roofline, t_roof = 12 BHN^2d / P_int + 2 BHN^2d / P_16 (x 1/2 causal),
    read two ways: P_int = the fp16 tcgen05 peak (the instruction the integer GEMMs execute, the
    honest figure) and P_int = the measured legacy INT8 mma.sync rate (the literal INT8 reading)."""
    unit = w.B * w.H * w.N * w.N * w.d * (0.5 if w.causal else 1.0)
    t16 = 14.0 * unit / (p16_tflops * 1e12) * 1e3
    t8 = (12.0 * unit / (INT8_MMA_SYNC_TOPS * 1e12) + 2.0 * unit / (p16_tflops * 1e12)) * 1e3
    return {"fp16_reading": {"p_int_tflops": p16_tflops, "t_roof_ms": round(t16, 4), "frac": round(t16 / step_ms, 4)},
            "int8_literal_reading": {"p_int_tops": INT8_MMA_SYNC_TOPS, "t_roof_ms": round(t8, 4),
                                     "frac": round(t8 / step_ms, 4),
                                     "caveat": "P_int is the legacy mma.sync s8 rate, 12x below the fp16 tcgen05 "
                                               "rate that actually runs the integer GEMMs, so this fraction exceeds 1"}}


def leg_roofline(ops: float, step_ms: float, p16_tflops: float, note: str) -> dict:
    """The roofline of a leg with no INT8 GEMM (the FP4 forward on dequantised fp16 operands, the
    16-bit Attn-QAT step): its own tensor ops at the fp16 rate."""
    t16 = ops / (p16_tflops * 1e12) * 1e3
    return {"fp16_reading": {"p_int_tflops": p16_tflops, "t_roof_ms": round(t16, 4), "frac": round(t16 / step_ms, 4)},
            "note": note}


def step_ops(w: workloads.Workload) -> float:
    """Algorithmic tensor ops of one quantise + forward + backward: 14 B H N^2 d (x 1/2 causal)."""
    ops = 14.0 * w.B * w.H * w.N * w.N * w.d
    return ops / 2 if w.causal else ops


def qknorm_bwd_bytes(w: workloads.Workload) -> int:
    """Algorithmic HBM bytes of one sage_qknorm_bwd call: X read (2 B an element), dY read and dX
    written (4 B each), the row factors read (4 B a row)."""
    n = w.B * w.H * w.N * w.d
    return 10 * n + 4 * w.B * w.H * w.N


def quant_bytes(w: workloads.Workload, ops16: bool = True) -> int:
    """Algorithmic HBM bytes of one sage_quantize_smooth call: Q, K, V read once (2 B an element),
    int8 codes written (1 B) and, with the operand copies (SAGE_FLAG_OPS16, the binding's default),
    their fp16 values (2 B), plus the float32 block scales and means.  The K-mean phase reads K a
    second time, but that read comes from L2 (K of the headline workload is 64 MiB of a 126 MiB
    L2), so it is not counted: the minimum DRAM traffic of the call."""
    n = w.B * w.H * w.N * w.d
    reads = 2 * n * 3
    writes = 3 * n + (6 * n if ops16 else 0)
    small = 4 * (3 * w.B * w.H * (w.N // 64) + w.B * w.H * w.d
                 + (w.B * w.H * (w.N // 64) * w.d if w.smooth_q else 0))
    return reads + writes + small


def qat_step_ops(w: workloads.Workload) -> float:
    """Algorithmic tensor ops of one Attn-QAT step: forward S, P^ V' and the high-precision
    P~ V' (6 B H N^2 d), backward S, dP, dV, dK, dQ (10 B H N^2 d); x 1/2 causal."""
    ops = 16.0 * w.B * w.H * w.N * w.N * w.d
    return ops / 2 if w.causal else ops


def bwd_ops(w: workloads.Workload) -> float:
    ops = 10.0 * w.B * w.H * w.N * w.N * w.d
    return ops / 2 if w.causal else ops


def fwd_ops(w: workloads.Workload) -> float:
    ops = 4.0 * w.B * w.H * w.N * w.N * w.d
    return ops / 2 if w.causal else ops


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self, path: str):
        self.path = path
        try:
            self.fh = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------------------
# the GPU arm
# ------------------------------------------------------------------------------------------
def source_sha() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(w) -> float | None:
    """DRAM bytes per launch of the backward kernel from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    try:
        rec = json.load(open(PROFILE_TRAFFIC))
    except (OSError, ValueError):
        return None
    if rec.get("source_sha") != source_sha():
        return None
    scale = (w.B * w.H) / rec["heads"] * (w.N / rec["N"]) ** 2 if rec.get("scale_with_work") else 1.0
    return rec["dram_bytes_per_launch"] * scale


def run_gpu(args, w: workloads.Workload):
    import numpy as np
    import torch
    import bit_trainable_attention_sage_gb300 as sg

    rank, world, local = rank_info()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    x = workloads.make_inputs(w, seed=rank)
    dt = torch.float16 if w.dtype == "fp16" else torch.bfloat16
    host = {k: torch.from_numpy(v).to(dt).pin_memory() for k, v in x.items()}
    del x
    dev = {k: v.to(device) for k, v in host.items()}
    stream = torch.cuda.current_stream(device)
    B, H, N, d = w.B, w.H, w.N, w.d

    # outputs and workspaces allocated once (the library allocates nothing)
    p = sg.make_params(B, H, N, d, 0 if w.dtype == "fp16" else 1, w.causal, fp8=args.fp8)
    import ctypes
    L = sg.lib()
    ws_f = torch.empty(L.sage_fwd_workspace_bytes(ctypes.byref(p)), dtype=torch.uint8, device=device)
    pb = sg.make_params(B, H, N, d, 0 if w.dtype == "fp16" else 1, w.causal, smooth_q=w.smooth_q,
                        fp8=args.fp8)
    if args.dp_int8:
        pb.flags |= sg.binding.SAGE_FLAG_DP_INT8
    ws_b = torch.empty(L.sage_bwd_workspace_bytes(ctypes.byref(pb)), dtype=torch.uint8, device=device)
    O = torch.empty((B, H, N, d), dtype=dt, device=device)
    Lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    grads = tuple(torch.empty((B, H, N, d), dtype=torch.float32, device=device) for _ in range(3))

    gam = None
    if args.qk_norm:
        gen = torch.Generator(device="cpu").manual_seed(rank)
        gam = [(0.5 + torch.rand(d, generator=gen)).to(device) for _ in range(2)]

    if args.fp4:
        # the FP4 leg is an inference forward: no dO
        host.pop("dO")
        dev.pop("dO")
    if args.qat:
        # Attn-QAT intermediates, shared by both buffer sets (one compute stream orders the steps)
        qat_f = tuple(torch.empty((B, H, N, d), dtype=dt, device=device) for _ in range(3))
        qat_op = torch.empty((B, H, N, d), dtype=torch.float32, device=device)
        qat_r = torch.empty((B, H, N // 64, N), dtype=torch.float32, device=device)
        pq = sg.make_params(B, H, N, d, 0 if w.dtype == "fp16" else 1, w.causal, smooth_k=False)
        ws_q = torch.empty(L.sage_qat_bwd_workspace_bytes(ctypes.byref(pq)), dtype=torch.uint8, device=device)
    # buffer set 0: the device-timed steps; sets 0 and 1 alternate in the pipelined end-to-end loop
    set0 = {"dev": dev, "O": O, "Lse": Lse, "grads": grads}

    def step(ev=None, bs=None):
        bs = set0 if bs is None else bs
        dev, O, Lse, grads = bs["dev"], bs["O"], bs["Lse"], bs["grads"]
        if ev is not None:
            ev[0].record(stream)
        if args.qat:
            sg.sage_qat_quantize(dev["Q"], dev["K"], dev["V"], out=qat_f)
            if ev is not None:
                ev[1].record(stream)
            sg.sage_qat_fwd(*qat_f, causal=w.causal, out=(O, qat_op, Lse, qat_r))
            if ev is not None:
                ev[2].record(stream)
            sg.sage_qat_bwd(*qat_f, qat_op, Lse, qat_r, dev["dO"], causal=w.causal, grads=grads, workspace=ws_q)
            if ev is not None:
                ev[3].record(stream)
                ev[4].record(stream)
            return
        if args.fp4:
            q4 = sg.sage_quantize_fp4(dev["Q"], dev["K"], dev["V"], smooth_q=w.smooth_q)
            if ev is not None:
                ev[1].record(stream)
            sg.sage_attn_fwd_fp4(q4, causal=w.causal, out=O, lse=Lse, workspace=ws_f)
            if ev is not None:
                for e in ev[2:]:
                    e.record(stream)
            return
        if args.qk_norm:
            q = sg.sage_quantize_smooth_qknorm(dev["Q"], dev["K"], dev["V"], gamma_q=gam[0], gamma_k=gam[1],
                                               smooth_q=w.smooth_q, fp8=args.fp8)
        else:
            q = sg.sage_quantize_smooth(dev["Q"], dev["K"], dev["V"], smooth_q=w.smooth_q, fp8=args.fp8)
        if ev is not None:
            ev[1].record(stream)
        sg.sage_attn_fwd(q, causal=w.causal, out=O, lse=Lse, workspace=ws_f)
        if ev is not None:
            ev[2].record(stream)
        sg.sage_attn_bwd(q, dev["V"], O, Lse, dev["dO"], causal=w.causal, grads=grads, workspace=ws_b,
                         dp_int8=args.dp_int8)
        if ev is not None:
            ev[3].record(stream)
        if args.qk_norm:
            # the attention gradients are those of the normalised Q and K: chain them through the norm
            sg.sage_qknorm_bwd(dev["Q"], q.rQ, grads[0], gamma=gam[0])
            sg.sage_qknorm_bwd(dev["K"], q.rK, grads[1], gamma=gam[1])
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    st = sg.sage_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {sg.sage_status_string(st)}")

    # ---- device-timed region -------------------------------------------------------------
    clocks = ClockSampler(local)
    if args.clock_log:
        clock_path = f"{args.clock_log}.rank{rank}.csv"
        os.makedirs(os.path.dirname(os.path.abspath(clock_path)), exist_ok=True)
    else:
        fd, clock_path = tempfile.mkstemp(prefix="sage_clocks_", suffix=".csv")
        os.close(fd)
    clocks.start(clock_path)
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize(device)
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    ms = t0.elapsed_time(t1)
    clk = clocks.stop()
    st = sg.sage_device_status()
    if st != 0:
        raise RuntimeError(f"device status after timing: {sg.sage_status_string(st)}")
    quant_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    fwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    bwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    qkn_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in evs) if args.qk_norm else 0.0
    ms_max = max_over_ranks(dist, ms, device)

    # ---- end to end through the public API with host buffers ------------------------------
    host_out = {"O": torch.empty_like(O, device="cpu").pin_memory()}
    if not args.fp4:
        host_out.update({"dQ": torch.empty_like(grads[0], device="cpu").pin_memory(),
                         "dK": torch.empty_like(grads[1], device="cpu").pin_memory(),
                         "dV": torch.empty_like(grads[2], device="cpu").pin_memory()})
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    # Pipelined over steps through two buffer sets and two copy streams: step k + 1's inputs are
    # copied in (pinned host -> device) while step k computes, and step k's results are copied out
    # while step k + 1 computes.  Every step still moves its own inputs and results across the
    # host link inside the timed region; a set is reused only after its copies have finished.
    set1 = {"dev": {k: torch.empty_like(v) for k, v in dev.items()}, "O": torch.empty_like(O),
            "Lse": torch.empty_like(Lse), "grads": tuple(torch.empty_like(g) for g in grads)}
    sets = (set0, set1)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def e2e_run(nsteps: int, start_ev=None):
        ev_in = [torch.cuda.Event() for _ in range(nsteps)]
        ev_comp = [torch.cuda.Event() for _ in range(nsteps)]
        ev_out = [torch.cuda.Event() for _ in range(nsteps)]
        for k in range(nsteps):
            bs = sets[k & 1]
            with torch.cuda.stream(s_in):
                if k == 0 and start_ev is not None:
                    s_in.wait_event(start_ev)
                if k >= 2:
                    s_in.wait_event(ev_comp[k - 2])           # step k - 2 has read this set's inputs
                for key in bs["dev"]:
                    bs["dev"][key].copy_(host[key], non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if k >= 2:
                stream.wait_event(ev_out[k - 2])              # this set's results have left
            step(bs=bs)
            ev_comp[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[k])
                host_out["O"].copy_(bs["O"], non_blocking=True)
                if not args.fp4:
                    for name, g in zip(("dQ", "dK", "dV"), bs["grads"]):
                        host_out[name].copy_(g, non_blocking=True)
                ev_out[k].record(s_out)
        stream.wait_event(ev_out[nsteps - 1])

    e2e_run(max(2, args.warmup // 2))
    barrier(dist, device)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps, start_ev=e0)
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1), device)
    assert np.isfinite(host_out["O" if args.fp4 else "dQ"].float().numpy()).all()

    ops = fwd_ops(w) if args.fp4 else (qat_step_ops(w) if args.qat else step_ops(w))
    value = world * ops * args.steps / (ms_max * 1e-3) / 1e12
    e2e_value = world * ops * args.steps / (e2e_ms * 1e-3) / 1e12

    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    # the timed region's length decides which measured peak applies: burst for a sub-second region
    burst = ms_max < BURST_REGION_MS
    if peaks:
        peak = peaks["bf16_tflops"] if burst else peaks["bf16_tflops_sustained"]
        peak_src = (f"of measured ({'bf16_tflops, burst' if burst else 'bf16_tflops_sustained'}: timed region "
                    f"{ms_max:.0f} ms; fp16 runs at the bf16 rate)")
    else:
        peak = 1900.0 if burst else 1700.0
        peak_src = f"of fallback ({'burst' if burst else 'sustained'})"
    bwd_tflops = bwd_ops(w) / (bwd_ms * 1e-3) / 1e12 if bwd_ms > 0 else 0.0
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    quant_gbs = quant_bytes(w) / (quant_ms * 1e-3) / 1e9
    fwd_tflops = (1.5 if args.qat else 1.0) * fwd_ops(w) / (fwd_ms * 1e-3) / 1e12
    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3" if args.fp8 else "s8") + " codes as f16 (f32 accumulate); dP "
                 + ("s8 codes (ablation)" if args.dp_int8 else "f16"),
        "data": "synthetic",
        "config": config_of(w),
        "roofline": {"kernel": "sage_attn_bwd call (bwd prologue + tcgen05 backward kernel)",
                     "bound": "tensor", "achieved": round(bwd_tflops, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "TFLOP/s", "frac": round(bwd_tflops / peak, 4),
                     "traffic": profiled_traffic(w), "flops_per_launch": bwd_ops(w)},
        "fwd_call": {"ms": round(fwd_ms, 4), "tflops": round(fwd_tflops, 1), "frac": round(fwd_tflops / peak, 4)},
        "bwd_call": {"ms": round(bwd_ms, 4), "tflops": round(bwd_tflops, 1), "frac": round(bwd_tflops / peak, 4)},
        "quantise_call": {"ms": round(quant_ms, 4), "bound": "hbm", "bytes": quant_bytes(w),
                          "gbs": round(quant_gbs, 1), "peak_gbs": hbm_peak,
                          "frac": round(quant_gbs / hbm_peak, 4)},
        "step_frac_of_fp16_peak": round(value / world / peak, 4),
        "step_roofline": step_roofline(w, ms_max / args.steps, peak),
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "mode": "pinned host buffers; copies of step k+1 in and step k-1 out overlap step k"},
        "gpu_launches": (KERNELS_PER_STEP + (2 if args.qk_norm else 0) + (2 if args.dp_int8 else 0)) * args.steps,
        "clocks": clk,
    }
    if args.qk_norm:
        # two gradient calls (Q and K) per step; the prologue's cost is inside quantise_call
        gbs = 2 * qknorm_bwd_bytes(w) / (qkn_ms * 1e-3) / 1e9
        line["qknorm_bwd_calls"] = {"ms": round(qkn_ms, 4), "bound": "hbm", "bytes": 2 * qknorm_bwd_bytes(w),
                                    "gbs": round(gbs, 1), "peak_gbs": hbm_peak, "frac": round(gbs / hbm_peak, 4)}
        line["config"]["qk_norm"] = True
    if args.fp4:
        # the FP4 leg times quantise + forward only: its value is forward TOPS
        line["metric"] = "SageAttention3 FP4 inference forward TOPS (N=8192,d=128)"
        line["dtype"] = "NVFP4 (e2m1 codes, e4m3 scales per 16) dequantised to f16 (f32 accumulate)"
        line["config"]["fp4_forward"] = True
        line["roofline"] = {"kernel": "sage_attn_fwd_fp4 call (widen + tcgen05 forward kernel)",
                            "bound": "tensor", "achieved": round(fwd_tflops, 1), "peak": peak,
                            "peak_source": peak_src, "unit": "TFLOP/s", "frac": round(fwd_tflops / peak, 4),
                            "traffic": None, "flops_per_launch": fwd_ops(w)}
        line.pop("bwd_call", None)
        line["step_roofline"] = leg_roofline(fwd_ops(w), ms_max / args.steps, peak,
                                             "quantise + forward only: the forward's 4 N^2 d at the fp16 rate")
        line["gpu_launches"] = 6 * args.steps        # K-mean, FP4 quantise, 3 widen, forward
    if args.qat:
        line["metric"] = "Attn-QAT fwd+bwd effective TOPS (N=8192,d=128)"
        line["dtype"] = ("NVFP4 fake-quantised Q, K, V and P in " + w.dtype + " operands (f32 accumulate); "
                         "16-bit backward")
        line["config"]["qat"] = True
        line["config"]["smooth_k"] = False
        line["roofline"] = {"kernel": "sage_qat_bwd call (prologue + tcgen05 backward kernel)",
                            "bound": "tensor", "achieved": round(bwd_tflops, 1), "peak": peak,
                            "peak_source": peak_src, "unit": "TFLOP/s", "frac": round(bwd_tflops / peak, 4),
                            "traffic": None, "flops_per_launch": bwd_ops(w)}
        line["fwd_call"]["note"] = "two forward passes (O and L, then O'); tflops counts the 6 N^2 d of the method"
        line["quantise_call"] = {"ms": round(quant_ms, 4), "bound": "hbm", "bytes": 12 * w.B * w.H * w.N * w.d,
                                 "gbs": round(12 * w.B * w.H * w.N * w.d / (quant_ms * 1e-3) / 1e9, 1),
                                 "peak_gbs": hbm_peak}
        line["quantise_call"]["frac"] = round(line["quantise_call"]["gbs"] / hbm_peak, 4)
        line["step_roofline"] = leg_roofline(qat_step_ops(w), ms_max / args.steps, peak,
                                             "16-bit operands throughout: the method's 16 N^2 d at the fp16 rate")
        line["gpu_launches"] = 5 * args.steps        # fake quantise, 2 forward passes, prologue, backward
    return line


# ------------------------------------------------------------------------------------------
# the CPU oracle (baseline leg and the reference arm)
# ------------------------------------------------------------------------------------------
def oracle_sample(w: workloads.Workload, q_blocks, kv_blocks, seed: int = 0) -> tuple[float, float]:
    """Time the oracle on head (0, 0) of the workload: quantise, forward over ``q_blocks`` (None =
    all) and backward over ``kv_blocks`` (None = all).  Returns (seconds, algorithmic ops)."""
    import numpy as np
    from oracle import sage as osage
    x = workloads.make_inputs(w, seed=seed, heads=1)
    x = {k: np.ascontiguousarray(v[:1]) for k, v in x.items()}
    T = w.N // 64
    qb = list(range(T)) if q_blocks is None else list(q_blocks)
    kb = list(range(T)) if kv_blocks is None else list(kv_blocks)
    t0 = time.perf_counter()
    prep = osage.prepare(x["Q"], x["K"], x["V"], smooth_q=w.smooth_q)
    prep["V16"] = x["V"]
    O, L = osage.sage_forward(prep, w.causal, q_blocks=None if q_blocks is None else qb)
    Os = workloads.round_to(O.astype(np.float32), w.dtype)
    if kv_blocks is None:
        osage.sage_backward(prep, Os, L.astype(np.float32), x["dO"], w.causal)
    else:
        osage.sage_backward(prep, Os, L.astype(np.float32), x["dO"], w.causal, kv_blocks=kb)
    secs = time.perf_counter() - t0
    tile = 64 * 64 * w.d
    n_f = sum((i + 1) if w.causal else T for i in qb)
    n_b = sum((T - j) if w.causal else T for j in kb)
    return secs, 4.0 * tile * n_f + 10.0 * tile * n_b


def qat_oracle_sample(w: workloads.Workload, q_blocks, kv_blocks, seed: int = 0) -> tuple[float, float]:
    """Time the Attn-QAT oracle on head (0, 0): fake quantisation, the whole forward (the backward
    needs O', L and R of every row) and the backward over ``kv_blocks`` (None = all).
    Returns (seconds, algorithmic ops)."""
    import numpy as np
    from oracle import qat as oqat
    x = workloads.make_inputs(w, seed=seed, heads=1)
    x = {k: np.ascontiguousarray(v[:1, :1]) for k, v in x.items()}
    T = w.N // 64
    kb = list(range(T)) if kv_blocks is None else list(kv_blocks)
    rnd = lambda a: workloads.round_to(a, w.dtype)
    t0 = time.perf_counter()
    fq = oqat.fake_quant(x["Q"], x["K"], x["V"])
    O, Op, L, R = oqat.qat_forward(fq, w.causal, rnd)
    oqat.qat_backward(fq, Op.astype(np.float32), L.astype(np.float32), R, x["dO"], w.causal, rnd,
                      kv_blocks=None if kv_blocks is None else kb, q_blocks=None if kv_blocks is None else [])
    secs = time.perf_counter() - t0
    tile = 64 * 64 * w.d
    n_f = sum((i + 1) if w.causal else T for i in range(T))
    n_b = sum((T - j) if w.causal else T for j in kb)
    return secs, 6.0 * tile * n_f + 10.0 * tile * n_b


def regime_sample(w: workloads.Workload, seed: int = 0, rows: int = 128) -> dict:
    """RMS of P, dP and dS of float64 full-precision attention (the oracle's FPA) on the first and
    last ``rows`` // 2 query rows of head (0, 0), every key: how close the synthetic workload comes
    to the gradient magnitudes the pages report for trained models (their dS near 1e-7)."""
    import numpy as np
    from oracle import fpa
    x = workloads.make_inputs(w, seed=seed, heads=1)
    Q, K, V, dO = (np.asarray(x[k][0, 0], np.float64) for k in ("Q", "K", "V", "dO"))
    h = rows // 2
    idx = np.r_[0:h, w.N - h:w.N]
    S = Q[idx] @ K.T / math.sqrt(w.d)
    if w.causal:
        S = np.where(np.arange(w.N)[None, :] > idx[:, None], -np.inf, S)
    P = fpa.softmax_rows(S)
    dP = dO[idx] @ V.T
    D = (P * dP).sum(axis=1, keepdims=True)
    dS = P * (dP - D)
    rms = lambda a: float(np.sqrt(np.mean(a * a)))
    return {"rms_P": rms(P), "rms_dP": rms(dP), "rms_dS": rms(dS),
            "sample": f"head (0,0), query rows 0-{h - 1} and {w.N - h}-{w.N - 1}, every key, float64 FPA"}


def cpu_baseline_subprocess(w: workloads.Workload, q_blocks, kv_blocks, label: str, fn: str = "oracle_sample") -> dict:
    """Run the oracle in a fresh interpreter with one BLAS thread per host core this process may use,
    and describe the sample."""
    n = str(HOST_CORES)
    env = dict(os.environ, OMP_NUM_THREADS=n, OPENBLAS_NUM_THREADS=n, MKL_NUM_THREADS=n)
    code = ("import json, sys; sys.path.insert(0, %r); import bench, workloads; "
            "w = workloads.get(%r, causal=%r); s, ops = bench.%s(w, %r, %r); "
            "print(json.dumps({'s': s, 'ops': ops, 'regime': bench.regime_sample(w)}))"
            % (ROOT, w.name, w.causal, fn, q_blocks, kv_blocks))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": HOST_CORES, "kind": "oracle", "sample": label,
                "error": r.stderr[-300:]}
    out = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": round(out["ops"] / out["s"] / 1e12, 8), "unit": UNIT, "cores": HOST_CORES,
            "threads": f"BLAS threads = {HOST_CORES} (the host cores this process may use)",
            "kind": "oracle", "sample": label, "seconds": round(out["s"], 2), "regime": out["regime"]}


def run_reference(args, w: workloads.Workload):
    """The reference arm: the CPU oracle as it stands, each step a bounded sample."""
    rank, world, _ = rank_info()
    if rank != 0:
        return None
    qb = list(range(4))
    kb = list(range(4))
    label = f"head (0,0) of the workload; forward over 4 of {w.N // 64} query blocks and backward " \
            f"over 4 of {w.N // 64} key blocks per step"
    for _ in range(args.warmup):
        oracle_sample(w, qb, kb)
    secs = ops = 0.0
    for _ in range(args.steps):
        s, o = oracle_sample(w, qb, kb)
        secs += s
        ops += o
    value = ops / secs / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 8), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 oracle (f32 codes)",
        "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": round(value, 8), "unit": UNIT, "cores": HOST_CORES, "kind": "oracle",
                         "sample": label, "threads": f"BLAS threads = {HOST_CORES}"},
        "e2e": {"value": round(value, 8), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--dp-int8", action="store_true",
                    help="backward with the INT8-dP ablation (dP from the dO and V codes)")
    ap.add_argument("--fp8", action="store_true",
                    help="the FP8 SageBwd variant (E4M3 codes in place of INT8)")
    ap.add_argument("--qk-norm", action="store_true",
                    help="QK-norm fused into the quantise call, and its gradient after the backward")
    ap.add_argument("--fp4", action="store_true",
                    help="the SageAttention3 FP4 inference forward (quantise + forward only)")
    ap.add_argument("--qat", action="store_true",
                    help="the Attn-QAT training step (NVFP4 fake quantisation, O', 16-bit backward)")
    ap.add_argument("--workload", default="headline", choices=["headline", "qknorm", "outlier", "longseq"],
                    help="the workload (default: the headline B2 H16 N8192 d128 fp16); the others are the "
                         "parity workloads of workloads.py, timed the same way")
    ap.add_argument("--clock-log", default=None,
                    help="keep the nvidia-smi clock samples of the timed region in PATH.rank<r>.csv "
                         "(default: a temporary file)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling of a smaller case)")
    ap.add_argument("--heads", type=int, default=None, help="override H (profiling of a smaller case)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    over = {"causal": True} if args.causal else {}
    if args.batch:
        over["B"] = args.batch
    if args.heads:
        over["H"] = args.heads
    w = workloads.get(args.workload, **over)
    if args.impl == "reference":
        line = run_reference(args, w)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    from __graft_entry__ import build
    build()
    line = run_gpu(args, w)
    if line is None:
        return
    rank, world, _ = rank_info()
    if not args.no_cpu_baseline and world == 1 and args.qat:
        line["cpu_baseline"] = cpu_baseline_subprocess(
            w, None, [0, 1], "head (0,0) of 32: fake quantisation, the whole forward and the backward over 2 of "
                             f"{w.N // 64} key blocks, value = their 6 / 10 x 64^2 d ops per tile / CPU seconds",
            fn="qat_oracle_sample")
    elif not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline_subprocess(
            w, None, None, "head (0,0) of 32: full quantise + forward + backward of one head, "
                           "value = its 14 N^2 d ops / CPU seconds")
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
