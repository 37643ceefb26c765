"""Benchmark of the FP8 block-scaled GEMM hot path on GB300 (one JSON line on stdout).

A step is one pass of the whole hot path over one batch of synthetic inputs: for each
workload of the suite, the activations' scale factors are packed on the GPU
(dg_pack_sf_ue8m0) and the GEMM runs (dense, contiguous-grouped or masked-grouped).  The
weights' scale factors are packed once, when the weights are set up (the packed layout is a
one-time transform of a static tensor), and stay resident like the weights.  The suite
(shapes from the DeepGEMM article's H800 tables):
    decode 64x2112x7168, 128x24576x1536, 128x7168x2048, 64x4096x7168  (dense, A with 1 % x20 outliers)
    prefill 4096x7168x16384                                            (dense)
    contiguous MoE: 4 experts, N=4096, K=7168, 32768 tokens (multinomial), segments padded to 128
    masked MoE: 4 groups, max_m=256, N=7168, K=2048, masked_m ~ U{1..256}
value = total valid FLOPs of all GEMMs / device time, in TFLOPS.

The small dense GEMM 128x512x1024 is timed beside the step as its own latency-bound row
(`workloads`, marked "in_value": false): it is not part of `value`.

L2: every GEMM's operands were last touched one step earlier, and one step streams about
1 GB, far more than the 129 MB L2, so every timed GEMM reads cold operands.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --impl reference the CPU oracle (float64 numpy) is timed instead, on a bounded sample
of the same workloads, on the host's cores.  Under torchrun (N > 1) every rank runs the
suite on its own GPU (independent replicas, weak scaling) and rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "FP8 block-scaled GEMM TFLOPS (dense+grouped) and % of GB300 FP8 peak"
WORKLOAD_NAME = ("fp8 block-scaled GEMM suite: decode 64x2112x7168, 128x24576x1536, 128x7168x2048, "
                 "64x4096x7168; prefill 4096x7168x16384; contiguous MoE 4x(32768 tok)x4096x7168; "
                 "masked MoE 4x256x7168x2048")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor ratio (4.5 / 2.25 PFLOP/s)
MMA_MACS_PER_CLK_SM = 8192   # FP8 block-scaled MMA rate of one SM, measured on GB300


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

def make_workloads(seed: int = 0):
    ws = []
    for i, (M, N, K) in enumerate(synth.DECODE_SHAPES):
        w = synth.make_dense(M, N, K, seed=seed + i, a_outliers=True, b_std=0.02)
        w["name"] = f"decode_{M}x{N}x{K}"
        ws.append(w)
    M, N, K = synth.PREFILL_SHAPE
    w = synth.make_dense(M, N, K, seed=seed + 10, b_std=0.02)
    w["name"] = f"prefill_{M}x{N}x{K}"
    ws.append(w)
    c = synth.CONTIGUOUS
    w = synth.make_contiguous(c["G"], c["N"], c["K"], c["tokens"], seed=seed + 20)
    w["name"] = f"contiguous_{c['G']}x{c['tokens']}tok_x{c['N']}x{c['K']}"
    ws.append(w)
    m = synth.MASKED
    w = synth.make_masked(m["G"], m["max_m"], m["N"], m["K"], seed=seed + 30)
    w["name"] = f"masked_{m['G']}x{m['max_m']}x{m['N']}x{m['K']}"
    ws.append(w)
    for w in ws:
        w["valid_rows"] = _valid_rows(w)
        w["flops"] = 2.0 * w["valid_rows"] * w["N"] * w["K"]
        w["bytes"] = _algorithmic_bytes(w)
    return ws


def suite_config(ws, world: int) -> dict:
    """The `config` object of the JSON line; both arms print the same one."""
    return {"workload": WORKLOAD_NAME, "flops_per_step": sum(w["flops"] for w in ws),
            "bytes_per_step": sum(w["bytes"] for w in ws),
            "weights": "packed weight scales resident (packed once at set-up); activation scales packed every step",
            "l2": "cold operands: each GEMM's inputs were last touched one step earlier and a step "
                  "streams ~1 GB (> 129 MB L2)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def _valid_rows(w) -> int:
    if w["kind"] == "dense":
        return w["M"]
    if w["kind"] == "contiguous":
        return int(np.sum(w["m_indices"] >= 0))
    return int(np.sum(w["masked_m"]))


def _algorithmic_bytes(w) -> float:
    """FP8 A (valid rows) + FP8 B (groups used) + BF16 D (valid rows) + packed scales."""
    N, K = w["N"], w["K"]
    rows = w["valid_rows"]
    kp = (K // 128 + 3) // 4
    if w["kind"] == "dense":
        groups = 1
        sf = 4 * kp * (synth.align_up(w["M"], 4) + synth.align_up(N, 4))
    elif w["kind"] == "contiguous":
        groups = int(np.sum(w["counts"] > 0))
        sf = 4 * kp * (synth.align_up(w["M_sum"], 4) + groups * synth.align_up(N, 4))
    else:
        groups = int(np.sum(w["masked_m"] > 0))
        sf = 4 * kp * groups * (synth.align_up(w["max_m"], 4) + synth.align_up(N, 4))
    return float(rows * K + groups * N * K + 2 * rows * N + sf)


class DeviceWorkload:
    """Device-resident operands and outputs of one workload, plus its launch."""

    def __init__(self, w, dev):
        import moe_grouped_gemm_02_gb300 as dg
        self.dg = dg
        self.w = w
        self.kind = w["kind"]
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        self.a = t(w["a"])
        self.b = t(w["b"])
        self.sfa_f = t(w["sfa"])
        self.sfb_f = t(w["sfb"])
        N, K = w["N"], w["K"]
        if self.kind == "dense":
            self.rows_a = w["M"]
            self.sfa = torch.empty(dg.packed_sf_shape(None, w["M"], K), dtype=torch.int32, device=dev)
            self.sfb = torch.empty(dg.packed_sf_shape(None, N, K), dtype=torch.int32, device=dev)
            self.d = torch.empty((w["M"], N), dtype=torch.bfloat16, device=dev)
        elif self.kind == "contiguous":
            self.rows_a = w["M_sum"]
            self.sfa = torch.empty(dg.packed_sf_shape(None, w["M_sum"], K), dtype=torch.int32, device=dev)
            self.sfb = torch.empty(dg.packed_sf_shape(w["G"], N, K), dtype=torch.int32, device=dev)
            self.d = torch.empty((w["M_sum"], N), dtype=torch.bfloat16, device=dev)
            self.idx = t(w["m_indices"])
        else:
            self.rows_a = w["max_m"]
            self.sfa = torch.empty(dg.packed_sf_shape(w["G"], w["max_m"], K), dtype=torch.int32, device=dev)
            self.sfb = torch.empty(dg.packed_sf_shape(w["G"], N, K), dtype=torch.int32, device=dev)
            self.d = torch.empty((w["G"], w["max_m"], N), dtype=torch.bfloat16, device=dev)
            self.idx = t(w["masked_m"])
        self.N = N

    def pack_weights(self):
        """The weights' scales, packed once at set-up (outside every timed region)."""
        self.dg.dg_pack_sf_ue8m0(self.sfb_f, self.sfb, self.N, 128)

    def pack(self, io=None):
        """The activations' scales, packed every step."""
        sfa_f = self.sfa_f if io is None else io["sfa_f"]
        self.dg.dg_pack_sf_ue8m0(sfa_f, self.sfa, self.rows_a, 1)

    def gemm(self, io=None):
        dg = self.dg
        a, d, idx = (self.a, self.d, getattr(self, "idx", None)) if io is None else (io["a"], io["d"], io["idx"])
        if self.kind == "dense":
            dg.dg_fp8_gemm_nt(a, self.sfa, self.b, self.sfb, d)
        elif self.kind == "contiguous":
            dg.dg_m_grouped_fp8_gemm_nt_contiguous(a, self.sfa, self.b, self.sfb, d, idx)
        else:
            dg.dg_m_grouped_fp8_gemm_nt_masked(a, self.sfa, self.b, self.sfb, d, idx)

    # end-to-end: the step's inputs (activations, their FP32 scales, routing) come from pinned
    # host memory and D goes back to pinned host memory; weights stay resident.  Two device
    # sets of the per-step inputs and of D alternate between steps, so that one step's copies
    # run while the previous step's GEMMs still use the other set.
    def setup_e2e(self, dev):
        self.h_a = self.a.cpu().pin_memory()
        self.h_sfa = self.sfa_f.cpu().pin_memory()
        self.h_idx = self.idx.cpu().pin_memory() if self.kind != "dense" else None
        self.h_d = torch.empty(self.d.shape, dtype=self.d.dtype).pin_memory()
        self.io = []
        for j in range(2):
            self.io.append({"a": torch.empty_like(self.a), "sfa_f": torch.empty_like(self.sfa_f),
                            "idx": torch.empty_like(self.idx) if self.h_idx is not None else None,
                            "d": torch.empty_like(self.d),
                            "ev_h2d": torch.cuda.Event(), "ev_gemm": torch.cuda.Event(), "ev_d2h": torch.cuda.Event()})
        self.e2e_n = 0
        h2d = self.h_a.numel() + self.h_sfa.numel() * 4 + (self.h_idx.numel() * 4 if self.h_idx is not None else 0)
        d2h = self.h_d.numel() * 2
        return h2d, d2h

    def e2e_step(self, h2d_stream, compute_stream, d2h_stream):
        """One end-to-end pass: inputs from pinned host memory (h2d_stream), scale pack and
        GEMM (compute_stream), D back to pinned host memory (d2h_stream).  Events keep each
        device set from being overwritten while an earlier step still uses it."""
        io = self.io[self.e2e_n % 2]
        if self.e2e_n < 2:
            io["ev_gemm"].record(compute_stream)
            io["ev_d2h"].record(d2h_stream)
        self.e2e_n += 1
        h2d_stream.wait_event(io["ev_gemm"])             # the GEMM two steps back is done with the set
        with torch.cuda.stream(h2d_stream):
            io["a"].copy_(self.h_a, non_blocking=True)
            io["sfa_f"].copy_(self.h_sfa, non_blocking=True)
            if self.h_idx is not None:
                io["idx"].copy_(self.h_idx, non_blocking=True)
        io["ev_h2d"].record(h2d_stream)
        compute_stream.wait_event(io["ev_h2d"])
        compute_stream.wait_event(io["ev_d2h"])          # D of two steps back has been read back
        with torch.cuda.stream(compute_stream):
            self.pack(io)
            self.gemm(io)
        io["ev_gemm"].record(compute_stream)
        d2h_stream.wait_event(io["ev_gemm"])
        with torch.cuda.stream(d2h_stream):
            self.h_d.copy_(io["d"], non_blocking=True)
        self.ev_d2h = io["ev_d2h"]
        io["ev_d2h"].record(d2h_stream)


# ---------------------------------------------------------------------------
# Measurement helpers
# ---------------------------------------------------------------------------

def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm_gbs=float(j["hbm_gbs"]), bf16=float(j["bf16_tflops"]),
                    bf16_sustained=float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), source="measured")
    return dict(hbm_gbs=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, bf16_sustained=1700.0, source="fallback")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "moe_grouped_gemm_02_gb300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernels."""
    p = os.path.join(ROOT, "profiles", "ncu_dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    if j.get("kernel_source_sha") != kernel_source_sha():
        return None
    e = j.get("workloads", {}).get(workload_name)
    return None if e is None else e.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            sel = str(device_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# Ranks (one process per GPU under torchrun; independent replicas, weak scaling)
# ---------------------------------------------------------------------------

def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's time: the whole job ends when its last replica does."""
    if world <= 1:
        return x
    t = torch.tensor([float(x)], device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, ms: float) -> float:
    """All ranks' work over the slowest rank's time: every replica runs the same suite."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# Arms
# ---------------------------------------------------------------------------

def run_gpu(args, rank: int, world: int, local_rank: int):
    from moe_grouped_gemm_02_gb300 import build as dg_build
    dg_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    ws = make_workloads(seed=0)
    dws = [DeviceWorkload(w, dev) for w in ws]
    for dw in dws:
        dw.pack_weights()
    stream = torch.cuda.current_stream()

    def step(events=None, only=None):
        """One pass of the hot path.  events[i] = (start, end) brackets GEMM i; with `only`,
        just that GEMM is bracketed (other kernels then run back to back, which lets
        programmatic dependent launch overlap their launches)."""
        for i, dw in enumerate(dws):
            dw.pack()
            timed = events is not None and (only is None or i == only)
            if timed:
                events[i][0].record(stream)
            dw.gemm()
            if timed:
                events[i][1].record(stream)

    def new_events():
        return [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in dws]

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    import moe_grouped_gemm_02_gb300 as dg
    dg.dg_check_device_error()

    # Per-workload GEMM times (separate, untimed pass, every GEMM bracketed); the largest is
    # the dominant kernel, which is then bracketed alone inside the timed region.
    n_profile = max(3, min(20, args.steps))
    pev = [new_events() for _ in range(n_profile)]
    for k in range(n_profile):
        step(pev[k])
    torch.cuda.synchronize()
    # median over the profiling steps (the first one follows a host synchronisation), with min and max
    samples = [[pev[k][i][0].elapsed_time(pev[k][i][1]) for k in range(n_profile)] for i in range(len(dws))]
    per_kernel_ms = [statistics.median(v) for v in samples]
    dom = int(np.argmax(per_kernel_ms))

    ev = [new_events() for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank)
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for k in range(args.steps):
        step(ev[k], only=dom)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    dg.dg_check_device_error()
    total_ms = t0.elapsed_time(t1)
    total_ms = max_over_ranks(total_ms, world, dev)
    dom_ms = statistics.mean(ev[k][dom][0].elapsed_time(ev[k][dom][1]) for k in range(args.steps))

    flops_step = sum(w["flops"] for w in ws)
    value = whole_job_tflops(flops_step, args.steps, world, total_ms)
    peaks = read_peaks()
    timed_s = total_ms * 1e-3
    bf16 = peaks["bf16_sustained"] if timed_s >= 1.0 else peaks["bf16"]
    fp8_peak = bf16 * FP8_OVER_BF16
    peak_label = ("sustained" if timed_s >= 1.0 else "burst") + f" bf16 x {FP8_OVER_BF16:g} (of {peaks['source']})"
    ridge = fp8_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)

    per_wl = []
    for w, ms, smp in zip(ws, per_kernel_ms, samples):
        tflops = w["flops"] / (ms * 1e-3) / 1e12
        gbs = w["bytes"] / (ms * 1e-3) / 1e9
        bound = "tensor" if w["flops"] / w["bytes"] > ridge else "hbm"
        frac = tflops / fp8_peak if bound == "tensor" else gbs / peaks["hbm_gbs"]
        per_wl.append({"workload": w["name"], "ms": round(ms, 5), "ms_min": round(min(smp), 5),
                       "ms_max": round(max(smp), 5), "tflops": round(tflops, 1),
                       "gbs": round(gbs, 1), "bound": bound, "frac": round(frac, 4)})
    dw_ = ws[dom]
    if per_wl[dom]["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": round(dw_["flops"] / (dom_ms * 1e-3) / 1e12, 1),
                "peak": round(fp8_peak, 1), "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": round(dw_["bytes"] / (dom_ms * 1e-3) / 1e9, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = ncu_traffic(dw_["name"])
    roof["kernel"] = dw_["name"]
    roof["peak_source"] = peak_label if roof["bound"] == "tensor" else f"hbm copy (of {peaks['source']})"
    roof["algorithmic_per_launch"] = dw_["flops"] if roof["bound"] == "tensor" else dw_["bytes"]
    if roof["bound"] == "tensor" and clocks.get("sm_mhz"):
        # the tensor pipe's own rate at the clock seen during the timed region: 8192 FP8
        # multiply-adds per cycle per SM (measured with back-to-back 128 x 256 x 32 MMAs)
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        clock_peak = 2.0 * MMA_MACS_PER_CLK_SM * n_sm * clocks["sm_mhz"] * 1e6 / 1e12
        roof["clock_mma_peak"] = round(clock_peak, 1)
        roof["frac_of_clock_mma"] = round(roof["achieved"] / clock_peak, 4)

    # end to end, through the same public calls, inputs from pinned host memory
    e2e = None
    if not args.no_e2e:
        h2d = d2h = 0
        for dw in dws:
            hb, db = dw.setup_e2e(dev)
            h2d += hb
            d2h += db
        h2d_stream, d2h_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        for _ in range(2):
            for dw in dws:
                dw.e2e_step(h2d_stream, stream, d2h_stream)
        torch.cuda.synchronize()
        e_steps = max(3, min(args.steps, 20))
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        h2d_stream.wait_event(a0)
        for _ in range(e_steps):
            for dw in dws:
                dw.e2e_step(h2d_stream, stream, d2h_stream)
        for dw in dws:                                   # the timed region ends after the last copy back
            stream.wait_event(dw.ev_d2h)
        a1.record(stream)
        torch.cuda.synchronize()
        e_ms = a0.elapsed_time(a1)
        e_ms = max_over_ranks(e_ms, world, dev)
        e2e = {"value": round(whole_job_tflops(flops_step, e_steps, world, e_ms), 2), "unit": "TFLOPS",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e_steps,
               "ms_per_step": round(e_ms / e_steps, 4),
               "how": "activations, their FP32 scales and routing copied from pinned host memory on one "
                      "stream, scale pack + GEMM on the compute stream, D copied back on a third stream; two "
                      "device sets of inputs and D alternate between steps so copies overlap the previous "
                      "step's GEMMs; weights resident"}

    time_hbm_streams(ws, dws, per_wl, peaks)
    for pw in per_wl:
        pw["in_value"] = True
    per_wl.append(time_small_dense(dev, peaks))
    next_rows = None if args.no_next else time_next_rows(dev, peaks)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = time_oracle(ws, budget_s=args.cpu_budget, rows_per_workload=1024)

    if rank != 0:
        return None
    launches_per_step = 2 * len(dws)        # activation-scale pack + GEMM per workload
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic",
        "config": suite_config(ws, world),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks, "workloads": per_wl, "next_rows": next_rows,
    }


# Kernels beyond the GEMM step, each timed alone on its own workload (not part of `value`).
NEXT_QUANTIZE = [("quantize_32768x7168_bf16", 32768, 7168),     # the contiguous MoE tokens
                 ("quantize_4096x16384_bf16", 4096, 16384)]     # the prefill A


# The K-grouped weight-gradient GEMM of the contiguous MoE layer: dW_e = dY_e^T X_e for 4
# experts, M = 4096 (the layer's N), N = 7168 (its K), the experts' token counts (the same
# multinomial draw as the forward workload) padded to multiples of 128, FP32 accumulation
# into the gradients in place.
NEXT_K_GROUPED = ("k_grouped_wgrad_4x4096x7168_32768tok_f32acc", 4096, 7168)
# The prefill shape in the NN layout (B stored [K, N]) with FP32 output accumulated in place.
NEXT_LAYOUT = ("prefill_nn_f32acc_4096x7168x16384", 4096, 7168, 16384)


def _time_launches(fn, stream, flush, reps):
    """Median, min and max ms of `reps` launches of fn: CUDA events on the launching stream,
    L2 flushed (256 MB written) before every rep."""
    ts = []
    for r in range(reps):
        flush.fill_(float(r))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts), min(ts), max(ts)


L2_BYTES = 129 * 1024 * 1024


def _graph_stream_ms(call, copies: int, reps: int = 5) -> float:
    """Per-launch ms of call(i, stream) for i in range(copies), back to back inside one CUDA
    graph: no host launch cost in the timing, programmatic-dependent-launch edges kept (each
    launch may overlap the one before).  Events around 4 replays."""
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for i in range(copies):           # warm-up outside the capture (plans, attributes)
            call(i, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(copies):
            call(i, s)
    per = []
    with torch.cuda.stream(s):            # replays go to the current stream
        g.replay()
        s.synchronize()
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(4):
                g.replay()
            e1.record(s)
            s.synchronize()
            per.append(e0.elapsed_time(e1) / (4 * copies))
    del g
    return statistics.median(per)


def _weight_copies(nbytes: int) -> int:
    """Copies of a weight tensor that together exceed twice the L2 (2..16)."""
    return max(2, min(16, -(-2 * L2_BYTES // nbytes)))


def time_hbm_streams(ws, dws, per_wl, peaks):
    """The HBM-bound GEMMs (decode shapes, masked MoE) as a model's decode step runs them: the
    same call back to back over distinct weight tensors (each workload's B and packed SFB copied
    until the copies exceed twice the L2, so every launch reads its weights from HBM), captured
    in one CUDA graph (`_graph_stream_ms`).  Same algorithmic bytes as the bracketed number.
    Adds stream_* keys to per_wl."""
    import moe_grouped_gemm_02_gb300 as dg
    for w, dw, pw in zip(ws, dws, per_wl):
        if pw["bound"] != "hbm":
            continue
        copies = _weight_copies(dw.b.numel() * dw.b.element_size())
        bs = [dw.b.clone() for _ in range(copies)]
        sfbs = [dw.sfb.clone() for _ in range(copies)]

        def call(i, s):
            if dw.kind == "dense":
                dg.dg_fp8_gemm_nt(dw.a, dw.sfa, bs[i], sfbs[i], dw.d, stream=s)
            else:
                dg.dg_m_grouped_fp8_gemm_nt_masked(dw.a, dw.sfa, bs[i], sfbs[i], dw.d, dw.idx, stream=s)

        ms = _graph_stream_ms(call, copies)
        gbs = w["bytes"] / (ms * 1e-3) / 1e9
        pw.update({"stream_ms": round(ms, 5), "stream_gbs": round(gbs, 1),
                   "stream_frac": round(gbs / peaks["hbm_gbs"], 4), "stream_weight_copies": copies})
        del bs, sfbs
    dg.dg_check_device_error()


def run_workload_only(args, local_rank: int):
    """One workload of the suite alone: its weights' scales packed once, then `warmup` untimed and
    `steps` timed launches of (activation-scale pack + GEMM), the GEMM bracketed by CUDA events
    with L2 flushed before each launch.  For profiling one kernel on its full-size workload."""
    from moe_grouped_gemm_02_gb300 import build as dg_build
    import moe_grouped_gemm_02_gb300 as dg
    dg_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    ws = [w for w in make_workloads(seed=0) if args.workload_only in w["name"]]
    if not ws:
        raise SystemExit(f"no workload matches {args.workload_only!r}")
    w = ws[0]
    dw = DeviceWorkload(w, dev)
    dw.pack_weights()
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        dw.pack()
        dw.gemm()
    ts = []
    for r in range(args.steps):
        flush.fill_(float(r))
        dw.pack()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dw.gemm()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    dg.dg_check_device_error()
    ms = statistics.median(ts)
    return {"workload": w["name"], "launches": args.steps, "ms": round(ms, 5), "ms_min": round(min(ts), 5),
            "tflops": round(w["flops"] / (ms * 1e-3) / 1e12, 1), "gbs": round(w["bytes"] / (ms * 1e-3) / 1e9, 1)}


def time_small_dense(dev, peaks, reps: int = 20):
    """The small dense GEMM 128x512x1024 (A, B ~ N(0, 1), seed 0), timed beside the step as a
    latency-bound row of its own: bracketed alone with L2 flushed before each rep, and back to
    back inside one CUDA graph (16 launches per replay over 16 weight copies; they fit in L2).
    Both fractions are reported, of the FP8 tensor peak and of HBM bandwidth."""
    import moe_grouped_gemm_02_gb300 as dg
    M, N, K = synth.SMALL_DENSE
    w = synth.make_dense(M, N, K, seed=0)
    w["kind"] = "dense"
    w["valid_rows"] = M
    dw = DeviceWorkload(w, dev)
    dw.pack_weights()
    dw.pack()
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(3):
        dw.gemm()
    ms, lo, hi = _time_launches(dw.gemm, stream, flush, reps)
    copies = 16
    bs = [dw.b.clone() for _ in range(copies)]
    sfbs = [dw.sfb.clone() for _ in range(copies)]
    sms = _graph_stream_ms(lambda i, st: dg.dg_fp8_gemm_nt(dw.a, dw.sfa, bs[i], sfbs[i], dw.d, stream=st), copies)
    dg.dg_check_device_error()
    flops = 2.0 * M * N * K
    nbytes = _algorithmic_bytes(w)
    fp8_peak = peaks["bf16"] * FP8_OVER_BF16

    def rates(t_ms):
        tf = flops / (t_ms * 1e-3) / 1e12
        gbs = nbytes / (t_ms * 1e-3) / 1e9
        return tf, gbs

    tf, gbs = rates(ms)
    stf, sgbs = rates(sms)
    del flush, bs, sfbs
    return {"workload": f"small_dense_{M}x{N}x{K}", "in_value": False, "bound": "latency",
            "ms": round(ms, 5), "ms_min": round(lo, 5), "ms_max": round(hi, 5), "us": round(ms * 1e3, 2),
            "flops": flops, "bytes": nbytes, "tflops": round(tf, 2), "gbs": round(gbs, 1),
            "frac_tensor": round(tf / fp8_peak, 4), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "stream_ms": round(sms, 5), "stream_tflops": round(stf, 2), "stream_gbs": round(sgbs, 1),
            "stream_frac_tensor": round(stf / fp8_peak, 4), "stream_frac_hbm": round(sgbs / peaks["hbm_gbs"], 4),
            "how": "bracketed: alone, L2 flushed before each of 20 reps (median); stream: back to back in one "
                   "CUDA graph over 16 weight copies (L2-resident)"}


def _random_e4m3(shape, gen, dev):
    """N(0, 1) values as E4M3 codes (timing inputs: the tensor cores' speed does not depend on them)."""
    return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


def time_next_rows(dev, peaks, reps: int = 20, only: str | None = None):
    """Kernels timed beside the GEMM step, each alone on its own workload, L2 flushed before every
    rep: the per-token quantisation (algorithmic bytes = 2 MK read + MK codes + 4 Kp al4(M)
    scale bytes written), the K-grouped weight-gradient GEMM and the NN-layout FP32-accumulating
    GEMM (2 M N K flops each)."""
    import moe_grouped_gemm_02_gb300 as dg
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)     # 256 MB > L2
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    fp8_peak = peaks["bf16"] * FP8_OVER_BF16
    rows = []

    def hbm_row(row, name, ms, lo, hi, nbytes):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"row": row, "workload": name, "ms": round(ms, 5), "ms_min": round(lo, 5), "ms_max": round(hi, 5),
                "bytes": nbytes, "gbs": round(gbs, 1), "bound": "hbm", "frac": round(gbs / peaks["hbm_gbs"], 4),
                "peak_source": f"hbm copy (of {peaks['source']})"}

    def stream_row(ms, nbytes):
        # back to back over weight copies in one CUDA graph (see time_hbm_streams)
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"stream_ms": round(ms, 5), "stream_gbs": round(gbs, 1), "stream_frac": round(gbs / peaks["hbm_gbs"], 4)}

    def tensor_row(row, name, ms, lo, hi, flops, nbytes):
        tf = flops / (ms * 1e-3) / 1e12
        return {"row": row, "workload": name, "ms": round(ms, 5), "ms_min": round(lo, 5), "ms_max": round(hi, 5),
                "flops": flops, "bytes": nbytes, "tflops": round(tf, 1), "bound": "tensor",
                "frac": round(tf / fp8_peak, 4),
                "peak_source": f"burst bf16 x {FP8_OVER_BF16:g} (of {peaks['source']})"}

    def skip(name):
        return only is not None and only not in name

    for name, M, K in NEXT_QUANTIZE:
        if skip(name):
            continue
        x = torch.randn((M, K), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
        q = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sf = torch.empty(dg.packed_sf_shape(None, M, K), dtype=torch.int32, device=dev)
        for _ in range(3):
            dg.dg_quantize_fp8_1x128(x, q, sf)
        ms, lo, hi = _time_launches(lambda: dg.dg_quantize_fp8_1x128(x, q, sf), stream, flush, reps)
        dg.dg_check_device_error()
        rows.append(hbm_row("per-token 1x128 FP8 quantisation (dg_quantize_fp8_1x128)", name, ms, lo, hi,
                            3 * M * K + 4 * sf.numel()))
        del x, q, sf

    # K-grouped weight gradient
    name, M, N = NEXT_K_GROUPED
    if not skip(name):
        _time_k_grouped(rows, name, M, N, gen, dev, stream, flush, reps, tensor_row)

    # NN layout, FP32 out accumulated in place
    name, M, N, K = NEXT_LAYOUT
    if not skip(name):
        _time_nn_layout(rows, name, M, N, K, gen, dev, stream, flush, reps, tensor_row)

    _time_fp8_fp4(rows, gen, dev, stream, flush, reps, hbm_row, tensor_row, stream_row, skip)
    return rows


def _time_k_grouped(rows, name, M, N, gen, dev, stream, flush, reps, tensor_row):
    """The K-grouped weight-gradient GEMM, D += A^T B in place (FP32)."""
    import moe_grouped_gemm_02_gb300 as dg
    counts = synth.rng(0, "counts").multinomial(synth.CONTIGUOUS["tokens"], [0.25] * 4)
    ks = [synth.align_up(int(c), 128) for c in counts]
    sum_k = sum(ks)
    a = _random_e4m3((sum_k, M), gen, dev)
    b = _random_e4m3((sum_k, N), gen, dev)
    rows_sf = dg.k_grouped_packed_sf_rows(ks)
    sfa = torch.full((rows_sf, dg.dg_get_tma_aligned_size(M)), 0x7F7F7F7F, dtype=torch.int32, device=dev)
    sfb = torch.full((rows_sf, dg.dg_get_tma_aligned_size(N)), 0x7F7F7F7F, dtype=torch.int32, device=dev)
    d = torch.zeros((4, M, N), dtype=torch.float32, device=dev)
    ks_d = torch.tensor(ks, dtype=torch.int32, device=dev)
    call = lambda: dg.dg_k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, d, ks_d, c=d)
    for _ in range(3):
        call()
    ms, lo, hi = _time_launches(call, stream, flush, reps)
    dg.dg_check_device_error()
    rows.append(tensor_row("K-grouped FP8 weight-gradient GEMM (dg_k_grouped_fp8_gemm_tn_contiguous), "
                           "D += A^T B in place", name, ms, lo, hi, 2.0 * M * N * sum_k,
                           sum_k * (M + N) + 2 * 4 * 4 * M * N))


def _time_nn_layout(rows, name, M, N, K, gen, dev, stream, flush, reps, tensor_row):
    """The prefill shape in the NN layout, FP32 D += A B^T in place."""
    import moe_grouped_gemm_02_gb300 as dg
    a = _random_e4m3((M, K), gen, dev)
    b = _random_e4m3((K, N), gen, dev)
    sfa = torch.full(dg.packed_sf_shape(None, M, K), 0x7F7F7F7F, dtype=torch.int32, device=dev)
    sfb = torch.full(dg.packed_sf_shape(None, N, K), 0x7F7F7F7F, dtype=torch.int32, device=dev)
    d = torch.zeros((M, N), dtype=torch.float32, device=dev)
    call = lambda: dg.dg_fp8_gemm(a, sfa, b, sfb, d, layout="nn", c=d)
    for _ in range(3):
        call()
    ms, lo, hi = _time_launches(call, stream, flush, reps)
    dg.dg_check_device_error()
    rows.append(tensor_row("FP8 GEMM, NN layout, D += A B^T in FP32 (dg_fp8_gemm)", name, ms, lo, hi,
                           2.0 * M * N * K, M * K + N * K + 2 * 4 * M * N))


def _time_fp8_fp4(rows, gen, dev, stream, flush, reps, hbm_row, tensor_row, stream_row, skip):
    """FP8 x FP4: the decode shapes and the masked MoE shape with E2M1 weights (HBM-bound: the
    weights are read once at half the FP8 bytes), and the prefill shape (tensor-bound)."""
    import moe_grouped_gemm_02_gb300 as dg

    def fp4_weights(shape):
        return torch.randint(0, 256, shape, generator=gen, device=dev, dtype=torch.int32).to(torch.uint8)

    for (M, N, K) in synth.DECODE_SHAPES + [synth.PREFILL_SHAPE]:
        name = f"fp8xfp4_{'prefill' if M == 4096 else 'decode'}_{M}x{N}x{K}"
        if skip(name):
            continue
        a = _random_e4m3((M, K), gen, dev)
        b = fp4_weights((N, K // 2))
        sfa = torch.full(dg.packed_sf_shape(None, M, K), 0x7F7F7F7F, dtype=torch.int32, device=dev)
        sfb = torch.full(dg.packed_sf_shape(None, N, K), 0x7F7F7F7F, dtype=torch.int32, device=dev)
        d = torch.empty((M, N), dtype=torch.int16, device=dev)
        call = lambda: dg.dg_fp8_fp4_gemm_nt(a, sfa, b, sfb, d)
        for _ in range(3):
            call()
        ms, lo, hi = _time_launches(call, stream, flush, reps)
        dg.dg_check_device_error()
        nbytes = M * K + N * K // 2 + 2 * M * N + 4 * (sfa.numel() + sfb.numel())
        row = "FP8 x FP4 GEMM (dg_fp8_fp4_gemm_nt)"
        if M == 4096:
            rows.append(tensor_row(row, name, ms, lo, hi, 2.0 * M * N * K, nbytes))
        else:
            rows.append(hbm_row(row, name, ms, lo, hi, nbytes))
            copies = _weight_copies(b.numel())
            bs = [b.clone() for _ in range(copies)]
            sms = _graph_stream_ms(lambda i, st: dg.dg_fp8_fp4_gemm_nt(a, sfa, bs[i], sfb, d, stream=st), copies)
            rows[-1].update(stream_row(sms, nbytes))
            del bs
    G, max_m, N, K = (synth.MASKED[k] for k in ("G", "max_m", "N", "K"))
    name = f"fp8xfp4_masked_{G}x{max_m}x{N}x{K}"
    if skip(name):
        return
    masked_m = synth.rng(0, "masked_m").integers(1, max_m + 1, size=G)
    a = _random_e4m3((G, max_m, K), gen, dev)
    b = fp4_weights((G, N, K // 2))
    sfa = torch.full(dg.packed_sf_shape(G, max_m, K), 0x7F7F7F7F, dtype=torch.int32, device=dev)
    sfb = torch.full(dg.packed_sf_shape(G, N, K), 0x7F7F7F7F, dtype=torch.int32, device=dev)
    d = torch.empty((G, max_m, N), dtype=torch.int16, device=dev)
    mm = torch.tensor(masked_m, dtype=torch.int32, device=dev)
    call = lambda: dg.dg_m_grouped_fp8_fp4_gemm_nt_masked(a, sfa, b, sfb, d, mm)
    for _ in range(3):
        call()
    ms, lo, hi = _time_launches(call, stream, flush, reps)
    dg.dg_check_device_error()
    valid = int(masked_m.sum())
    nbytes = valid * K + G * N * K // 2 + 2 * valid * N + 4 * (sfa.numel() + sfb.numel())
    rows.append(hbm_row("FP8 x FP4 masked grouped GEMM (dg_m_grouped_fp8_fp4_gemm_nt_masked)", name, ms, lo, hi,
                        nbytes))
    copies = _weight_copies(b.numel())
    bs = [b.clone() for _ in range(copies)]
    sms = _graph_stream_ms(lambda i, st: dg.dg_m_grouped_fp8_fp4_gemm_nt_masked(a, sfa, bs[i], sfb, d, mm, stream=st),
                           copies)
    rows[-1].update(stream_row(sms, nbytes))
    del bs


def time_oracle(ws, budget_s: float = 20.0, rows_per_workload: int = 4):
    """Times the float64 oracle as it stands on a bounded sample: `rows_per_workload` output rows
    of every workload (all columns, all of K), including the scale-factor packing."""
    import oracle
    rs = np.random.default_rng(0)
    t_total = 0.0
    flops = 0.0
    done = []
    t_start = time.perf_counter()
    for w in ws:
        if time.perf_counter() - t_start > budget_s:
            break
        N, K = w["N"], w["K"]
        t0 = time.perf_counter()
        if w["kind"] == "dense":
            rows = np.sort(rs.choice(w["M"], size=min(rows_per_workload, w["M"]), replace=False))
            sfa = oracle.pack_sf_ue8m0(w["sfa"][rows], len(rows), 1)[0]
            sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
            oracle.fp8_gemm_nt(w["a"][rows], sfa, w["b"], sfb)
            n_rows = len(rows)
        elif w["kind"] == "contiguous":
            valid = np.nonzero(w["m_indices"] >= 0)[0]
            rows = np.sort(rs.choice(valid, size=rows_per_workload, replace=False))
            sfa = oracle.pack_sf_ue8m0(w["sfa"], w["M_sum"], 1)[0]
            sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)
            oracle.m_grouped_fp8_gemm_nt_contiguous(w["a"], sfa, w["b"], sfb, w["m_indices"], rows=rows)
            n_rows = len(rows)
        else:
            # the first rows of each group, about rows_per_workload in all
            mm = np.minimum(w["masked_m"], max(1, rows_per_workload // w["G"]))
            sfa = oracle.pack_sf_ue8m0(w["sfa"], w["max_m"], 1)
            sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)
            prior = np.zeros((w["G"], w["max_m"], N), np.uint16)
            oracle.m_grouped_fp8_gemm_nt_masked(w["a"], sfa, w["b"], sfb, mm, prior)
            n_rows = int(mm.sum())
        t_total += time.perf_counter() - t0
        flops += 2.0 * n_rows * N * K
        done.append(f"{w['name']}:{n_rows}rows")
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": flops / t_total / 1e12, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
            "sample": "output rows (all N columns, full K, incl. scale packing) of each workload: " + ", ".join(done),
            "seconds": round(t_total, 2)}


REFERENCE_BUDGET_S = 150.0   # the whole --impl reference run (warm-up and timed steps)


def run_reference(args, rank: int, world: int):
    """The oracle timed as it stands: each step is a bounded sample of the suite.  The sample
    (output rows per workload, the same for every step) is sized from two timed warm-up passes
    so that all warm-up and timed steps together take about REFERENCE_BUDGET_S: each oracle
    call decodes the whole weight matrix, so a one-row sample would time mostly that decode."""
    if rank != 0:
        return None
    ws = make_workloads(seed=0)
    t_1 = time_oracle(ws, budget_s=1e9, rows_per_workload=1)["seconds"]
    t_16 = time_oracle(ws, budget_s=1e9, rows_per_workload=16)["seconds"]
    per_row = max(t_16 - t_1, 1e-3) / 15.0
    per_step = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)
    rows = int(max(1, min(1024, (per_step - t_1) / per_row)))
    for _ in range(args.warmup):
        time_oracle(ws, budget_s=1e9, rows_per_workload=rows)
    vals = []
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        r = time_oracle(ws, budget_s=1e9, rows_per_workload=rows)
        vals.append(r)
    elapsed = time.perf_counter() - t0
    value = statistics.mean(v["value"] for v in vals)
    cpu = dict(vals[-1])
    cpu["value"] = value
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed * 1e3 / max(1, args.steps), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": suite_config(ws, world),
            "cpu_baseline": cpu, "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                                         "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="dg", choices=["dg", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next", action="store_true", help="skip the kernels timed beside the GEMM step")
    ap.add_argument("--cpu-budget", type=float, default=30.0)
    ap.add_argument("--workload-only", default=None, metavar="NAME",
                    help="set up only the suite workload whose name contains NAME and time its GEMM alone "
                         "(activation-scale pack + GEMM per launch, L2 flushed before each); prints one line")
    ap.add_argument("--next-only", default=None, metavar="NAME",
                    help="time only the kernels beside the step whose workload name contains NAME (for "
                         "profiling one kernel); prints their rows")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "dg":
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if args.impl == "dg" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend=backend)
    try:
        if args.workload_only is not None:
            print(json.dumps(run_workload_only(args, local_rank)))
            return
        if args.next_only is not None:
            from moe_grouped_gemm_02_gb300 import build as dg_build
            dg_build.build()
            dev = torch.device("cuda", local_rank)
            torch.cuda.set_device(dev)
            print(json.dumps({"next_rows": time_next_rows(dev, read_peaks(), reps=5, only=args.next_only)}))
            return
        out = run_reference(args, rank, world) if args.impl == "reference" else run_gpu(args, rank, world, local_rank)
        if rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
