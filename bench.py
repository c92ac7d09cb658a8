#!/usr/bin/env python3
"""Benchmark of the fused FP8 MoE layer on GB300.

One step = one forward of the whole layer (routing, gather, gate_up GEMM + SwiGLU +
requant, down GEMM + weighted scatter, combine) over one synthetic batch.  The headline
workload is the largest single-GPU batch: T=16384 tokens, H=4096, I=1536, E=128, topk=8,
R=8, uniform routing, FP8 e4m3 activations and weights with fp32 block scales.  The same
run also times the other batch shapes (tiny, decode, prefill, skewed) and reports them
under ``per_config``.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line.  ``value`` is routed (token, slot) rows per second of the whole
job with inputs resident in HBM, timed with CUDA events on the forward's stream; ``e2e``
is the same metric through ``moe_forward_host_async`` (pinned host buffers, copies inside
the timed region).  ``roofline`` covers the dominant kernel, timed live with CUDA events the
library records around each of its kernels; its tensor peak is the larger of a dense FP8
GEMM measured at the start of the run and the measured bf16 peak times the nominal FP8/bf16
ratio.  ``--impl reference`` times the plain CPU oracle on a bounded sample of the same
workload instead (the reference arm).
Several GPUs run independent replicas (the layer is single-GPU): ``value`` sums the rows
of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused MoE routed tokens/s"
UNIT = "routed tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor-rate ratio on GB300
L2_BYTES = 129 * 2 ** 20
PROFILE_EVERY = 8            # timed steps per step carrying the per-kernel stage events

# DRAM bytes per launch from one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum),
# valid only while the kernel sources hash to `src_sha`; see profiles/.
NCU_TRAFFIC = {
    ("large", "expert_ffn"): {"bytes": 3246707712 + 1247772416, "src_sha": "05d9ff51cb1a7884"},
    ("decode", "expert_ffn"): {"bytes": 1421868032 + 4820736, "src_sha": "05d9ff51cb1a7884"},
    ("prefill", "expert_ffn"): {"bytes": 1998627328 + 515535104, "src_sha": "05d9ff51cb1a7884"},
    # the block-scaled kernel (power-of-two scales, MXFP4 weights)
    ("decode-mxfp4", "expert_ffn"): {"bytes": 759937792 + 4401664, "src_sha": "a2befd31d661562d"},
    ("prefill-pow2", "expert_ffn"): {"bytes": 2100153088 + 516071168, "src_sha": "a2befd31d661562d"},
}
# sources each stage's kernel is compiled from (a recorded traffic figure is used only while
# these hash to its `src_sha`)
KERNEL_SOURCES = {
    "expert_ffn": ["combine_persistent_warp_gb300/csrc/ffn.cu",
                   "combine_persistent_warp_gb300/csrc/ptx.cuh",
                   "combine_persistent_warp_gb300/csrc/moe_internal.cuh",
                   "combine_persistent_warp_gb300/csrc/topk_combine.cuh"],
    # power-of-two scales: the expert FFN stage runs the block-scaled kernel
    "expert_ffn_bs": ["combine_persistent_warp_gb300/csrc/ffn_bs.cu",
                      "combine_persistent_warp_gb300/csrc/ptx.cuh",
                      "combine_persistent_warp_gb300/csrc/moe_internal.cuh",
                      "combine_persistent_warp_gb300/csrc/topk_combine.cuh"],
    "dispatch": ["combine_persistent_warp_gb300/csrc/routing.cu",
                 "combine_persistent_warp_gb300/csrc/route_device.cuh",
                 "combine_persistent_warp_gb300/csrc/ptx.cuh",
                 "combine_persistent_warp_gb300/csrc/moe_internal.cuh",
                 "combine_persistent_warp_gb300/csrc/topk_combine.cuh"],
    "combine": ["combine_persistent_warp_gb300/csrc/routing.cu",
                "combine_persistent_warp_gb300/csrc/moe_internal.cuh",
                "combine_persistent_warp_gb300/csrc/topk_combine.cuh"],
}

KERNEL_FN = {"expert_ffn": "ffn_kernel", "expert_ffn_bs": "ffn_bs_kernel", "dispatch": "dispatch_kernel",
             "combine": "combine_kernel"}


def kernel_sources_sha(stage: str = "expert_ffn") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[stage]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ distributed ---
class Dist:
    """Rank bookkeeping; N>1 runs under torchrun, one process per GPU."""

    def __init__(self, backend: str | None = None, init: bool = True):
        import torch
        import torch.distributed as td
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.td = td
        if not init:                 # ranks that never communicate (the reference arm)
            return
        if self.world > 1 and not td.is_initialized():
            if backend is None:
                backend = "nccl" if torch.cuda.is_available() else "gloo"
            kw = {}
            if backend == "nccl":
                kw["device_id"] = torch.device("cuda", self.local_rank)
            td.init_process_group(backend=backend, **kw)

    def barrier(self):
        if self.world > 1 and self.td.is_initialized():
            self.td.barrier()

    def max(self, v: float) -> float:
        return self._reduce(v, "max")

    def sum(self, v: float) -> float:
        return self._reduce(v, "sum")

    def _reduce(self, v: float, op: str) -> float:
        if self.world == 1 or not self.td.is_initialized():
            return float(v)
        import torch
        dev = "cuda" if self.td.get_backend() == "nccl" else "cpu"
        t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
        self.td.all_reduce(t, op=self.td.ReduceOp.MAX if op == "max" else self.td.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.world > 1 and self.td.is_initialized():
            self.td.destroy_process_group()


def aggregate(local_units: float, local_seconds: float, dist: Dist) -> tuple[float, float]:
    """(units of all ranks / slowest rank's seconds, slowest rank's seconds)."""
    t = dist.max(local_seconds)
    u = dist.sum(local_units)
    return u / t, t


# ------------------------------------------------------------------ clocks --------
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []          # (host time, sm, max, reasons)
        self.proc = None
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            reasons = [n for n, v in zip(names, parts[4:8]) if v.lower().startswith("active")]
            self.samples.append((time.time(), sm, mx, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        if not inside:            # region shorter than the sampling period: nearest samples
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            window = "nearest to timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({r for s in inside for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


def gpu_query_id(torch, dev: int) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev)


# ------------------------------------------------------------------ work model ----
def work_model(inp) -> dict:
    """Algorithmic bytes and FLOPs of one forward (valid rows only).

    compulsory_bytes: what the layer must move at least once (the expert weights and scales
    of the experts the batch touches, x and its scales, the routing ids and gate weights, the
    bf16 output); intermediate_bytes: what this design writes and reads back on the way (the
    gathered pool, the SwiGLU rows, the bf16 combine planes)."""
    import torch
    wl = inp.wl
    T, H, I, E, K = wl.T, wl.H, wl.I, wl.E, wl.topk
    idx = inp.topk_idx
    M = int((idx >= 0).sum().item())
    touched = int(torch.unique(idx[idx >= 0]).numel())
    if getattr(wl, "weights", "fp8") == "mxfp4":
        # packed E2M1 (half a byte per element) + one UE8M0 byte per 32 elements
        w1 = touched * (2 * I * H // 2 + 2 * I * H // 32)
        w2 = touched * (H * I // 2 + H * I // 32)
    else:
        w1 = touched * (2 * I * H + (2 * I // 128) * (H // 128) * 4)
        w2 = touched * (H * I + (H // 128) * (I // 128) * 4)
    x_rows = M * (H + (H // 128) * 4)            # gathered activation rows + scales
    act_rows = M * (I + (I // 128) * 4)
    compulsory = w1 + w2 + T * (H + (H // 128) * 4) + T * K * 12 + T * H * 2
    intermediate = 2 * x_rows + 2 * act_rows + 2 * M * H * 2 + M * 12
    st = {
        "dispatch": {"bytes": T * K * 8 + 2 * x_rows + M * (12 + 8) + T * 4, "flops": 0},
        # gate_up GEMM + SwiGLU + down GEMM + weighted scatter (one kernel): weights, the
        # gathered rows in, the SwiGLU rows out and back in, the bf16 planes out
        "expert_ffn": {"bytes": w1 + w2 + x_rows + 2 * act_rows + M * H * 2 + M * 16,
                       "flops": 2 * M * H * 2 * I + 2 * M * I * H},
        # the bf16 planes in, the output out, one slot-mask word per token
        "combine": {"bytes": M * H * 2 + T * H * 2 + T * 4, "flops": M * H},
    }
    from combine_persistent_warp_gb300.workloads import skew_ratio
    return {"M": M, "touched_experts": touched, "stages": st, "compulsory_bytes": compulsory,
            "hot_expert_rows_over_mean": round(float(skew_ratio(idx, E)), 3),
            "intermediate_bytes": intermediate, "flops": 6 * M * H * I, "weight_bytes": w1 + w2}


def peaks() -> tuple[dict, str]:
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"]))}, "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0}, "fallback"


def measure_fp8_gemm_tflops(dev, n: int = 8192, reps: int = 10) -> float | None:
    """Dense FP8 e4m3 GEMM n x n x n through cuBLAS (torch._scaled_mm, bf16 out), best of
    `reps` CUDA-event-timed calls after a warm-up; TFLOP/s, or None where unavailable."""
    import torch
    try:
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()   # column-major operand
        one = torch.ones((), device=dev)
        mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            mm()
        torch.cuda.synchronize(dev)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mm()
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3)
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / best / 1e12
    except Exception:
        return None


def tensor_peak(fp8_measured: float | None) -> tuple[float, str]:
    """FP8 tensor denominator: the larger of the measured dense FP8 GEMM and the measured bf16
    burst peak times the nominal FP8/bf16 ratio (the larger one never flatters a fraction)."""
    pk, src = peaks()
    via_bf16 = pk["bf16_tflops"] * FP8_OVER_BF16
    if fp8_measured is not None and fp8_measured > via_bf16:
        return fp8_measured, "measured dense FP8 GEMM (torch._scaled_mm 8192^3, best of 10)"
    return via_bf16, f"{src} bf16 burst x {FP8_OVER_BF16} (nominal fp8/bf16)"


def roofline_for(stage: str, avg_s: float, model: dict, workload: str, fp8_measured: float | None) -> dict:
    """Roofline of the dominant kernel.  HBM-bound shapes count the layer's compulsory bytes
    (all of them pass through this kernel or its neighbours once; the intermediates of the
    design are reported beside them, not counted); tensor-bound shapes count 6*M*H*I."""
    pk, src = peaks()
    st = model["stages"][stage]
    flops = st["flops"]
    bytes_ = model["compulsory_bytes"] if stage == "expert_ffn" else st["bytes"]
    fp8_peak, fp8_src = tensor_peak(fp8_measured)
    t_hbm = bytes_ / (pk["hbm_gbs"] * 1e9)
    t_tensor = flops / (fp8_peak * 1e12) if flops else 0.0
    traffic = None
    block_scaled = workload.endswith("-pow2") or workload.endswith("-mxfp4")
    src_key = "expert_ffn_bs" if stage == "expert_ffn" and block_scaled else stage
    rec = NCU_TRAFFIC.get((workload, stage))
    if rec and rec.get("src_sha") == kernel_sources_sha(src_key):
        traffic = rec["bytes"]
    common = {"kernel": stage, "kernel_fn": KERNEL_FN.get(src_key, stage), "traffic": traffic,
              "avg_launch_us": avg_s * 1e6}
    if t_tensor > t_hbm and flops:
        achieved = flops / avg_s / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak, "algorithmic_flops": flops, "peak_source": fp8_src,
                "fp8_gemm_measured_tflops": fp8_measured,
                "bf16_x2_tflops": pk["bf16_tflops"] * FP8_OVER_BF16, "nominal_fp8_tflops": 4500.0,
                **common}
    achieved = bytes_ / avg_s / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "algorithmic_bytes": bytes_,
            "kernel_bytes_with_intermediates": st["bytes"],
            "peak_source": f"{src} (hbm_gbs, copy bandwidth)", **common}


def layer_roofline(model: dict, step_s: float, fp8_measured: float | None) -> dict:
    """The whole step against t_roof = max(FLOPs / FP8 peak, compulsory bytes / HBM)."""
    pk, _ = peaks()
    fp8_peak, _ = tensor_peak(fp8_measured)
    t_t = model["flops"] / (fp8_peak * 1e12)
    t_b = model["compulsory_bytes"] / (pk["hbm_gbs"] * 1e9)
    return {"t_roof_us": max(t_t, t_b) * 1e6, "bound": "tensor" if t_t > t_b else "hbm",
            "frac": max(t_t, t_b) / step_s, "compulsory_bytes": model["compulsory_bytes"],
            "intermediate_bytes": model["intermediate_bytes"], "flops": model["flops"]}


# ------------------------------------------------------------------ CPU oracle ----
def oracle_rows_per_s(host, tokens, row_mask=None) -> tuple[float, float, int]:
    """Time the CPU oracle on the given tokens (optionally keeping only some slots)."""
    import numpy as np
    import oracle
    full_idx = host.idx
    if row_mask is not None:
        host.idx = np.ascontiguousarray(np.where(row_mask, full_idx, -1), dtype=np.int64)
    try:
        rows = int((host.idx[tokens] >= 0).sum())
        t0 = time.perf_counter()
        oracle.forward_tokens(host, tokens)
        dt = time.perf_counter() - t0
    finally:
        host.idx = full_idx
    return rows / dt, dt, rows


def cpu_baseline(inp, n_tokens: int, min_seconds: float = 10.0) -> dict:
    """The oracle on the first `n_tokens` tokens of the batch, repeated until at least
    `min_seconds` of wall time have passed (at most 50 passes)."""
    import numpy as np
    import oracle
    toks = np.arange(min(n_tokens, inp.wl.T))
    oracle.set_scale_rule(inp.wl.scales)
    host = oracle.HostInputs.from_inputs(inp)
    total_rows, total_dt, passes = 0, 0.0, 0
    try:
        while passes == 0 or (total_dt < min_seconds and passes < 50):
            _, dt, rows = oracle_rows_per_s(host, toks)
            total_rows += rows
            total_dt += dt
            passes += 1
    finally:
        oracle.set_scale_rule("fp32")
    return {"value": total_rows / total_dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{toks.size} tokens ({total_rows // passes} routed rows) of the {inp.wl.name} batch, "
                      f"{passes} passes, {total_dt:.1f} s wall"}


# ------------------------------------------------------------------ arms -----------
def _l2_flush_buffer(torch, dev):
    return torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)


def needs_l2_flush(model: dict) -> bool:
    """A batch whose weights and intermediate buffers fit in twice the L2 gets an L2 flush
    before every timed step; larger ones stream more than the L2 every step."""
    return model["weight_bytes"] + model["intermediate_bytes"] < 2 * L2_BYTES


def config_of(wl, model: dict, world: int, flush: bool) -> dict:
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
            "topk": wl.topk, "R": wl.R, "routing": wl.routing, "scales": wl.scales,
            "weights": wl.weights, "routed_rows_per_step": model["M"],
            **({"hot_expert_rows_over_mean": model["hot_expert_rows_over_mean"]} if wl.routing == "zipf" else {}),
            "parallelism": f"replicas x{world}",
            "l2": ("L2 flushed (%d MB written) before every timed step, steps timed one by one"
                   % (2 * L2_BYTES >> 20) if flush else
                   "inputs larger than L2: %.2f GB of expert weights streamed per step, no flush"
                   % (model["weight_bytes"] / 1e9))}


def bench_config(name: str, args, dist: Dist, steps: int, warmup: int, *, e2e_steps: int,
                 cpu_seconds: float | None, fp8_measured: float | None, sampler=None) -> dict:
    """Time `steps` forwards of one workload (after `warmup` untimed ones) and describe them.

    Workloads whose weights and buffers fit in twice the L2 get an L2 flush (a write of twice
    its size) before every timed forward, and each forward is timed alone; larger ones stream
    more than the L2 every step and run back to back."""
    import torch
    from combine_persistent_warp_gb300 import FusedMoE, native
    from combine_persistent_warp_gb300.workloads import make_inputs

    dev = torch.device("cuda", dist.local_rank)
    inp = make_inputs(name, device=dev)
    wl = inp.wl
    model = work_model(inp)
    M = model["M"]
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R).reserve(wl.T)
    moe.load(inp)   # FP8 or MXFP4 weights, by the workload
    if args.ffn_mode:
        moe.set_option(native.OPT_FFN_MODE, args.ffn_mode)
    if wl.scales == "pow2":   # power-of-two scales: the hardware block-scaled path
        moe.set_option(native.OPT_SCALE_MODE, 1)
    # the automatic mode runs the combine inside the FFN kernel only for an output in pinned host
    # memory (the end-to-end loop below, not the device-buffer loop) and only on the block-scaled
    # kernel (power-of-two scales or MXFP4 weights)
    in_ffn = args.combine == "in-ffn"
    block_scaled = wl.scales == "pow2" or wl.weights == "mxfp4"
    moe.set_option(native.OPT_COMBINE_MODE, {"kernel": native.COMBINE_KERNEL, "in-ffn": native.COMBINE_IN_FFN,
                                             "auto": native.COMBINE_AUTO}[args.combine])
    if in_ffn:
        # the FFN kernel also reads the bf16 planes back and writes the output
        model["stages"]["expert_ffn"]["bytes"] += model["stages"]["combine"]["bytes"]
        model["stages"]["expert_ffn"]["flops"] += model["stages"]["combine"]["flops"]
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = needs_l2_flush(model)
    scratch = _l2_flush_buffer(torch, dev) if flush else None

    for _ in range(warmup):
        moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w, out=out)
    torch.cuda.synchronize()
    if moe.get_error() != 0:
        raise RuntimeError(f"{name}: device error during warm-up")

    # per-kernel CUDA events on every PROFILE_EVERY-th step of the timed region (events
    # between kernels serialise them, so recording them on every step would slow it)
    moe.profile_enable(True, every=1 if flush else PROFILE_EVERY)
    dist.barrier()
    torch.cuda.synchronize()
    h0 = time.time()
    if flush:
        local_s = 0.0
        for _ in range(steps):
            scratch.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w, out=out)
            e1.record(stream)
            e1.synchronize()
            local_s += e0.elapsed_time(e1) / 1e3
    else:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w, out=out)
        ev1.record(stream)
        torch.cuda.synchronize()
        local_s = ev0.elapsed_time(ev1) / 1e3
    h1 = time.time()
    dist.barrier()
    prof = moe.profile_read()
    moe.profile_enable(False)
    if moe.get_error() != 0:
        raise RuntimeError(f"{name}: device error during the timed region")
    value, t_max = aggregate(M * steps, local_s, dist)
    stage_ms = dict(prof["stage_ms"])
    if in_ffn:
        stage_ms.pop("combine", None)   # no combine launch: its events only bracket nothing
    calls = max(1, prof["calls"])
    dominant = max(stage_ms, key=stage_ms.get)
    res = {
        "value": value, "unit": UNIT, "steps": steps, "warmup": warmup,
        "ms_per_step": t_max / steps * 1e3,
        "config": config_of(wl, model, dist.world, flush),
        "combine": {"device_buffers": "inside the expert FFN kernel" if in_ffn else "separate kernel",
                    "host_buffers": ("inside the expert FFN kernel"
                                     if args.combine == "in-ffn" or (args.combine == "auto" and block_scaled)
                                     else "separate kernel")},
        "roofline": roofline_for(dominant, stage_ms[dominant] / calls / 1e3, model, wl.name, fp8_measured),
        "layer_roofline": layer_roofline(model, t_max / steps, fp8_measured),
        "stages_us_per_launch": {k: v / calls * 1e3 for k, v in stage_ms.items()},
        "stage_events": {"every_nth_step": 1 if flush else PROFILE_EVERY, "steps_with_events": prof["calls"]},
        "gpu_launches": (2 if in_ffn else 3) * steps,
        "dtype": ("fp8e4m3 x e2m1 (MXFP4 weights; fp32 accumulate, bf16 out)" if wl.weights == "mxfp4"
                  else "fp8e4m3 (fp32 accumulate, bf16 out)"),
    }
    if sampler is not None:
        res["clocks"] = sampler.summary(h0, h1)

    if e2e_steps > 0:
        # end to end through the host-buffer entry point: pinned host inputs read and the
        # result written back every step inside the timed region (moe_forward_host_async,
        # which lets the host enqueue step i+1 while step i runs)
        pin = lambda t: t.cpu().pin_memory()
        hx, hsf, hidx, hw = pin(inp.x), pin(inp.x_sf), pin(inp.topk_idx), pin(inp.topk_w)
        hout = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
        for _ in range(max(3, min(warmup, 20))):
            moe.forward_host(hx, hsf, hidx, hw, out=hout, wait=False)
        dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            moe.forward_host(hx, hsf, hidx, hw, out=hout, wait=False)
        e1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        if moe.get_error() != 0:
            raise RuntimeError(f"{name}: device error in the end-to-end loop")
        e2e_value = aggregate(M * e2e_steps, e0.elapsed_time(e1) / 1e3, dist)[0]
        res["e2e"] = {"value": e2e_value, "unit": UNIT,
                      "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (hx, hsf, hidx, hw)),
                      "d2h_bytes_per_step": hout.numel() * hout.element_size(), "steps": e2e_steps,
                      "entry_point": "moe_forward_host_async (one stream, synchronized after the last step)"}
        del hx, hsf, hidx, hw, hout
    if cpu_seconds is not None and dist.rank == 0 and dist.world == 1:
        res["cpu_baseline"] = cpu_baseline(inp, args.cpu_tokens, cpu_seconds)
    moe.close()
    del inp, out, scratch
    torch.cuda.empty_cache()
    return res


def run_ours(args, dist: Dist) -> dict | None:
    import torch

    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    fp8_tflops = measure_fp8_gemm_tflops(dev) if not args.no_fp8_peak else None
    sampler = ClockSampler(gpu_query_id(torch, dist.local_rank))
    sampler.start()
    time.sleep(0.3)
    try:
        head = bench_config(args.workload, args, dist, args.steps, args.warmup,
                            e2e_steps=max(1, min(args.steps, args.e2e_steps)),
                            cpu_seconds=None if args.no_cpu_baseline else args.cpu_seconds,
                            fp8_measured=fp8_tflops, sampler=sampler)
        per = {}
        for name in [n for n in args.per_config.split(",") if n and n != args.workload]:
            small = name.split("-")[0] in ("tiny", "decode")
            per[name] = bench_config(name, args, dist, max(args.steps, 200) if small else args.steps,
                                     max(args.warmup, 5),
                                     e2e_steps=max(1, min(args.steps, args.e2e_steps)),
                                     cpu_seconds=None if args.no_cpu_baseline else args.per_config_cpu_seconds,
                                     fp8_measured=fp8_tflops, sampler=sampler)
    finally:
        time.sleep(0.15)
        sampler.stop()
    res = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": head["dtype"], "data": "synthetic", "config": head["config"],
        "e2e": head["e2e"], "gpu_launches": head["gpu_launches"], "roofline": head["roofline"],
        "layer_roofline": head["layer_roofline"], "stages_us_per_launch": head["stages_us_per_launch"],
        "stage_events": head["stage_events"], "clocks": head.get("clocks"), "combine": head["combine"],
        "fp8_gemm_tflops_measured": fp8_tflops,
    }
    if "cpu_baseline" in head:
        res["cpu_baseline"] = head["cpu_baseline"]
    if per:
        res["per_config"] = per
        res["clocks_whole_run"] = sampler.summary(0.0, time.time())
    return res if dist.rank == 0 else None


def run_reference(args, dist: Dist) -> dict | None:
    """The CPU oracle as the reference arm: each step is a bounded sample of the batch."""
    import numpy as np
    import oracle
    from combine_persistent_warp_gb300.workloads import make_inputs

    if dist.rank != 0:
        return None
    import torch
    # the inputs are synthesised where the other arm makes them (the device generator draws
    # other numbers than the CPU one), then copied to the host
    if torch.cuda.is_available():
        inp = make_inputs(args.workload, device=torch.device("cuda", dist.local_rank)).to("cpu")
        torch.cuda.empty_cache()
    else:
        inp = make_inputs(args.workload, device="cpu")
    oracle.set_scale_rule(inp.wl.scales)
    wl = inp.wl
    model = work_model(inp)
    host = oracle.HostInputs.from_inputs(inp)
    h_idx = host.idx
    cores = oracle.num_threads()
    valid = np.argwhere(h_idx >= 0)
    # calibrate: one routed row on each core
    rng = np.random.default_rng(0)
    pick = valid[rng.choice(len(valid), min(cores, len(valid)), replace=False)]

    def step_rows(rows):
        mask = np.zeros_like(h_idx, dtype=bool)
        mask[rows[:, 0], rows[:, 1]] = True
        toks = np.unique(rows[:, 0])
        return oracle_rows_per_s(host, toks, row_mask=mask)

    _, dt_cal, _ = step_rows(pick[:1])
    t_row = max(dt_cal, 1e-4)                    # seconds per routed row on one core
    budget = args.ref_budget_s
    rows_per_step = max(1, int(budget * cores / ((args.steps + args.warmup) * t_row)))
    rows_per_step = min(rows_per_step, len(valid))
    order = valid[rng.permutation(len(valid))]
    cursor = 0

    def next_rows():
        nonlocal cursor
        if cursor + rows_per_step > len(order):
            cursor = 0
        r = order[cursor:cursor + rows_per_step]
        cursor += rows_per_step
        return r

    for _ in range(args.warmup):
        step_rows(next_rows())
    total_rows, total_s = 0, 0.0
    for _ in range(args.steps):
        _, dt, rows = step_rows(next_rows())
        total_rows += rows
        total_s += dt
    value = total_rows / total_s
    sample = (f"{rows_per_step} routed rows per step of the {wl.name} batch "
              f"({args.steps} steps, {total_s:.1f} s)")
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        # the workload's description as the other arm prints it (the CPU steps each take a
        # bounded sample of this batch: see cpu_baseline.sample)
        "config": config_of(wl, model, dist.world, needs_l2_flush(model)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)   # ~0.6 s timed at the large batch: several clock samples
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="large",
                    help="tiny, decode, prefill, skewed, large, or one of them with -pow2 "
                         "(power-of-two scales: the block-scaled UMMA path) or -mxfp4 (MXFP4 "
                         "weights on the block-scaled path)")
    ap.add_argument("--per-config", default="tiny,decode,prefill,skewed",
                    help="comma-separated workloads also timed in the same run (reported under "
                         "per_config; empty for none)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--cpu-tokens", type=int, default=128)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum wall time of the oracle baseline sample (repeated passes)")
    ap.add_argument("--per-config-cpu-seconds", type=float, default=3.0)
    ap.add_argument("--ref-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8-peak", action="store_true")
    ap.add_argument("--ffn-mode", type=int, default=0,
                    help="expert FFN kernel mode: 0 automatic, 1 one CTA per tile")
    ap.add_argument("--combine", choices=["auto", "kernel", "in-ffn"], default="auto",
                    help="top-k combine: a separate kernel, inside the expert FFN kernel, or automatic "
                         "(inside the block-scaled FFN kernel for an output in pinned host memory)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist = Dist(init=args.impl == "ours")
    try:
        res = run_reference(args, dist) if args.impl == "reference" else run_ours(args, dist)
        if res is not None:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
