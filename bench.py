#!/usr/bin/env python3
"""Benchmark of the fused FP8 MoE layer on GB300.

One step = one forward of the whole layer (routing, gather, gate_up GEMM + SwiGLU +
requant, down GEMM + weighted scatter, combine) over one synthetic batch.  The default
workload is the decode batch: T=128 tokens, H=7168, I=2048, E=32, topk=8, R=8, uniform
routing, FP8 e4m3 activations and weights with fp32 block scales.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line.  ``value`` is routed (token, slot) rows per second of the whole
job with inputs resident in HBM, timed with CUDA events on the forward's stream; ``e2e``
is the same metric through ``moe_forward_host`` (pinned host buffers, copies inside the
timed region).  ``roofline`` covers the dominant kernel, timed live with CUDA events the
library records around each of its kernels.  ``--impl reference`` times the plain CPU
oracle on a bounded sample of the same workload instead (the reference arm).
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
    ("decode", "expert_ffn"): {"bytes": 1425256448 + 14529792, "src_sha": "fbc87d810249e61e"},
    ("prefill", "expert_ffn"): {"bytes": 1892651264 + 534686208, "src_sha": "fbc87d810249e61e"},
    ("decode-pow2", "expert_ffn"): {"bytes": 1431475200 + 3602944, "src_sha": "471a697d4cd814f3"},
    ("prefill-pow2", "expert_ffn"): {"bytes": 2108371200 + 514178816, "src_sha": "471a697d4cd814f3"},
    ("decode-mxfp4", "expert_ffn"): {"bytes": 759860224 + 3274752, "src_sha": "471a697d4cd814f3"},
    ("prefill-mxfp4", "expert_ffn"): {"bytes": 1060229888 + 511471872, "src_sha": "471a697d4cd814f3"},
}
# sources each stage's kernel is compiled from (a recorded traffic figure is used only while
# these hash to its `src_sha`)
KERNEL_SOURCES = {
    "expert_ffn": ["combine_persistent_warp_gb300/csrc/ffn.cu",
                   "combine_persistent_warp_gb300/csrc/ptx.cuh",
                   "combine_persistent_warp_gb300/csrc/moe_internal.cuh"],
    # power-of-two scales: the expert FFN stage runs the block-scaled kernel
    "expert_ffn_bs": ["combine_persistent_warp_gb300/csrc/ffn_bs.cu",
                      "combine_persistent_warp_gb300/csrc/ptx.cuh",
                      "combine_persistent_warp_gb300/csrc/moe_internal.cuh"],
    "dispatch": ["combine_persistent_warp_gb300/csrc/routing.cu",
                 "combine_persistent_warp_gb300/csrc/route_device.cuh",
                 "combine_persistent_warp_gb300/csrc/ptx.cuh",
                 "combine_persistent_warp_gb300/csrc/moe_internal.cuh"],
    "combine": ["combine_persistent_warp_gb300/csrc/routing.cu",
                "combine_persistent_warp_gb300/csrc/moe_internal.cuh"],
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
    """Algorithmic bytes and FLOPs of each stage for one forward (valid rows only)."""
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
    # expert_ffn = gate_up GEMM (W1, gathered rows in, SwiGLU rows out) + down GEMM (W2,
    # SwiGLU rows in, weighted bf16 rows out); one kernel
    st = {
        "dispatch": {"bytes": T * K * 8 + 2 * x_rows + M * (12 + 8), "flops": 0},
        "expert_ffn": {"bytes": w1 + w2 + x_rows + 2 * act_rows + M * H * 2 + M * 16,
                       "flops": 2 * M * H * 2 * I + 2 * M * I * H},
        "combine": {"bytes": M * H * 2 + T * H * 2 + T * K * 8, "flops": M * H},
    }
    compulsory = (w1 + w2 + T * (H + (H // 128) * 4) + T * K * 12 + T * H * 2)
    return {"M": M, "touched_experts": touched, "stages": st, "compulsory_bytes": compulsory,
            "flops": 6 * M * H * I, "weight_bytes": w1 + w2}


def peaks() -> tuple[dict, str]:
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"]))}, "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0}, "fallback"


def roofline_for(stage: str, avg_s: float, model: dict, workload: str) -> dict:
    pk, src = peaks()
    st = model["stages"][stage]
    bytes_ = st["bytes"]
    flops = st["flops"]
    t_hbm = bytes_ / (pk["hbm_gbs"] * 1e9)
    fp8_peak = pk["bf16_tflops"] * FP8_OVER_BF16
    t_tensor = flops / (fp8_peak * 1e12) if flops else 0.0
    traffic = None
    block_scaled = workload.endswith("-pow2") or workload.endswith("-mxfp4")
    src_key = "expert_ffn_bs" if stage == "expert_ffn" and block_scaled else stage
    rec = NCU_TRAFFIC.get((workload, stage))
    if rec and rec.get("src_sha") == kernel_sources_sha(src_key):
        traffic = rec["bytes"]
    if t_tensor > t_hbm and flops:
        achieved = flops / avg_s / 1e12
        return {"bound": "tensor", "kernel": stage, "kernel_fn": KERNEL_FN.get(src_key, stage),
                "achieved": achieved, "peak": fp8_peak,
                "unit": "TFLOP/s", "frac": achieved / fp8_peak, "traffic": traffic,
                "algorithmic_flops": flops, "peak_source": f"{src} bf16 x {FP8_OVER_BF16} (fp8/bf16 nominal)"}
    achieved = bytes_ / avg_s / 1e9
    return {"bound": "hbm", "kernel": stage, "kernel_fn": KERNEL_FN.get(src_key, stage),
            "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
            "algorithmic_bytes": bytes_, "peak_source": f"{src} (hbm_gbs, copy bandwidth)"}


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
    while passes == 0 or (total_dt < min_seconds and passes < 50):
        _, dt, rows = oracle_rows_per_s(host, toks)
        total_rows += rows
        total_dt += dt
        passes += 1
    return {"value": total_rows / total_dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{toks.size} tokens ({total_rows // passes} routed rows) of the {inp.wl.name} batch, "
                      f"{passes} passes, {total_dt:.1f} s wall"}


# ------------------------------------------------------------------ arms -----------
def run_ours(args, dist: Dist) -> dict | None:
    import torch
    from combine_persistent_warp_gb300 import FusedMoE
    from combine_persistent_warp_gb300.workloads import make_inputs

    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    inp = make_inputs(args.workload, device=dev)
    wl = inp.wl
    model = work_model(inp)
    M = model["M"]
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R).reserve(wl.T)
    moe.load(inp)   # FP8 or MXFP4 weights, by the workload
    from combine_persistent_warp_gb300 import native
    if args.ffn_mode:
        moe.set_option(native.OPT_FFN_MODE, args.ffn_mode)
    if wl.scales == "pow2":   # power-of-two scales: the hardware block-scaled path
        moe.set_option(native.OPT_SCALE_MODE, 1)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w, out=out)
    torch.cuda.synchronize()
    if moe.get_error() != 0:
        raise RuntimeError("device error during warm-up")

    sampler = ClockSampler(gpu_query_id(torch, dist.local_rank))
    sampler.start()
    time.sleep(0.3)
    # per-kernel CUDA events on every PROFILE_EVERY-th step of the timed region (events
    # between kernels serialise them, so recording them on every step would slow it)
    moe.profile_enable(True, every=PROFILE_EVERY)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    h0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w, out=out)
    ev1.record(stream)
    torch.cuda.synchronize()
    h1 = time.time()
    dist.barrier()
    prof = moe.profile_read()
    moe.profile_enable(False)
    time.sleep(0.15)
    sampler.stop()
    if moe.get_error() != 0:
        raise RuntimeError("device error during the timed region")
    local_s = ev0.elapsed_time(ev1) / 1e3
    value, t_max = aggregate(M * args.steps, local_s, dist)

    # end to end through the host-buffer entry points (pinned host inputs read and the
    # result written back every step inside the timed region): the asynchronous one, which
    # lets the host enqueue step i+1 while step i runs, and the synchronous one
    pin = lambda t: t.cpu().pin_memory()
    hx, hsf, hidx, hw = pin(inp.x), pin(inp.x_sf), pin(inp.topk_idx), pin(inp.topk_w)
    hout = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(1, min(args.steps, args.e2e_steps))

    def host_loop(wait: bool) -> float:
        for _ in range(max(3, min(args.warmup, 20))):
            moe.forward_host(hx, hsf, hidx, hw, out=hout, wait=wait)
        dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            moe.forward_host(hx, hsf, hidx, hw, out=hout, wait=wait)
        e1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        if moe.get_error() != 0:
            raise RuntimeError("device error in the end-to-end loop")
        return aggregate(M * e2e_steps, e0.elapsed_time(e1) / 1e3, dist)[0]

    e2e_value = host_loop(wait=False)
    e2e_sync_value = host_loop(wait=True)
    h2d = sum(t.numel() * t.element_size() for t in (hx, hsf, hidx, hw))
    d2h = hout.numel() * hout.element_size()

    stage_ms = prof["stage_ms"]
    calls = max(1, prof["calls"])
    dominant = max(stage_ms, key=stage_ms.get)
    roof = roofline_for(dominant, stage_ms[dominant] / calls / 1e3, model, wl.name)
    stages = {k: v / calls * 1e3 for k, v in stage_ms.items()}   # us per launch

    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("fp8e4m3 x e2m1 (MXFP4 weights; fp32 accumulate, bf16 out)" if wl.weights == "mxfp4"
                  else "fp8e4m3 (fp32 accumulate, bf16 out)"), "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
                   "topk": wl.topk, "R": wl.R, "routing": wl.routing, "scales": wl.scales,
                   "weights": wl.weights,
                   "routed_rows_per_step": M, "parallelism": f"replicas x{dist.world}",
                   "l2": ("inputs larger than L2: %.2f GB of expert weights streamed per step, "
                          "no flush" % (model["weight_bytes"] / 1e9))},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "entry_point": "moe_forward_host_async (one stream, synchronized after the last step)",
                "sync_value": e2e_sync_value,
                "sync_entry_point": "moe_forward_host (returns after each step)"},
        "gpu_launches": 3 * args.steps,
        "roofline": roof,
        "stages_us_per_launch": stages,
        "stage_events": {"every_nth_step": PROFILE_EVERY, "steps_with_events": prof["calls"]},
        "clocks": sampler.summary(h0, h1),
    }
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(inp, args.cpu_tokens, args.cpu_seconds)
    moe.close()
    return res if dist.rank == 0 else None


def run_reference(args, dist: Dist) -> dict | None:
    """The CPU oracle as the reference arm: each step is a bounded sample of the batch."""
    import numpy as np
    import oracle
    from combine_persistent_warp_gb300.workloads import make_inputs

    if dist.rank != 0:
        return None
    inp = make_inputs(args.workload, device="cpu")
    oracle.set_scale_rule(inp.wl.scales)
    wl = inp.wl
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
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
                   "topk": wl.topk, "R": wl.R, "routing": wl.routing, "scales": wl.scales,
                   "weights": wl.weights, "routed_rows_per_step": int(len(valid)),
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="decode",
                    help="tiny, decode, prefill, skewed, large, or one of them with -pow2 "
                         "(power-of-two scales: the block-scaled UMMA path) or -mxfp4 (MXFP4 "
                         "weights on the block-scaled path)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--cpu-tokens", type=int, default=128)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum wall time of the oracle baseline sample (repeated passes)")
    ap.add_argument("--ref-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ffn-mode", type=int, default=0,
                    help="expert FFN kernel mode: 0 automatic, 1 one CTA per tile, 2 CTA pairs")
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
