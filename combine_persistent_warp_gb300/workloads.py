"""Seeded synthetic workloads for the fused MoE layer.

This module only *synthesises inputs*: routing decisions, FP8 activations with
1x128 fp32 scales, and FP8 expert weights with 128x128 fp32 block scales (or
MXFP4 expert weights: E2M1 codes with one E8M0 scale per 32 elements).  It
holds none of the layer's own arithmetic (no GEMM, no SwiGLU, no combine).  The
FP8 encoding of the synthetic tensors is done by PyTorch's ``float8_e4m3fn``
cast (a library routine); both the CUDA path and the CPU oracle receive the
resulting bytes and scales as plain inputs.

The five named workloads follow the shapes of the layer the pages describe
(hidden 7168 / intermediate 2048 decode and prefill, a Zipf-skewed prefill with
skipped slots, a 128-expert large case, and a tiny case the oracle finishes in
well under a second).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, asdict

import torch

FP8_MAX = 448.0          # largest finite e4m3 magnitude (OCP FP8 E4M3)
SCALE_FLOOR = 1e-4       # amax floor so an all-zero group still gets a finite scale


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # tokens
    H: int                 # hidden size
    I: int                 # expert intermediate size (gate_up has 2*I rows)
    E: int                 # experts (all local)
    topk: int
    R: int                 # logical source partitions of T/R tokens each
    routing: str = "uniform"   # "uniform" or "zipf"
    zipf_s: float = 0.0
    skip_frac: float = 0.0     # fraction of topk_idx entries set to -1
    seed: int = 0
    scales: str = "fp32"       # "fp32": sf = max(amax,1e-4)/448; "pow2": the smallest power
                               # of two >= that (UE8M0-representable, block-scaled UMMA path)
    weights: str = "fp8"       # "fp8": e4m3 with 128x128 scales; "mxfp4": E2M1 with 1x32
                               # E8M0 scales (needs scales == "pow2")

    @property
    def T_src(self) -> int:
        return self.T // self.R

    def describe(self) -> dict:
        return asdict(self)


WORKLOADS = {
    "tiny": Workload("tiny", T=64, H=256, I=128, E=8, topk=2, R=2, seed=0),
    "decode": Workload("decode", T=128, H=7168, I=2048, E=32, topk=8, R=8, seed=1),
    "prefill": Workload("prefill", T=4096, H=7168, I=2048, E=32, topk=8, R=8, seed=2),
    "skewed": Workload("skewed", T=8192, H=7168, I=2048, E=64, topk=8, R=8,
                       routing="zipf", zipf_s=1.2, skip_frac=0.05, seed=3),
    "large": Workload("large", T=16384, H=4096, I=1536, E=128, topk=8, R=8, seed=4),
}
# the same batches with power-of-two (UE8M0-representable) scales everywhere
POW2_WORKLOADS = {f"{k}-pow2": Workload(**{**asdict(v), "name": f"{k}-pow2", "scales": "pow2"})
                  for k, v in WORKLOADS.items()}


# the same batches with MXFP4 expert weights (and power-of-two activation scales)
MXFP4_WORKLOADS = {f"{k}-mxfp4": Workload(**{**asdict(v), "name": f"{k}-mxfp4", "scales": "pow2",
                                            "weights": "mxfp4"})
                   for k, v in WORKLOADS.items()}


def workload(name: str) -> Workload:
    for table in (WORKLOADS, POW2_WORKLOADS, MXFP4_WORKLOADS):
        if name in table:
            return table[name]
    raise KeyError(name)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


# ---------------------------------------------------------------- routing ---
def make_routing(T: int, E: int, topk: int, *, seed: int, routing: str = "uniform",
                 zipf_s: float = 0.0, skip_frac: float = 0.0):
    """Top-k expert choice per token, drawn without replacement from softmax(logits).

    logits ~ N(0,1) [T,E]; for "zipf" a log-prior log p_e with p_e ~ 1/rank^s over a
    fixed random permutation of the experts is added.  Sampling without replacement
    uses Gumbel-top-k; the gate weights are the chosen softmax probabilities,
    renormalised to sum to one.  A ``skip_frac`` share of (token, slot) entries is
    then set to -1 (their weights are kept).  Runs on the CPU so every device sees
    the same routing.
    """
    g = _gen(seed * 7919 + 17, "cpu")
    logits = torch.randn(T, E, generator=g, dtype=torch.float64)
    if routing == "zipf":
        perm = torch.randperm(E, generator=g)
        ranks = torch.empty(E, dtype=torch.float64)
        ranks[perm] = torch.arange(1, E + 1, dtype=torch.float64)
        prior = ranks.pow(-zipf_s)
        prior = prior / prior.sum()
        logits = logits + prior.log()[None, :]
    elif routing != "uniform":
        raise ValueError(routing)
    u = torch.rand(T, E, generator=g, dtype=torch.float64).clamp_(1e-300, 1.0)
    gumbel = -torch.log(-torch.log(u))
    idx = torch.topk(logits + gumbel, topk, dim=1).indices
    probs = torch.softmax(logits, dim=1)
    w = probs.gather(1, idx)
    w = (w / w.sum(dim=1, keepdim=True)).to(torch.float32)
    idx = idx.to(torch.int64)
    if skip_frac > 0:
        n_skip = int(round(skip_frac * T * topk))
        flat = torch.randperm(T * topk, generator=g)[:n_skip]
        idx.view(-1)[flat] = -1
    return idx.contiguous(), w.contiguous()


# ------------------------------------------------------ FP8 synthesis -------
def pow2_ceil(v: torch.Tensor) -> torch.Tensor:
    """Smallest power of two >= v (positive fp32): v = m * 2^e with m in [0.5, 1)."""
    m, e = torch.frexp(v)
    return torch.where(m == 0.5, v, torch.ldexp(torch.ones_like(v), e))


def quantize_1x128(x: torch.Tensor, scales: str = "fp32"):
    """fp32 [rows, K] -> (e4m3 bytes uint8 [rows, K], fp32 scales [rows, K/128])."""
    rows, K = x.shape
    g = x.float().view(rows, K // 128, 128)
    sf = g.abs().amax(dim=2).clamp_min(SCALE_FLOOR) / FP8_MAX
    if scales == "pow2":
        sf = pow2_ceil(sf)
    q = (g / sf[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.view(rows, K).contiguous(), sf.contiguous()


def quantize_128x128(w: torch.Tensor, scales: str = "fp32"):
    """fp32 [N, K] -> (e4m3 bytes uint8 [N, K], fp32 scales [N/128, K/128])."""
    N, K = w.shape
    g = w.float().view(N // 128, 128, K // 128, 128)
    sf = g.abs().amax(dim=(1, 3)).clamp_min(SCALE_FLOOR) / FP8_MAX
    if scales == "pow2":
        sf = pow2_ceil(sf)
    q = (g / sf[:, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.view(N, K).contiguous(), sf.contiguous()


def make_weights(E: int, H: int, I: int, *, seed: int, device="cpu", std: float = 0.02,
                 scales: str = "fp32"):
    """Expert weights W ~ N(0, std) as FP8 with 128x128 fp32 block scales.

    Returns w_gate_up uint8 [E, 2I, H] (rows 0..I-1 gate, I..2I-1 up),
    sf_gate_up fp32 [E, 2I/128, H/128], w_down uint8 [E, H, I], sf_down fp32
    [E, H/128, I/128].  Generated one expert at a time on ``device``.
    """
    g = _gen(seed * 104729 + 3, device)
    w1 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=device)
    s1 = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device=device)
    w2 = torch.empty(E, H, I, dtype=torch.uint8, device=device)
    s2 = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=device)
    for e in range(E):
        a = torch.randn(2 * I, H, generator=g, device=device) * std
        w1[e], s1[e] = quantize_128x128(a, scales)
        b = torch.randn(H, I, generator=g, device=device) * std
        w2[e], s2[e] = quantize_128x128(b, scales)
    return w1, s1, w2, s2


# ------------------------------------------------------ MXFP4 synthesis -----
E2M1_MAX_EXP = 2                      # exponent of the largest E2M1 magnitude, 6 = 1.5 * 2^2
E2M1_MAGS = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)   # codes 0..7 (bit 3 = sign)


def quantize_mxfp4(w: torch.Tensor):
    """fp32 [N, K] -> (packed E2M1 bytes uint8 [N, K/2], E8M0 scale bytes uint8 [N, K/32]).

    OCP Microscaling conversion: each run of 32 elements of a row shares the scale
    X = 2^(floor(log2(amax)) - 2) (2 = the largest E2M1 exponent; an all-zero run takes
    X = 2^-127), stored as the byte log2(X) + 127; each element becomes the nearest E2M1
    value of v / X (ties to the even code), saturated to +-6.  Element 2j sits in the low
    nibble of byte j, element 2j + 1 in the high nibble."""
    N, K = w.shape
    g = w.float().view(N, K // 32, 32)
    amax = g.abs().amax(dim=2)
    _, e = torch.frexp(amax)                       # amax = m * 2^e, m in [0.5, 1)
    sexp = torch.where(amax > 0, e - 1 - E2M1_MAX_EXP, torch.full_like(e, -127)).clamp(-127, 127)
    a = (g / torch.ldexp(torch.ones_like(amax), sexp)[:, :, None]).abs()
    mags = torch.tensor(E2M1_MAGS, device=w.device)
    mids = (mags[1:] + mags[:-1]) / 2
    lo = torch.bucketize(a, mids, right=False)     # ties -> the smaller magnitude
    hi = torch.bucketize(a, mids, right=True)      # ties -> the larger magnitude
    code = torch.where(lo % 2 == 0, lo, hi).to(torch.uint8)
    code = code | ((g < 0) & (code > 0)).to(torch.uint8) << 3
    code = code.view(N, K)
    packed = code[:, 0::2] | (code[:, 1::2] << 4)
    return packed.contiguous(), (sexp + 127).to(torch.uint8).contiguous()


def make_weights_mxfp4(E: int, H: int, I: int, *, seed: int, device="cpu", std: float = 0.02):
    """Expert weights W ~ N(0, std) (the same draws as ``make_weights``) as MXFP4.

    Returns w_gate_up uint8 [E, 2I, H/2] (rows 0..I-1 gate, I..2I-1 up), sf_gate_up uint8
    [E, 2I, H/32], w_down uint8 [E, H, I/2], sf_down uint8 [E, H, I/32]."""
    g = _gen(seed * 104729 + 3, device)
    w1 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=device)
    s1 = torch.empty(E, 2 * I, H // 32, dtype=torch.uint8, device=device)
    w2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=device)
    s2 = torch.empty(E, H, I // 32, dtype=torch.uint8, device=device)
    for e in range(E):
        a = torch.randn(2 * I, H, generator=g, device=device) * std
        w1[e], s1[e] = quantize_mxfp4(a)
        b = torch.randn(H, I, generator=g, device=device) * std
        w2[e], s2[e] = quantize_mxfp4(b)
    return w1, s1, w2, s2


def make_activations(T: int, H: int, *, seed: int, device="cpu", scales: str = "fp32"):
    """x ~ N(0,1), rounded to bf16, then FP8 e4m3 with 1x128 fp32 scales."""
    g = _gen(seed * 15485863 + 11, device)
    x = torch.randn(T, H, generator=g, device=device).to(torch.bfloat16).float()
    if T == 0:
        return (torch.empty(0, H, dtype=torch.uint8, device=device),
                torch.empty(0, H // 128, dtype=torch.float32, device=device))
    return quantize_1x128(x, scales)


@dataclass
class Inputs:
    wl: Workload
    x: torch.Tensor
    x_sf: torch.Tensor
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    w_gate_up: torch.Tensor
    sf_gate_up: torch.Tensor
    w_down: torch.Tensor
    sf_down: torch.Tensor
    extra: dict = field(default_factory=dict)

    def to(self, device) -> "Inputs":
        mv = lambda t: t.to(device)
        return Inputs(self.wl, mv(self.x), mv(self.x_sf), mv(self.topk_idx), mv(self.topk_w),
                      mv(self.w_gate_up), mv(self.sf_gate_up), mv(self.w_down),
                      mv(self.sf_down), dict(self.extra))


def make_inputs(wl: Workload | str, device="cpu", *, T: int | None = None) -> Inputs:
    """All inputs of one workload.  ``T`` overrides the token count (same seed)."""
    if isinstance(wl, str):
        wl = workload(wl)
    if T is not None and T != wl.T:
        wl = Workload(**{**asdict(wl), "T": T})
    idx, w = make_routing(wl.T, wl.E, wl.topk, seed=wl.seed, routing=wl.routing,
                          zipf_s=wl.zipf_s, skip_frac=wl.skip_frac)
    x, x_sf = make_activations(wl.T, wl.H, seed=wl.seed, device=device, scales=wl.scales)
    if wl.weights == "mxfp4":
        w1, s1, w2, s2 = make_weights_mxfp4(wl.E, wl.H, wl.I, seed=wl.seed, device=device)
    else:
        w1, s1, w2, s2 = make_weights(wl.E, wl.H, wl.I, seed=wl.seed, device=device, scales=wl.scales)
    return Inputs(wl, x, x_sf, idx.to(device), w.to(device), w1, s1, w2, s2)


def routed_rows(topk_idx: torch.Tensor) -> int:
    """M = number of (token, slot) entries that name an expert."""
    return int((topk_idx >= 0).sum().item())


def expert_rows(topk_idx: torch.Tensor, E: int) -> torch.Tensor:
    v = topk_idx[topk_idx >= 0].flatten().cpu()
    return torch.bincount(v, minlength=E)


def skew_ratio(topk_idx: torch.Tensor, E: int) -> float:
    c = expert_rows(topk_idx, E).double()
    return float(c.max() / c.mean()) if c.sum() > 0 else math.nan
