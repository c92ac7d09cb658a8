"""CPU oracle of the fused FP8 MoE layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product library never loads it, and it shares no code
with the CUDA path: the arithmetic lives in ``moe_oracle.c`` (plain C, fp64 sums),
this module only marshals numpy arrays into it.

Pins (what ties each function to something other than itself) are in
``tests/test_oracle_pins.py``:
  * e4m3 codec        -- all 256 codes and in-range rounding vs. torch.float8_e4m3fn,
                         tie-to-even midpoints, saturation closed forms
  * bf16 rounding     -- vs. torch's bfloat16 cast
  * packed claim      -- worked example (3 then 2 -> start 3, word (2<<32)|5)
  * round robin       -- worked example 3/5/2 and position 7 -> (source 1, slot 2);
                         brute-force enumeration of every count vector R<=4, counts<=5
  * block offsets     -- worked example 100/10/30
  * expert FFN        -- single expert, k=1, w=1 reduces to a dense FFN checked against
                         numpy matmuls + torch FP8 casts; zero down weights; identical
                         experts; linearity in the gate weights
  * combine           -- closed form 0.73*E2(T0) + 0.27*E7(T0); the bf16-plane diagnostic
                         mode against numpy (bf16 casts by torch) on the per-slot outputs
  * power-of-two scale rule -- closed forms (exact powers, neighbours), the defining
                         inequalities sf/2 < q <= sf, and the requantised stage against
                         numpy with the rule applied by exponent arithmetic
  * MXFP4 weights     -- all 16 E2M1 codes against the OCP MX element table, E8M0 bytes
                         against 2^(b-127), nibble order and per-32 scale index by single-
                         element weights, and the whole layer against its FP8 twin (the
                         same weight values written as e4m3 codes with 128x128 scales)
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        L.orc_init.restype = None
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode_array.argtypes = [ctypes.c_int64, P, P]
        L.orc_e4m3_decode_array.argtypes = [ctypes.c_int64, P, P]
        L.orc_bf16_rne_array.argtypes = [ctypes.c_int64, P, P]
        L.orc_packed_claim.restype = ctypes.c_uint64
        L.orc_packed_claim.argtypes = [ctypes.c_int, P, P]
        L.orc_round_robin.restype = ctypes.c_int
        L.orc_round_robin.argtypes = [ctypes.c_int, P, P, P]
        L.orc_round_robin_one.restype = ctypes.c_int
        L.orc_round_robin_one.argtypes = [ctypes.c_int, P, ctypes.c_uint32, P, P]
        L.orc_block_offsets.argtypes = [ctypes.c_int, P, ctypes.c_int, P]
        L.orc_route_counts.restype = ctypes.c_int
        L.orc_route_counts.argtypes = [ctypes.c_int] * 4 + [P, P, P]
        L.orc_expert_ffn.argtypes = [ctypes.c_int, ctypes.c_int] + [P] * 9
        L.orc_set_scale_rule.argtypes = [ctypes.c_int]
        L.orc_set_scale_rule.restype = None
        L.orc_set_plane_bf16.argtypes = [ctypes.c_int]
        L.orc_set_plane_bf16.restype = None
        L.orc_pow2_ceil.argtypes = [ctypes.c_float]
        L.orc_pow2_ceil.restype = ctypes.c_float
        L.orc_forward_tokens.restype = ctypes.c_int
        L.orc_forward_tokens.argtypes = [ctypes.c_int] * 5 + [P] * 8 + [ctypes.c_int, P, P, P]
        L.orc_forward_tokens_fmt.restype = ctypes.c_int
        L.orc_forward_tokens_fmt.argtypes = [ctypes.c_int] * 6 + [P] * 8 + [ctypes.c_int, P, P, P]
        L.orc_expert_ffn_fmt.argtypes = [ctypes.c_int] * 3 + [P] * 9
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e8m0_decode.restype = ctypes.c_double
        L.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
        L.orc_num_threads.restype = ctypes.c_int
        L.orc_init()
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(t, dtype):
    """torch tensor or array-like -> contiguous numpy array of ``dtype`` (host copy)."""
    if hasattr(t, "detach"):
        t = t.detach().cpu()
        if dtype == np.uint8:
            import torch
            t = t.view(torch.uint8) if t.dtype != torch.uint8 else t
        t = t.numpy()
    return np.ascontiguousarray(np.asarray(t), dtype=dtype)


# ------------------------------------------------------------- scalar codecs ---
def e4m3_decode(codes) -> np.ndarray:
    c = _np(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_e4m3_decode_array(c.size, _p(c), _p(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    v = _np(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(v.size, _p(v), _p(out))
    return out


def bf16_rne(values) -> np.ndarray:
    """fp32 -> bf16 bits (uint16), round to nearest even."""
    v = _np(values, np.float32)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_rne_array(v.size, _p(v), _p(out))
    return out


def bf16_bits_to_float(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ routing ---
def packed_claim(counts):
    c = np.ascontiguousarray(counts, dtype=np.uint32)
    starts = np.empty(c.shape, np.uint32)
    word = lib().orc_packed_claim(c.size, _p(c), _p(starts))
    return starts, int(word)


def round_robin(recv):
    """(source, slot) of every position of one expert's received rows."""
    r = np.ascontiguousarray(recv, dtype=np.uint32)
    n = int(r.sum())
    src = np.empty(n, np.uint32)
    slot = np.empty(n, np.uint32)
    if lib().orc_round_robin(r.size, _p(r), _p(src), _p(slot)):
        raise ValueError("round robin failed")
    return src, slot


def round_robin_one(recv, p: int):
    r = np.ascontiguousarray(recv, dtype=np.uint32)
    s = np.zeros(1, np.uint32)
    sl = np.zeros(1, np.uint32)
    if lib().orc_round_robin_one(r.size, _p(r), p, _p(s), _p(sl)):
        raise ValueError("position beyond the expert's rows")
    return int(s[0]), int(sl[0])


def block_offsets(counts, BM: int) -> np.ndarray:
    c = np.ascontiguousarray(counts, dtype=np.uint32)
    off = np.empty(c.size + 1, np.int32)
    lib().orc_block_offsets(c.size, _p(c), BM, _p(off))
    return off


def route_counts(topk_idx, E: int, R: int):
    """(counts [E], recv [E,R], bad) by direct counting."""
    idx = _np(topk_idx, np.int64)
    T, k = idx.shape
    counts = np.empty(E, np.uint32)
    recv = np.empty((E, R), np.uint32)
    bad = lib().orc_route_counts(T, k, E, R, _p(idx), _p(counts), _p(recv))
    return counts, recv, bool(bad)


def route_multiset(topk_idx, E: int, R: int):
    """For each (expert, source): sorted list of (token, slot k) routed there."""
    idx = _np(topk_idx, np.int64)
    T, k = idx.shape
    Tsrc = T // R
    out = {(e, r): [] for e in range(E) for r in range(R)}
    ts, ks = np.nonzero(idx >= 0)
    for t, kk in zip(ts.tolist(), ks.tolist()):
        out[(int(idx[t, kk]), t // Tsrc)].append((t, kk))
    for v in out.values():
        v.sort()
    return out


# -------------------------------------------------------------------- numerics -
def set_scale_rule(rule: str):
    """SwiGLU re-quantisation scale rule: "fp32" (max(amax,1e-4)/448) or "pow2" (the
    smallest power of two >= that quotient)."""
    if rule not in ("fp32", "pow2"):
        raise ValueError(rule)
    lib().orc_set_scale_rule(1 if rule == "pow2" else 0)


def set_plane_bf16(on: bool):
    """Diagnostic combine: each slot's weighted output rounded to a bf16 plane value, planes
    summed in fp32 ascending k (as the bf16 combine buffer + fp32 reduce do); default off:
    the top-k sum kept in double."""
    lib().orc_set_plane_bf16(1 if on else 0)


def pow2_ceil(v: float) -> float:
    """Smallest power of two >= v (positive normal fp32 v)."""
    return float(lib().orc_pow2_ceil(float(v)))


WEIGHT_FORMATS = {"fp8": 0, "mxfp4": 1}


def e2m1_decode(codes) -> np.ndarray:
    """Values of FP4 E2M1 codes (low 4 bits of each byte)."""
    c = _np(codes, np.uint8)
    return np.array([lib().orc_e2m1_decode(int(v) & 0xF) for v in c.ravel()], np.float64).reshape(c.shape)


def e8m0_decode(codes) -> np.ndarray:
    """Values of E8M0 scale bytes."""
    c = _np(codes, np.uint8)
    return np.array([lib().orc_e8m0_decode(int(v)) for v in c.ravel()], np.float64).reshape(c.shape)


def expert_ffn(x_row, xsf_row, w1_e, s1_e, w2_e, s2_e, weights: str = "fp8"):
    """One expert on one token: (y [H] float64, hq [I] uint8, hsf [I/128] float32).

    weights "fp8": w1 [2I][H] e4m3, s1 [2I/128][H/128] fp32, w2 [H][I], s2 [H/128][I/128];
    "mxfp4": w1 [2I][H/2] packed E2M1, s1 [2I][H/32] E8M0, w2 [H][I/2], s2 [H][I/32]."""
    fmt = WEIGHT_FORMATS[weights]
    sdt = np.uint8 if fmt else np.float32
    x = _np(x_row, np.uint8)
    xs = _np(xsf_row, np.float32)
    w1 = _np(w1_e, np.uint8)
    s1 = _np(s1_e, sdt)
    w2 = _np(w2_e, np.uint8)
    s2 = _np(s2_e, sdt)
    H = x.size
    I = w2.shape[-1] * (2 if fmt else 1)
    y = np.empty(H, np.float64)
    hq = np.empty(I, np.uint8)
    hsf = np.empty(I // 128, np.float32)
    lib().orc_expert_ffn_fmt(fmt, H, I, _p(x), _p(xs), _p(w1), _p(s1), _p(w2), _p(s2),
                             _p(y), _p(hq), _p(hsf))
    return y, hq, hsf


class HostInputs:
    """Host copies of one workload's inputs, in the layouts the oracle reads (weight
    layouts of ``weights`` as in ``expert_ffn``)."""

    def __init__(self, x, x_sf, topk_idx, topk_w, w_gate_up, sf_gate_up, w_down, sf_down,
                 weights: str = "fp8"):
        self.weights = weights
        fmt = WEIGHT_FORMATS[weights]
        sdt = np.uint8 if fmt else np.float32
        self.x = _np(x, np.uint8)
        self.x_sf = _np(x_sf, np.float32)
        self.idx = _np(topk_idx, np.int64)
        self.w = _np(topk_w, np.float32)
        self.w1 = _np(w_gate_up, np.uint8)
        self.s1 = _np(sf_gate_up, sdt)
        self.w2 = _np(w_down, np.uint8)
        self.s2 = _np(sf_down, sdt)
        self.T, self.H = self.x.shape if self.x.ndim == 2 else (0, self.w2.shape[1])
        self.E, twoI, _ = self.w1.shape
        self.I = twoI // 2
        self.k = self.idx.shape[1]

    @classmethod
    def from_inputs(cls, inp):
        return cls(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w, inp.w_gate_up, inp.sf_gate_up,
                   inp.w_down, inp.sf_down, weights=getattr(inp.wl, "weights", "fp8"))


def forward_tokens(h: HostInputs, tokens):
    """Layer output for the given tokens: (bf16 bits [n,H] uint16, fp32 [n,H], bad)."""
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    n = tok.size
    out = np.empty((n, h.H), np.uint16)
    out32 = np.empty((n, h.H), np.float32)
    bad = lib().orc_forward_tokens_fmt(WEIGHT_FORMATS[h.weights], h.T, h.H, h.I, h.E, h.k,
                                       _p(h.x), _p(h.x_sf), _p(h.idx), _p(h.w), _p(h.w1),
                                       _p(h.s1), _p(h.w2), _p(h.s2), n, _p(tok), _p(out),
                                       _p(out32))
    return out, out32, bool(bad)


def num_threads() -> int:
    return int(lib().orc_num_threads())
