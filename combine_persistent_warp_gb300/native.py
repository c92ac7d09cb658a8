"""ctypes binding of the C ABI in include/cpw_moe.h (argument marshalling only).

Every step of the layer runs in the CUDA library ``libcpw_moe.so``; this module only
checks tensor shapes/dtypes, passes ``data_ptr()`` values and the CUDA stream handle,
and turns status codes into exceptions.  There is no fallback: if the library is
missing or cannot be loaded, importing the layer fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
HEADER = os.path.join(ROOT, "include", "cpw_moe.h")
LIB_PATH = os.path.join(PKG, "libcpw_moe.so")

MOE_OK = 0
STATUS = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_CUDA", 3: "MOE_ERR_CAPACITY",
    4: "MOE_ERR_NO_WEIGHTS", 5: "MOE_ERR_UNSUPPORTED_DEVICE", 6: "MOE_ERR_BAD_INDEX",
    7: "MOE_ERR_TIMEOUT", 8: "MOE_ERR_SLOT_OVERFLOW", 9: "MOE_ERR_NOT_RESERVED",
    10: "MOE_ERR_BAD_SCALE",
}
BUFFERS = {"pool_x": 0, "pool_sf": 1, "act": 2, "act_sf": 3, "combine": 4, "table": 5}
OPT_TIMEOUT_NS = 0
OPT_DEBUG_SKIP_BARRIER = 1
OPT_FFN_MODE = 2
OPT_SCALE_MODE = 3
OPT_COMBINE_MODE = 4
COMBINE_KERNEL, COMBINE_IN_FFN, COMBINE_AUTO = 0, 1, 2   # values of OPT_COMBINE_MODE (default COMBINE_AUTO)
SCALE_FP32, SCALE_POW2, SCALE_AUTO = 0, 1, 2   # values of OPT_SCALE_MODE (default SCALE_AUTO)
WEIGHTS_FP8, WEIGHTS_MXFP4 = 0, 1              # values of MoeInfo.weight_format


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class MoeInfo(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("topk", ctypes.c_int), ("R", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("pool_rows", ctypes.c_int), ("block_m", ctypes.c_int), ("block_n", ctypes.c_int),
                ("num_sms", ctypes.c_int), ("workspace_bytes", ctypes.c_uint64),
                ("weight_bytes", ctypes.c_uint64), ("n_shared", ctypes.c_int),
                ("weight_format", ctypes.c_int)]


def header_functions() -> list[str]:
    """Names of the functions declared in include/cpw_moe.h."""
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


_lib = None


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        from . import build as _build
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library {LIB_PATH} is not built (run __graft_entry__.build())")
    L = ctypes.CDLL(LIB_PATH)
    P, I, I64, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
    H = ctypes.c_void_p
    sig = {
        "moe_create": [I, I, I, I, I, ctypes.POINTER(H)],
        "moe_create_shared": [I, I, I, I, I, I, ctypes.POINTER(H)],
        "moe_reserve": [H, I],
        "moe_load_weights": [H, P, P, P, P, P],
        "moe_load_shared_weights": [H, P, P, P, P, P],
        "moe_load_weights_mxfp4": [H, P, P, P, P, P],
        "moe_load_shared_weights_mxfp4": [H, P, P, P, P, P],
        "moe_forward": [H, I, P, P, P, P, P, P],
        "moe_forward_host": [H, I, P, P, P, P, P, P],
        "moe_forward_host_async": [H, I, P, P, P, P, P, P],
        "moe_get_error": [H, ctypes.POINTER(I)],
        "moe_debug_routing": [H, P, P, P, P, ctypes.POINTER(I), ctypes.POINTER(I)],
        "moe_cumulative_expert_rows": [H, P],
        "moe_debug_buffer": [H, I, P, U64],
        "moe_get_info": [H, ctypes.POINTER(MoeInfo)],
        "moe_set_option": [H, I, I64],
        "moe_destroy": [H],
        "moe_profile_enable": [H, I],
        "moe_profile_read": [H, P, ctypes.POINTER(I), ctypes.POINTER(I)],
        "moe_route_noalloc": [I, I, I, I, P, P, P, P, P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.moe_status_string.argtypes = [ctypes.c_int]
    L.moe_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(code: int, what: str):
    if code != MOE_OK:
        raise MoeError(code, what)


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


class FusedMoE:
    """The fused FP8 MoE layer on the current CUDA device (one handle of the C ABI).
    `n_shared` shared experts (moe_create_shared): every token also goes through each, its
    output added with weight 1; their weights come from load_shared_weights.  `E` and
    `topk` are the routed counts; the debug views use the handle's expert slots
    (E + n_shared) and combine planes (topk + n_shared)."""

    def __init__(self, E: int, H: int, I: int, topk: int, R: int, n_shared: int = 0):
        self.lib = load()
        self.E, self.H, self.I, self.topk, self.R = E, H, I, topk, R
        self.n_shared = n_shared
        self.E_slots, self.K_planes = E + n_shared, topk + n_shared
        h = ctypes.c_void_p()
        if n_shared:
            _check(self.lib.moe_create_shared(E, H, I, topk, R, n_shared, ctypes.byref(h)), "moe_create_shared")
        else:
            _check(self.lib.moe_create(E, H, I, topk, R, ctypes.byref(h)), "moe_create")
        self.h = h
        self.max_tokens = 0

    # -------------------------------------------------------------- set-up ------
    def reserve(self, max_tokens: int):
        _check(self.lib.moe_reserve(self.h, max_tokens), "moe_reserve")
        self.max_tokens = max(self.max_tokens, max_tokens)
        return self

    def load_weights(self, w_gate_up, sf_gate_up, w_down, sf_down, stream=None):
        self._load(self.lib.moe_load_weights, self.E, "moe_load_weights",
                   w_gate_up, sf_gate_up, w_down, sf_down, stream)
        return self

    def load_shared_weights(self, w_gate_up, sf_gate_up, w_down, sf_down, stream=None):
        # (a handle without shared experts refuses in the C call, with MOE_ERR_INVALID_ARG)
        self._load(self.lib.moe_load_shared_weights, self.n_shared or w_gate_up.shape[0],
                   "moe_load_shared_weights", w_gate_up, sf_gate_up, w_down, sf_down, stream)
        return self

    def load_weights_mxfp4(self, w_gate_up, sf_gate_up, w_down, sf_down, stream=None):
        """MXFP4 weights: packed E2M1 uint8 [E, 2I, H/2] / [E, H, I/2] (element 2j in the low
        nibble) with UE8M0 uint8 scales [E, 2I, H/32] / [E, H, I/32] (one per 32 elements)."""
        self._load(self.lib.moe_load_weights_mxfp4, self.E, "moe_load_weights_mxfp4",
                   w_gate_up, sf_gate_up, w_down, sf_down, stream, mxfp4=True)
        return self

    def load_shared_weights_mxfp4(self, w_gate_up, sf_gate_up, w_down, sf_down, stream=None):
        self._load(self.lib.moe_load_shared_weights_mxfp4, self.n_shared or w_gate_up.shape[0],
                   "moe_load_shared_weights_mxfp4", w_gate_up, sf_gate_up, w_down, sf_down, stream,
                   mxfp4=True)
        return self

    def _load(self, fn, E, what, w_gate_up, sf_gate_up, w_down, sf_down, stream, mxfp4=False):
        import torch
        H, I = self.H, self.I
        if mxfp4:
            _expect(w_gate_up, (E, 2 * I, H // 2), torch.uint8, "w_gate_up")
            _expect(sf_gate_up, (E, 2 * I, H // 32), torch.uint8, "sf_gate_up")
            _expect(w_down, (E, H, I // 2), torch.uint8, "w_down")
            _expect(sf_down, (E, H, I // 32), torch.uint8, "sf_down")
        else:
            _expect(w_gate_up, (E, 2 * I, H), torch.uint8, "w_gate_up")
            _expect(sf_gate_up, (E, 2 * I // 128, H // 128), torch.float32, "sf_gate_up")
            _expect(w_down, (E, H, I), torch.uint8, "w_down")
            _expect(sf_down, (E, H // 128, I // 128), torch.float32, "sf_down")
        _check(fn(self.h, w_gate_up.data_ptr(), sf_gate_up.data_ptr(), w_down.data_ptr(),
                  sf_down.data_ptr(), _stream_handle(stream)), what)

    def load(self, inp, stream=None):
        """Weights of a workloads.Inputs in its format (FP8 or MXFP4)."""
        if getattr(inp.wl, "weights", "fp8") == "mxfp4":
            return self.load_weights_mxfp4(inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down, stream)
        return self.load_weights(inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down, stream)

    def set_option(self, option: int, value: int):
        _check(self.lib.moe_set_option(self.h, option, value), "moe_set_option")

    # -------------------------------------------------------------- forward -----
    def forward(self, x, x_sf, topk_idx, topk_w, out=None, stream=None):
        import torch
        T = x.shape[0]
        self._check_inputs(x, x_sf, topk_idx, topk_w, T, cuda=True)
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=x.device)
        _expect(out, (T, self.H), torch.bfloat16, "out", cuda=True)
        _check(self.lib.moe_forward(self.h, T, x.data_ptr(), x_sf.data_ptr(), topk_idx.data_ptr(),
                                    topk_w.data_ptr(), out.data_ptr(), _stream_handle(stream)),
               "moe_forward")
        return out

    def forward_host(self, x, x_sf, topk_idx, topk_w, out=None, stream=None, wait=True):
        """Same layer from host (ideally pinned) CPU tensors.  wait=True returns when done;
        wait=False returns once enqueued (moe_forward_host_async): keep the tensors alive and
        unchanged, and read `out`, only after the stream has been synchronized."""
        import torch
        T = x.shape[0]
        self._check_inputs(x, x_sf, topk_idx, topk_w, T, cuda=False)
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, pin_memory=True)
        _expect(out, (T, self.H), torch.bfloat16, "out", cuda=False)
        fn = self.lib.moe_forward_host if wait else self.lib.moe_forward_host_async
        _check(fn(self.h, T, x.data_ptr(), x_sf.data_ptr(), topk_idx.data_ptr(), topk_w.data_ptr(),
                  out.data_ptr(), _stream_handle(stream)),
               "moe_forward_host" if wait else "moe_forward_host_async")
        return out

    def _check_inputs(self, x, x_sf, topk_idx, topk_w, T, cuda):
        import torch
        _expect(x, (T, self.H), torch.uint8, "x", cuda=cuda)
        _expect(x_sf, (T, self.H // 128), torch.float32, "x_sf", cuda=cuda)
        _expect(topk_idx, (T, self.topk), torch.int64, "topk_idx", cuda=cuda)
        _expect(topk_w, (T, self.topk), torch.float32, "topk_w", cuda=cuda)

    # -------------------------------------------------------------- inspection --
    def get_error(self) -> int:
        st = ctypes.c_int(0)
        _check(self.lib.moe_get_error(self.h, ctypes.byref(st)), "moe_get_error")
        return st.value

    def info(self) -> MoeInfo:
        inf = MoeInfo()
        _check(self.lib.moe_get_info(self.h, ctypes.byref(inf)), "moe_get_info")
        return inf

    def debug_routing(self, T: int) -> dict:
        import numpy as np
        E, R = self.E_slots, self.R
        inf = self.info()
        counts = np.zeros(E, np.uint32)
        recv = np.zeros((E, R), np.uint32)
        off = np.zeros(E + 1, np.int32)
        rows_cap = (-(-T * self.K_planes // inf.block_m) + E) * inf.block_m
        meta = np.zeros((max(rows_cap, 1), 3), np.uint32)
        P = ctypes.c_int(0)
        bm = ctypes.c_int(0)
        _check(self.lib.moe_debug_routing(self.h, counts.ctypes.data, recv.ctypes.data,
                                          off.ctypes.data, meta.ctypes.data, ctypes.byref(P),
                                          ctypes.byref(bm)), "moe_debug_routing")
        return {"counts": counts, "recv": recv, "block_offset": off, "meta": meta[:P.value],
                "P": P.value, "block_m": bm.value}

    def cumulative_expert_rows(self):
        import numpy as np
        rows = np.zeros(self.E_slots, np.uint64)
        _check(self.lib.moe_cumulative_expert_rows(self.h, rows.ctypes.data), "moe_cumulative_expert_rows")
        return rows

    def debug_buffer(self, which: str):
        import numpy as np
        inf = self.info()
        P, H, I, K = inf.pool_rows, self.H, self.I, self.K_planes
        shapes = {
            "pool_x": ((P, H), np.uint8), "pool_sf": ((H // 128, P), np.float32),
            "act": ((P, I), np.uint8), "act_sf": ((I // 128, P), np.float32),
            "combine": ((K, inf.max_tokens, H), np.uint16),
            "table": ((self.E_slots, self.R, max(1, inf.max_tokens // self.R)), np.int32),
        }
        shape, dt = shapes[which]
        a = np.zeros(shape, dt)
        _check(self.lib.moe_debug_buffer(self.h, BUFFERS[which], a.ctypes.data, a.nbytes),
               "moe_debug_buffer")
        return a

    STAGES = ("dispatch", "expert_ffn", "combine")

    def profile_enable(self, on=True, every: int = 1):
        """Record stage events on every `every`-th forward (on=False stops)."""
        _check(self.lib.moe_profile_enable(self.h, max(1, int(every)) if on else 0), "moe_profile_enable")

    def profile_read(self) -> dict:
        import numpy as np
        ms = np.zeros(len(self.STAGES), np.float64)
        calls = ctypes.c_int(0)
        dropped = ctypes.c_int(0)
        _check(self.lib.moe_profile_read(self.h, ms.ctypes.data, ctypes.byref(calls),
                                         ctypes.byref(dropped)), "moe_profile_read")
        return {"stage_ms": dict(zip(self.STAGES, ms.tolist())), "calls": calls.value,
                "dropped": dropped.value}

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            self.lib.moe_destroy(self.h)
            self.h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def route_noalloc(topk_idx, E: int, R: int, stream=None) -> dict:
    """Routing of one batch through moe_route_noalloc (no device allocation inside the
    library; the output tensors here are allocated by PyTorch, as a caller would).
    Returns device tensors counts [E], recv [E,R], block_offset [E+1], meta [rows,3] and
    status [1]."""
    import torch
    T, K = topk_idx.shape
    _expect(topk_idx, (T, K), torch.int64, "topk_idx", cuda=True)
    dev = topk_idx.device
    rows = (-(-T * K // 128) + E) * 128
    out = {
        "counts": torch.zeros(E, dtype=torch.int32, device=dev),
        "recv": torch.zeros(E, R, dtype=torch.int32, device=dev),
        "block_offset": torch.zeros(E + 1, dtype=torch.int32, device=dev),
        "meta": torch.full((rows, 3), -1, dtype=torch.int32, device=dev),
        "status": torch.zeros(1, dtype=torch.int32, device=dev),
    }
    _check(load().moe_route_noalloc(T, E, K, R, topk_idx.data_ptr(), out["counts"].data_ptr(),
                                    out["recv"].data_ptr(), out["block_offset"].data_ptr(),
                                    out["meta"].data_ptr(), out["status"].data_ptr(),
                                    _stream_handle(stream)), "moe_route_noalloc")
    return out


def _expect(t, shape, dtype, name, cuda=None):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype} != {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if cuda is not None and t.is_cuda != cuda:
        raise ValueError(f"{name} must be a {'CUDA' if cuda else 'host'} tensor")
