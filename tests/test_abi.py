"""The C-ABI library builds, loads and exports every function its header declares.

CPU only: no call here reaches the GPU (argument checks return before any CUDA call).
"""
import ctypes

from combine_persistent_warp_gb300 import native

EXPECTED = {
    "moe_create", "moe_reserve", "moe_load_weights", "moe_forward", "moe_forward_host",
    "moe_get_error", "moe_debug_routing", "moe_cumulative_expert_rows", "moe_debug_buffer",
    "moe_get_info", "moe_set_option", "moe_destroy", "moe_status_string",
    "moe_profile_enable", "moe_profile_read",
}


def test_header_declares_the_boundary():
    assert EXPECTED <= set(native.header_functions())


def test_library_exports_every_declared_symbol():
    lib = native.load()
    for name in native.header_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    lib = native.load()
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(7) == b"device wait timed out"
    assert lib.moe_status_string(99) == b"unknown status"


def test_host_side_argument_checks_need_no_gpu():
    lib = native.load()
    h = ctypes.c_void_p()
    assert lib.moe_create(8, 256, 128, 2, 2, None) == 1
    assert lib.moe_create(0, 256, 128, 2, 2, ctypes.byref(h)) == 1      # E
    assert lib.moe_create(8, 320, 128, 2, 2, ctypes.byref(h)) == 1      # H % 128
    assert lib.moe_create(8, 0, 128, 2, 2, ctypes.byref(h)) == 1        # H
    # H an odd multiple of 128 passes the shape checks (without a GPU it then fails later)
    rc = lib.moe_create(8, 384, 128, 2, 2, ctypes.byref(h))
    assert rc != 1
    if rc == 0:
        lib.moe_destroy(h)
    assert lib.moe_create(8, 256, 96, 2, 2, ctypes.byref(h)) == 1       # I % 128
    assert lib.moe_create(8, 256, 128, 9, 2, ctypes.byref(h)) == 1      # topk > E
    assert lib.moe_create(8, 256, 128, 33, 2, ctypes.byref(h)) == 1     # topk > 32
    assert lib.moe_create(8, 256, 128, 2, 65, ctypes.byref(h)) == 1     # R > 64
    assert lib.moe_create(1024, 256, 128, 2, 64, ctypes.byref(h)) == 1  # E*R > 16384
    assert lib.moe_reserve(None, 16) == 1
    assert lib.moe_forward(None, 0, None, None, None, None, None, None) == 1
    assert lib.moe_set_option(None, 0, 10 ** 9) == 1
    st = ctypes.c_int()
    assert lib.moe_get_error(None, ctypes.byref(st)) == 1
    assert lib.moe_destroy(None) == 1


def _header_enum_values():
    """NAME = value pairs of the header's enums (comments stripped)."""
    import re
    text = open(native.HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(MOE_[A-Z0-9_]+)\s*=\s*(\d+)", text)}


def test_binding_constants_match_the_header():
    v = _header_enum_values()
    for code, name in native.STATUS.items():
        assert v[name] == code, name
    assert v["MOE_OPT_TIMEOUT_NS"] == native.OPT_TIMEOUT_NS
    assert v["MOE_OPT_DEBUG_SKIP_BARRIER"] == native.OPT_DEBUG_SKIP_BARRIER
    assert v["MOE_OPT_FFN_MODE"] == native.OPT_FFN_MODE
    assert v["MOE_OPT_SCALE_MODE"] == native.OPT_SCALE_MODE
    assert v["MOE_OPT_COMBINE_MODE"] == native.OPT_COMBINE_MODE
    assert v["MOE_WEIGHTS_FP8"] == native.WEIGHTS_FP8 and v["MOE_WEIGHTS_MXFP4"] == native.WEIGHTS_MXFP4
    for name, idx in native.BUFFERS.items():
        assert v["MOE_BUF_" + name.upper()] == idx


def test_mxfp4_loaders_refuse_null_handles_without_a_gpu():
    lib = native.load()
    assert lib.moe_load_weights_mxfp4(None, None, None, None, None, None) == 1
    assert lib.moe_load_shared_weights_mxfp4(None, None, None, None, None, None) == 1
