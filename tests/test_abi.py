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
    assert lib.moe_create(8, 384, 128, 2, 2, ctypes.byref(h)) == 1      # H % 256
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
