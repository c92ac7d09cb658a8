"""The allocation-free routing entry point, checked against the regular forward path and
against the CPU oracle's routing.

moe_route_noalloc exists for callers that may not allocate device memory -- code that
runs under another framework's memory pool or a fixed memory budget, or a loop that must
stay out of the allocator.  Its scratch lives in one fixed array inside the library that
every call shares.  Its results must equal what the allocating path (moe_forward, then
moe_debug_routing) reports, on two calls in a row: the second call starts from the
first call's leftovers in that shared array.  Integers are compared exactly; the slot
order inside one (expert, source) pair comes from atomics, so those rows are compared
as sorted multisets, as in the other routing tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_persistent_warp_gb300 import FusedMoE, native
from combine_persistent_warp_gb300.workloads import make_inputs


def _forward_routing(inp):
    wl = inp.wl
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R).reserve(wl.T)
    moe.load_weights(inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down)
    moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    dbg = moe.debug_routing(wl.T)
    moe.close()
    return dbg


def _check_same(ref, got, wl):
    torch.cuda.synchronize()
    assert int(got["status"].item()) == 0
    counts = got["counts"].cpu().numpy().astype(np.uint32)
    recv = got["recv"].cpu().numpy().astype(np.uint32)
    off = got["block_offset"].cpu().numpy()
    meta = got["meta"].cpu().numpy().astype(np.int64)
    assert np.array_equal(counts, ref["counts"])
    assert np.array_equal(recv, ref["recv"])
    assert np.array_equal(off, ref["block_offset"])
    BM = ref["block_m"]
    ref_meta = ref["meta"].astype(np.int64)
    Tsrc = wl.T // wl.R
    for e in range(wl.E):
        rows = off[e] * BM + np.arange(int(counts[e]))
        a, b = meta[rows], ref_meta[rows]
        assert np.array_equal(a[:, 0], b[:, 0])                  # round-robin sources
        assert np.all(a[:, 1] // Tsrc == a[:, 0])
        for r in range(wl.R):
            sa = sorted(map(tuple, a[a[:, 0] == r][:, 1:].tolist()))
            sb = sorted(map(tuple, b[b[:, 0] == r][:, 1:].tolist()))
            assert sa == sb


def _check_oracle(got, idx, wl):
    """The same outputs against the CPU oracle's routing: counts and per-source counts by
    direct counting, block offsets by ceil_div prefix, the round-robin source order of every
    expert, and the (token, slot) multiset of every (expert, source)."""
    torch.cuda.synchronize()
    assert int(got["status"].item()) == 0
    counts, recv, bad = oracle.route_counts(idx, wl.E, wl.R)
    assert not bad
    assert np.array_equal(got["counts"].cpu().numpy().astype(np.uint32), counts)
    assert np.array_equal(got["recv"].cpu().numpy().astype(np.uint32), recv)
    off = oracle.block_offsets(counts, 128)
    assert np.array_equal(got["block_offset"].cpu().numpy(), off)
    meta = got["meta"].cpu().numpy().astype(np.int64)
    groups = oracle.route_multiset(idx, wl.E, wl.R)
    for e in range(wl.E):
        rows = off[e] * 128 + np.arange(int(counts[e]))
        src, _ = oracle.round_robin(recv[e])
        assert np.array_equal(meta[rows, 0], src)
        for r in range(wl.R):
            m = meta[rows][meta[rows, 0] == r]
            assert sorted(map(tuple, m[:, 1:].tolist())) == groups[(e, r)]


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "decode", "skewed"])
def test_noalloc_routing_matches_forward_twice(name):
    torch.cuda.set_device(0)
    inp = make_inputs(name, device="cuda")
    ref = _forward_routing(inp)
    for _ in range(2):
        got = native.route_noalloc(inp.topk_idx, inp.wl.E, inp.wl.R)
        _check_same(ref, got, inp.wl)
        _check_oracle(got, inp.topk_idx, inp.wl)


@pytest.mark.gpu
def test_noalloc_reports_bad_index_on_device():
    torch.cuda.set_device(0)
    idx = make_inputs("tiny", device="cuda").topk_idx.clone()
    idx[3, 1] = 8                                   # == E
    got = native.route_noalloc(idx, 8, 2)
    torch.cuda.synchronize()
    assert int(got["status"].item()) == 6          # MOE_ERR_BAD_INDEX


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = native.load()
    p = ctypes.c_void_p(16)    # never dereferenced: the size check comes first
    # E*T above the 1,048,576-entry index table
    assert lib.moe_route_noalloc(16384, 128, 8, 8, p, p, p, p, p, p, None) == 3
    # T*topk above 131,072 routed entries
    assert lib.moe_route_noalloc(32768, 16, 8, 8, p, p, p, p, p, p, None) == 3
    # E*R above 4,096 counters
    assert lib.moe_route_noalloc(128, 128, 8, 64, p, p, p, p, p, p, None) == 3
    # T not a multiple of R
    assert lib.moe_route_noalloc(127, 32, 8, 8, p, p, p, p, p, p, None) == 1
