"""The boundary's largest shapes against the oracle, every token.

moe_create accepts H and I up to 16384 (128 K blocks of 128: the FFN kernels' per-tile scale
arrays and the routing kernel's 16 KB row copies are at their sizes), R up to 64 sources and
(E + shared) * R up to 16384 index-table rows (the routing kernel's shared-memory histogram at
its largest, leaving the least room for the gather's row buffers).  Each case runs one small
batch at that limit with fp32 block scales and with power-of-two scales (the block-scaled
kernel), and the hidden-size limit also with MXFP4 weights; integers and the per-token
relative L2 bound as in the other parity tests, and the combine inside the FFN kernel bit for
bit against the combine kernel.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_persistent_warp_gb300 import FusedMoE
from combine_persistent_warp_gb300 import native
from combine_persistent_warp_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2

CASES = {
    # H at its limit: 128 K blocks per gate_up tile, 16 KB rows gathered
    "h16384": dict(T=32, H=16384, I=256, E=3, topk=2, R=2),
    # I at its limit: 128 gate_up N-tiles per M-block, 128 K blocks per down tile
    "i16384": dict(T=32, H=256, I=16384, E=3, topk=2, R=2),
    # (E * R) at its limit: the routing kernel's largest index table and histogram
    "er16384": dict(T=256, H=256, I=128, E=1024, topk=4, R=16),
    # R at its limit: 64 sources of 2 tokens each
    "r64": dict(T=128, H=256, I=128, E=8, topk=2, R=64),
}
RUNS = [(c, s, "fp8") for c in CASES for s in ("fp32", "pow2")] + [("h16384", "pow2", "mxfp4")]


@pytest.mark.parametrize("case,scales,weights", RUNS, ids=[f"{c}-{s}-{w}" for c, s, w in RUNS])
def test_shape_limits_match_the_oracle(case, scales, weights):
    torch.cuda.set_device(0)
    wl = Workload(f"limit-{case}", **CASES[case], seed=90, scales=scales, weights=weights)
    inp = make_inputs(wl, device="cuda")
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R).reserve(wl.T)
    moe.load(inp)
    if scales == "pow2":
        moe.set_option(native.OPT_SCALE_MODE, 1)
    out = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    counts, recv, bad = oracle.route_counts(inp.topk_idx, wl.E, wl.R)
    assert not bad
    dbg = moe.debug_routing(wl.T)
    assert np.array_equal(dbg["counts"], counts) and np.array_equal(dbg["recv"], recv)
    h = oracle.HostInputs.from_inputs(inp)
    oracle.set_scale_rule(scales)
    try:
        _, ref, bad = oracle.forward_tokens(h, np.arange(wl.T))
    finally:
        oracle.set_scale_rule("fp32")
    assert not bad
    g = out.float().cpu().numpy()
    den = np.linalg.norm(ref, axis=1)
    num = np.linalg.norm(g - ref, axis=1)
    rel = np.where(den > 0, num / np.maximum(den, 1e-30), num)
    assert np.all(rel <= TOL), rel.max()
    # the combine inside the FFN kernel gives the same bits at these sizes
    moe.set_option(native.OPT_COMBINE_MODE, native.COMBINE_IN_FFN)
    out2 = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    moe.close()
