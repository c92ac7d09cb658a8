"""Degenerate routing shapes against the oracle, every token.

One source partition (R = 1: the index table has one source row per expert and the
round-robin order is that source's slot order), one expert with top-1 (every token's only
slot goes to expert 0: one expert segment holding every row, several M-blocks), and every
expert on every token (topk = E: each token appears once in every expert's segment).  Each
runs with fp32 block scales, power-of-two scales (the block-scaled kernel) and MXFP4
weights; integers bit-exact, the per-token relative L2 bound of the other parity tests, and
the combine inside the FFN kernel bit for bit against the combine kernel.
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
    # one source partition of 96 tokens
    "one-source": dict(T=96, H=384, I=256, E=8, topk=2, R=1),
    # one expert, top-1: 300 rows in one segment (three M-blocks, the last one partly filled)
    "one-expert": dict(T=300, H=256, I=128, E=1, topk=1, R=3),
    # every expert on every token
    "topk-equals-e": dict(T=64, H=256, I=256, E=4, topk=4, R=2),
}
RUNS = [(c, s, w) for c in CASES for s, w in (("fp32", "fp8"), ("pow2", "fp8"), ("pow2", "mxfp4"))]


@pytest.mark.parametrize("case,scales,weights", RUNS, ids=[f"{c}-{s}-{w}" for c, s, w in RUNS])
def test_degenerate_routing_matches_the_oracle(case, scales, weights):
    torch.cuda.set_device(0)
    wl = Workload(f"degenerate-{case}", **CASES[case], seed=91, scales=scales, weights=weights)
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
    # the combine inside the FFN kernel gives the same bits
    moe.set_option(native.OPT_COMBINE_MODE, native.COMBINE_IN_FFN)
    out2 = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    moe.close()
