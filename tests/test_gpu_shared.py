"""Shared experts (moe_create_shared): every token also goes through each shared expert,
whose output is added to its top-k sum with weight 1 ("DeepGEMM Mega MoE 对称内存（Symmetric
Memory）深度分析" §8.2: one more combine plane after the top-k ones).

The oracle sees the same layer as E + S experts with every token's route extended by slots
topk + s naming expert E + s with weight 1 (the plain definition of that sum), so it needs no
shared-expert code of its own.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_persistent_warp_gb300 import FusedMoE, MoeError
from combine_persistent_warp_gb300 import native
from combine_persistent_warp_gb300.workloads import Workload, make_inputs, make_weights

pytestmark = pytest.mark.gpu

TOL = 2e-2


def shared_case(wl: Workload, S: int):
    torch.cuda.set_device(0)
    inp = make_inputs(wl, device="cuda")
    sw = make_weights(S, wl.H, wl.I, seed=wl.seed + 1000, device="cuda", scales=wl.scales)
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R, n_shared=S).reserve(wl.T)
    moe.load_weights(inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down)
    moe.load_shared_weights(*sw)
    return moe, inp, sw


def extended(inp, sw, S):
    """The same layer as E + S routed experts: route slots topk + s -> expert E + s, weight 1."""
    T, E = inp.topk_idx.shape[0], inp.w_gate_up.shape[0]
    ext_idx = torch.cat([inp.topk_idx, (E + torch.arange(S, device=inp.topk_idx.device)).expand(T, S)], 1)
    ext_w = torch.cat([inp.topk_w, torch.ones(T, S, device=inp.topk_w.device)], 1)
    w = [torch.cat([a, b]) for a, b in zip((inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down), sw)]
    return ext_idx.contiguous(), ext_w.contiguous(), w


def rel_l2(got, ref):
    g = got.float().cpu().numpy()
    den = np.linalg.norm(ref, axis=1)
    return np.where(den > 0, np.linalg.norm(g - ref, axis=1) / np.maximum(den, 1e-30), np.linalg.norm(g - ref, axis=1))


@pytest.mark.parametrize("scales,S", [("fp32", 1), ("pow2", 1), ("fp32", 2)])
def test_shared_experts_match_oracle(scales, S):
    wl = Workload("shared-tiny", T=256, H=256, I=256, E=8, topk=2, R=2, seed=41, scales=scales)
    moe, inp, sw = shared_case(wl, S)
    out = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    ext_idx, ext_w, w = extended(inp, sw, S)
    h = oracle.HostInputs(inp.x, inp.x_sf, ext_idx, ext_w, *w)
    oracle.set_scale_rule(scales)
    try:
        _, ref, bad = oracle.forward_tokens(h, np.arange(wl.T))
    finally:
        oracle.set_scale_rule("fp32")
    assert not bad
    rel = rel_l2(out, ref)
    assert np.all(rel <= TOL), rel.max()
    # the shared experts saw every token: T rows each, per source T/R
    dbg = moe.debug_routing(wl.T)
    assert np.all(dbg["counts"][wl.E:] == wl.T)
    assert np.all(dbg["recv"][wl.E:] == wl.T // wl.R)


def test_shared_experts_equal_an_explicit_extra_expert():
    """Bit-identical to a plain layer of E + S experts whose routes carry the shared slots."""
    S = 1
    wl = Workload("shared-eq", T=512, H=512, I=256, E=16, topk=4, R=4, seed=43,
                  routing="zipf", zipf_s=1.2, skip_frac=0.05)
    moe, inp, sw = shared_case(wl, S)
    out = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w).clone()
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    ext_idx, ext_w, w = extended(inp, sw, S)
    plain = FusedMoE(wl.E + S, wl.H, wl.I, wl.topk + S, wl.R).reserve(wl.T)
    plain.load_weights(*w)
    ref = plain.forward(inp.x, inp.x_sf, ext_idx, ext_w)
    torch.cuda.synchronize()
    assert plain.get_error() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_shared_experts_full_width_sampled():
    """Hidden 7168 / intermediate 2048, 32 routed experts top-8 and one shared expert, on
    1024 tokens (the shared expert's 1024 rows span 8 M-blocks): sampled tokens against
    the oracle, fp32 and power-of-two scales."""
    for scales in ("fp32", "pow2"):
        wl = Workload("shared-wide", T=1024, H=7168, I=2048, E=32, topk=8, R=8, seed=45, scales=scales)
        moe, inp, sw = shared_case(wl, 1)
        out = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
        torch.cuda.synchronize()
        assert moe.get_error() == 0
        ext_idx, ext_w, w = extended(inp, sw, 1)
        h = oracle.HostInputs(inp.x, inp.x_sf, ext_idx, ext_w, *w)
        toks = np.array([0, 1, 255, 512, 777, 1023])
        oracle.set_scale_rule(scales)
        try:
            _, ref, _ = oracle.forward_tokens(h, toks)
        finally:
            oracle.set_scale_rule("fp32")
        rel = rel_l2(out[torch.as_tensor(toks, device=out.device)], ref)
        assert np.all(rel <= TOL), (scales, rel.max())
        moe.close()


def test_shared_weights_required_and_only_with_shared_experts():
    wl = Workload("shared-err", T=64, H=256, I=128, E=8, topk=2, R=2, seed=47)
    inp = make_inputs(wl, device="cuda")
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R, n_shared=1).reserve(wl.T)
    moe.load_weights(inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down)
    with pytest.raises(MoeError) as ei:
        moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    assert ei.value.code == 4
    assert moe.info().n_shared == 1 and moe.info().E == wl.E + 1 and moe.info().topk == wl.topk + 1
    plain = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R).reserve(wl.T)
    sw = make_weights(1, wl.H, wl.I, seed=1, device="cuda")
    with pytest.raises(MoeError) as ei:
        plain.load_shared_weights(*sw)
    assert ei.value.code == 1
    assert native.STATUS[4] == "MOE_ERR_NO_WEIGHTS"
