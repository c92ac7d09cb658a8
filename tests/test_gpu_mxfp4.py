"""GPU parity of the MXFP4-weight path (FP8 activations x E2M1 weights with one UE8M0 scale
per 32 elements, on the block-scaled UMMA with a 4-bit B operand) against the CPU oracle's
MXFP4 weight format with the power-of-two requant rule, through the C ABI.

The pages name an FP8 x FP4 variant of the SM100 kernel ("DeepGEMM Mega MoE 对称内存
（Symmetric Memory）深度分析" §11) without its format; the OCP MXFP4 block is the reading
taken.  Bar: per-token relative L2 <= 2e-2, as for the FP8 paths.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import block_cover_tokens, blocks_of_tokens, fp8_twin_of_mxfp4
from combine_persistent_warp_gb300 import FusedMoE, MoeError
from combine_persistent_warp_gb300 import native
from combine_persistent_warp_gb300.workloads import Workload, make_inputs, make_weights, make_weights_mxfp4

pytestmark = pytest.mark.gpu

TOL = 2e-2


def mx_layer(wl, T_max=None):
    torch.cuda.set_device(0)
    inp = make_inputs(wl, device="cuda")
    wl = inp.wl
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R).reserve(T_max or wl.T)
    moe.load_weights_mxfp4(inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down)
    return moe, inp


def rel_l2(got, ref):
    g = got.float().cpu().numpy()
    den = np.linalg.norm(ref, axis=1)
    diff = np.linalg.norm(g - ref, axis=1)
    return np.where(den > 0, diff / np.maximum(den, 1e-30), diff)


def oracle_out(inp, toks, idx=None, w=None, x=None, xs=None):
    h = oracle.HostInputs(inp.x if x is None else x, inp.x_sf if xs is None else xs,
                          inp.topk_idx if idx is None else idx, inp.topk_w if w is None else w,
                          inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down, weights="mxfp4")
    oracle.set_scale_rule("pow2")
    try:
        _, ref, bad = oracle.forward_tokens(h, toks)
    finally:
        oracle.set_scale_rule("fp32")
    assert not bad
    return ref


def sample(T, n):
    if n is None or n >= T:
        return np.arange(T)
    rng = np.random.default_rng(2468)
    return np.array(sorted(set(rng.choice(T, n - 2, replace=False).tolist()) | {0, T - 1}))


CASES = {
    # name: (workload, sampled tokens or None = all)
    "tiny": (Workload("mx-tiny", T=64, H=256, I=128, E=8, topk=2, R=2, seed=61, scales="pow2",
                      weights="mxfp4"), None),
    # 3 N-tiles of gate_up, K blocks 4 (H) and 3 (I), Zipf routing with skipped slots
    "ragged": (Workload("mx-ragged", T=520, H=512, I=384, E=6, topk=3, R=4, routing="zipf", zipf_s=1.1,
                        skip_frac=0.05, seed=62, scales="pow2", weights="mxfp4"), None),
    # 10 and 5 K blocks: A scale groups end mid-way through tiles
    "groups": (Workload("mx-groups", T=256, H=1280, I=640, E=4, topk=2, R=2, seed=63, scales="pow2",
                        weights="mxfp4"), None),
    # H = 5 x 128: the last down tile's second column half lies past H (zero weight rows)
    "odd-h": (Workload("mx-odd-h", T=256, H=640, I=256, E=4, topk=2, R=2, seed=65, scales="pow2",
                       weights="mxfp4"), None),
    # the decode and prefill shapes (hidden 7168, intermediate 2048, 32 experts, top-8)
    "decode": (Workload("mx-decode", T=128, H=7168, I=2048, E=32, topk=8, R=8, seed=1, scales="pow2",
                        weights="mxfp4"), None),
    "prefill": (Workload("mx-prefill", T=4096, H=7168, I=2048, E=32, topk=8, R=8, seed=2, scales="pow2",
                         weights="mxfp4"), 10),
    # the skewed (Zipf, 5% skipped slots, 64 experts) and large (128 experts) batches
    "skewed": ("skewed-mxfp4", 10),
    "large": ("large-mxfp4", 10),
}


@pytest.mark.parametrize("case", list(CASES))
def test_mxfp4_matches_oracle(case):
    wl, n = CASES[case]
    moe, inp = mx_layer(wl)
    wl = inp.wl
    out = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    assert moe.info().weight_format == native.WEIGHTS_MXFP4
    # a seeded sample plus a cover of the pool: every M-block of every expert holds a row of
    # a compared token
    dbg = moe.debug_routing(wl.T)
    toks = block_cover_tokens(dbg, extra=sample(wl.T, n).tolist())
    assert blocks_of_tokens(dbg, toks) == set(range(int(dbg["block_offset"][-1])))
    ref = oracle_out(inp, toks)
    rel = rel_l2(out[torch.as_tensor(toks, device=out.device)], ref)
    assert np.all(rel <= TOL), f"max per-token rel L2 {rel.max():.3e}"
    # routing is format-independent: bit-exact counts
    counts, recv, _ = oracle.route_counts(inp.topk_idx, wl.E, wl.R)
    dbg = moe.debug_routing(wl.T)
    assert np.array_equal(dbg["counts"], counts) and np.array_equal(dbg["recv"], recv)


def test_mxfp4_zipf_multi_block_experts():
    """Zipf routing leaves experts with several M-blocks (odd counts among them) and partly
    filled last blocks; a seeded sample plus a cover of every M-block against the oracle."""
    wl = Workload("mx-zipf", T=2048, H=1024, I=512, E=8, topk=4, R=4, routing="zipf", zipf_s=1.2,
                  seed=64, scales="pow2", weights="mxfp4")
    moe, inp = mx_layer(wl)
    out = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    dbg = moe.debug_routing(wl.T)
    toks = block_cover_tokens(dbg, extra=sample(wl.T, 12).tolist())
    rel = rel_l2(out[torch.as_tensor(toks, device="cuda")], oracle_out(inp, toks))
    assert np.all(rel <= TOL), rel.max()


def test_mxfp4_equals_its_fp8_twin_on_the_gpu():
    """The layer with MXFP4 weights and the layer with the FP8 twin weights (the same element
    values as e4m3 codes with 128x128 power-of-two scales) run on the same block-scaled kernel
    with B formats E2M1 and e4m3: the products are the same exact values, so the outputs
    agree to accumulation order (here: identical or within 1e-3)."""
    wl = Workload("mx-twin", T=256, H=512, I=256, E=4, topk=2, R=2, seed=65, scales="pow2", weights="mxfp4")
    moe4, inp = mx_layer(wl)
    out4 = moe4.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w).clone()
    tw = [[fp8_twin_of_mxfp4(w[e].cpu(), s[e].cpu()) for e in range(wl.E)]
          for w, s in ((inp.w_gate_up, inp.sf_gate_up), (inp.w_down, inp.sf_down))]
    w1 = torch.stack([a for a, _ in tw[0]]).cuda()
    s1 = torch.stack([b for _, b in tw[0]]).cuda()
    w2 = torch.stack([a for a, _ in tw[1]]).cuda()
    s2 = torch.stack([b for _, b in tw[1]]).cuda()
    moe8 = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R).reserve(wl.T)
    moe8.load_weights(w1, s1, w2, s2)
    moe8.set_option(native.OPT_SCALE_MODE, 1)
    out8 = moe8.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe4.get_error() == 0 and moe8.get_error() == 0
    rel = rel_l2(out4, out8.float().cpu().numpy())
    assert np.all(rel <= 1e-3), rel.max()


def test_mxfp4_shared_expert():
    """One shared expert with MXFP4 weights: the same layer as E + 1 routed MXFP4 experts with
    every route extended by the shared slot (weight 1), against the oracle."""
    wl = Workload("mx-shared", T=256, H=256, I=256, E=8, topk=2, R=2, seed=66, scales="pow2", weights="mxfp4")
    torch.cuda.set_device(0)
    inp = make_inputs(wl, device="cuda")
    sw = make_weights_mxfp4(1, wl.H, wl.I, seed=wl.seed + 1000, device="cuda")
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R, n_shared=1).reserve(wl.T)
    moe.load_weights_mxfp4(inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down)
    # routed MXFP4 with shared FP8 weights is not a loadable state
    moe.load_shared_weights(*make_weights(1, wl.H, wl.I, seed=5, device="cuda", scales="pow2"))
    with pytest.raises(MoeError) as ei:
        moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    assert ei.value.code == 4
    moe.load_shared_weights_mxfp4(*sw)
    out = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    ext_idx = torch.cat([inp.topk_idx, torch.full((wl.T, 1), wl.E, dtype=torch.int64, device="cuda")], 1)
    ext_w = torch.cat([inp.topk_w, torch.ones(wl.T, 1, device="cuda")], 1)
    h = oracle.HostInputs(inp.x, inp.x_sf, ext_idx.contiguous(), ext_w.contiguous(),
                          *[torch.cat([a, b]) for a, b in zip((inp.w_gate_up, inp.sf_gate_up, inp.w_down,
                                                              inp.sf_down), sw)], weights="mxfp4")
    oracle.set_scale_rule("pow2")
    try:
        _, ref, _ = oracle.forward_tokens(h, np.arange(wl.T))
    finally:
        oracle.set_scale_rule("fp32")
    rel = rel_l2(out, ref)
    assert np.all(rel <= TOL), rel.max()


def test_mxfp4_ragged_hot_expert_empty_and_all_skipped():
    wl = Workload("mx-edge", T=160, H=256, I=256, E=8, topk=2, R=2, seed=67, scales="pow2", weights="mxfp4")
    moe, inp = mx_layer(wl)
    # 158 tokens, expert 3 in every token's slot 0: two M-blocks, the second partly filled
    T = 158
    idx = inp.topk_idx[:T].clone()
    idx[:, 0] = 3
    idx[:, 1] = torch.where(idx[:, 1] == 3, torch.full_like(idx[:, 1], -1), idx[:, 1])
    idx, w = idx.contiguous(), inp.topk_w[:T].contiguous()
    x, xs = inp.x[:T].contiguous(), inp.x_sf[:T].contiguous()
    out = moe.forward(x, xs, idx, w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    rel = rel_l2(out, oracle_out(inp, np.arange(T), idx=idx, w=w, x=x, xs=xs))
    assert np.all(rel <= TOL), rel.max()
    e = torch.empty(0, wl.H, dtype=torch.uint8, device="cuda")
    out = moe.forward(e, torch.empty(0, wl.H // 128, device="cuda"),
                      torch.empty(0, 2, dtype=torch.int64, device="cuda"), torch.empty(0, 2, device="cuda"))
    assert out.shape == (0, wl.H) and moe.get_error() == 0
    skip = torch.full((wl.T, 2), -1, dtype=torch.int64, device="cuda")
    out = moe.forward(inp.x, inp.x_sf, skip, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    assert not torch.any(out.float() != 0)


def test_mxfp4_errors():
    wl = Workload("mx-err", T=64, H=256, I=128, E=8, topk=2, R=2, seed=68, scales="pow2", weights="mxfp4")
    moe, inp = mx_layer(wl)
    # the fp32-scale kernel takes FP8 weights only
    moe.set_option(native.OPT_SCALE_MODE, native.SCALE_FP32)
    with pytest.raises(MoeError) as ei:
        moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    assert ei.value.code == 10
    moe.set_option(native.OPT_SCALE_MODE, native.SCALE_AUTO)
    # activation scales that are not powers of two: reported by the device, then the handle
    # recovers
    xs_bad = inp.x_sf * 1.5
    moe.forward(inp.x, xs_bad, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 10
    out = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0 and torch.isfinite(out.float()).all()
    # a NaN scale byte is refused at load, and the weights count as not loaded
    bad = inp.sf_down.clone()
    bad[1, 7, 2] = 0xFF
    with pytest.raises(MoeError) as ei:
        moe.load_weights_mxfp4(inp.w_gate_up, inp.sf_gate_up, inp.w_down, bad)
    assert ei.value.code == 10
    with pytest.raises(MoeError) as ei:
        moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    assert ei.value.code == 4
    # shape checks of the binding
    with pytest.raises(ValueError):
        moe.load_weights_mxfp4(inp.w_gate_up[:, :, :-16].contiguous(), inp.sf_gate_up, inp.w_down, inp.sf_down)


def test_mxfp4_host_buffers_match_device_forward():
    """The host-buffer entry points (pinned inputs, synchronous and asynchronous) give the same
    bits as the device-pointer forward with MXFP4 weights."""
    wl = Workload("mx-host", T=256, H=512, I=256, E=8, topk=4, R=4, seed=69, scales="pow2", weights="mxfp4")
    moe, inp = mx_layer(wl)
    dev = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w).clone()
    torch.cuda.synchronize()
    pin = lambda t: t.cpu().pin_memory()
    px, psf, pidx, pw = pin(inp.x), pin(inp.x_sf), pin(inp.topk_idx), pin(inp.topk_w)
    host = moe.forward_host(px, psf, pidx, pw)
    o_async = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
    moe.forward_host(px, psf, pidx, pw, out=o_async, wait=False)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    assert torch.equal(host.view(torch.int16), dev.cpu().view(torch.int16))
    assert torch.equal(o_async.view(torch.int16), dev.cpu().view(torch.int16))


@pytest.mark.parametrize("hot", [64, 65])
@pytest.mark.parametrize("weights", ["mxfp4", "fp8"])
def test_block_scaled_stage_layout_at_the_64_row_boundary(hot, weights):
    """The block-scaled kernel stages 8 KB of A rows per K block (one more stage in flight)
    when no M-block of the forward holds more than 64 rows, else 16 KB: expert 0 receives
    exactly 64 rows (compact layout; the UMMA's padding rows 64-127 then read the stage's weight
    tile) or 65 (standard layout); every token against the oracle, both weight formats."""
    T = 256
    wl = Workload(f"mx-edge-{weights}", T=T, H=512, I=256, E=6, topk=1, R=2, seed=66, scales="pow2",
                  weights=weights)
    torch.cuda.set_device(0)
    inp = make_inputs(wl, device="cuda")
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R).reserve(T)
    moe.load(inp)
    moe.set_option(native.OPT_SCALE_MODE, 1)
    idx = (1 + torch.arange(T, device="cuda") % 5).view(T, 1)     # 5 experts x <= 52 rows
    sel = torch.randperm(T, generator=torch.Generator().manual_seed(hot))[:hot].cuda()
    idx[sel] = 0                                                  # expert 0: `hot` rows
    idx = idx.contiguous()
    counts = torch.bincount(idx.view(-1), minlength=wl.E)
    assert int(counts.max()) == hot
    out = moe.forward(inp.x, inp.x_sf, idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    h = oracle.HostInputs(inp.x, inp.x_sf, idx, inp.topk_w, inp.w_gate_up, inp.sf_gate_up, inp.w_down,
                          inp.sf_down, weights=weights)
    oracle.set_scale_rule("pow2")
    try:
        _, ref, bad = oracle.forward_tokens(h, np.arange(T))
    finally:
        oracle.set_scale_rule("fp32")
    assert not bad
    rel = rel_l2(out, ref)
    assert np.all(rel <= TOL), rel.max()
    moe.close()
