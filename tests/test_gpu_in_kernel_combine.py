"""The top-k combine run inside the expert FFN kernel (MOE_OPT_COMBINE_MODE = 1).

With it, every down tile's scattered rows are counted per (token, 256-column n-tile) and the
FFN kernel's epilogue warps reduce each (token, n-tile) whose routed rows are all stored
("DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §9: the top-k reduce in the
persistent kernel's epilogue warps; §8.2: one bf16 plane per top-k slot).  The reduce is the
separate combine kernel's arithmetic in the same order (fp32 over the valid slots, ascending,
then bf16), so the two modes must give the same output bits; the in-kernel mode is also
compared with the oracle directly (per-token relative L2 <= 2e-2), on batches with skipped
slots, unrouted tokens, one slot per token, shared experts and H an odd multiple of 128.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_persistent_warp_gb300 import FusedMoE, MoeError
from combine_persistent_warp_gb300 import native
from combine_persistent_warp_gb300.workloads import Workload, make_inputs, make_weights
from conftest import block_cover_tokens, blocks_of_tokens

pytestmark = pytest.mark.gpu

TOL = 2e-2
IN_FFN, KERNEL = native.COMBINE_IN_FFN, native.COMBINE_KERNEL


def rel_l2(got, ref):
    g = got.float().cpu().numpy()
    den = np.linalg.norm(ref, axis=1)
    num = np.linalg.norm(g - ref, axis=1)
    return np.where(den > 0, num / np.maximum(den, 1e-30), num)


def bits(t):
    return t.view(torch.int16)


def layer(wl_or_name, T_max=None):
    torch.cuda.set_device(0)
    inp = make_inputs(wl_or_name, device="cuda")
    wl = inp.wl
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R).reserve(T_max or wl.T)
    moe.load(inp)
    return moe, inp


def oracle_ref(inp, toks, idx=None, w=None):
    wl = inp.wl
    h = oracle.HostInputs(inp.x, inp.x_sf, inp.topk_idx if idx is None else idx, inp.topk_w if w is None else w,
                          inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down,
                          weights=getattr(wl, "weights", "fp8"))
    oracle.set_scale_rule(wl.scales)
    try:
        _, ref, bad = oracle.forward_tokens(h, np.asarray(toks))
    finally:
        oracle.set_scale_rule("fp32")
    assert not bad
    return ref


def forward_mode(moe, inp, mode, idx=None, w=None, out=None):
    moe.set_option(native.OPT_COMBINE_MODE, mode)
    o = moe.forward(inp.x, inp.x_sf, inp.topk_idx if idx is None else idx, inp.topk_w if w is None else w, out=out)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    return o


CASES = ["tiny", "decode", "prefill", "skewed", "large", "tiny-pow2", "decode-pow2", "skewed-pow2",
         "tiny-mxfp4", "decode-mxfp4", "large-mxfp4"]


@pytest.mark.parametrize("name", CASES)
def test_in_kernel_combine_equals_the_combine_kernel(name):
    """Same output bits in both modes, twice in a row in the in-kernel mode (the last FFN CTA's
    workspace reset) and again after switching back."""
    moe, inp = layer(name)
    ref = forward_mode(moe, inp, KERNEL).clone()
    for _ in range(2):
        out = forward_mode(moe, inp, IN_FFN)
        assert torch.equal(bits(out), bits(ref))
    assert torch.equal(bits(forward_mode(moe, inp, KERNEL)), bits(ref))
    moe.close()


@pytest.mark.parametrize("name", ["prefill", "skewed-pow2", "large-mxfp4"])
def test_in_kernel_combine_against_the_oracle_on_every_m_block(name):
    """The in-kernel mode against the oracle on a cover of the pool: at least one compared row
    in every M-block of every expert (the last partly filled one and the last wave included)."""
    moe, inp = layer(name)
    out = forward_mode(moe, inp, IN_FFN)
    dbg = moe.debug_routing(inp.wl.T)
    toks = block_cover_tokens(dbg, extra=(0, inp.wl.T - 1))
    assert blocks_of_tokens(dbg, toks) == set(range(int(dbg["block_offset"][-1])))
    ref = oracle_ref(inp, toks)
    rel = rel_l2(out[torch.as_tensor(toks, device=out.device)], ref)
    assert np.all(rel <= TOL), rel.max()
    moe.close()


def test_skipped_slots_unrouted_tokens_and_odd_hidden_size():
    """H = 5 x 128 (the last n-tile has 128 columns), Zipf routing with skipped slots, and a
    few tokens with no routed slot at all (zero rows written by the routing kernel into an
    output buffer that starts as NaN): every token against the oracle."""
    T = 512
    wl = Workload("in-ffn-odd-h", T=T, H=640, I=256, E=6, topk=3, R=4, routing="zipf", zipf_s=1.1,
                  skip_frac=0.05, seed=81)
    moe, inp = layer(wl)
    idx = inp.topk_idx.clone()
    idx[[3, 100, 511]] = -1
    idx = idx.contiguous()
    nan = torch.full((T, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = forward_mode(moe, inp, IN_FFN, idx=idx, out=nan)
    assert not torch.any(out[[3, 100, 511]].float() != 0)
    ref = oracle_ref(inp, np.arange(T), idx=idx)
    rel = rel_l2(out, ref)
    assert np.all(rel <= TOL), rel.max()
    assert torch.equal(bits(out), bits(forward_mode(moe, inp, KERNEL, idx=idx)))
    moe.close()


def test_every_slot_skipped_and_one_slot_per_token():
    moe, inp = layer(Workload("in-ffn-k1", T=256, H=256, I=128, E=8, topk=1, R=2, seed=82))
    out = forward_mode(moe, inp, IN_FFN)          # top-1: every scattered row completes its token
    ref = oracle_ref(inp, np.arange(256))
    assert np.all(rel_l2(out, ref) <= TOL)
    idx = torch.full((256, 1), -1, dtype=torch.int64, device="cuda")
    nan = torch.full((256, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = forward_mode(moe, inp, IN_FFN, idx=idx, out=nan)
    assert not torch.any(out.float() != 0)
    moe.close()


def test_shared_experts_in_kernel_combine():
    """A shared expert's plane (slot topk) is reduced like the routed ones."""
    wl = Workload("in-ffn-shared", T=256, H=256, I=256, E=8, topk=2, R=2, seed=83)
    torch.cuda.set_device(0)
    inp = make_inputs(wl, device="cuda")
    sw = make_weights(1, wl.H, wl.I, seed=wl.seed + 1000, device="cuda", scales=wl.scales)
    moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R, n_shared=1).reserve(wl.T)
    moe.load_weights(inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down)
    moe.load_shared_weights(*sw)
    a = forward_mode(moe, inp, KERNEL).clone()
    b = forward_mode(moe, inp, IN_FFN)
    assert torch.equal(bits(a), bits(b))
    moe.close()


def test_in_kernel_combine_errors_then_recovers():
    """A routing-kernel time-out and a bad expert id in the in-kernel mode: reported, and the
    next forward (after moe_get_error) is correct again."""
    moe, inp = layer("tiny")
    ref = forward_mode(moe, inp, KERNEL).clone()
    moe.set_option(native.OPT_COMBINE_MODE, IN_FFN)
    moe.set_option(native.OPT_TIMEOUT_NS, 20_000_000)
    moe.set_option(native.OPT_DEBUG_SKIP_BARRIER, 1)
    moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 7
    moe.set_option(native.OPT_DEBUG_SKIP_BARRIER, 0)
    moe.set_option(native.OPT_TIMEOUT_NS, 2_000_000_000)
    assert torch.equal(bits(forward_mode(moe, inp, IN_FFN)), bits(ref))
    bad = inp.topk_idx.clone()
    bad[5, 1] = 8
    moe.forward(inp.x, inp.x_sf, bad, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 6
    assert torch.equal(bits(forward_mode(moe, inp, IN_FFN)), bits(ref))
    for v in (-1, 3):
        with pytest.raises(MoeError) as ei:
            moe.set_option(native.OPT_COMBINE_MODE, v)
        assert ei.value.code == 1
    moe.close()


@pytest.mark.parametrize("name", ["tiny", "tiny-pow2", "tiny-mxfp4"])
def test_in_kernel_combine_host_entry_point(name):
    """Host buffers: the pinned output written in place by the FFN kernel (in-kernel mode, and
    the automatic mode, which picks it for a pinned output of the block-scaled kernel and the
    combine kernel otherwise), a misaligned pinned output through the staging buffer, and
    pageable buffers: all equal the device entry point."""
    moe, inp = layer(name)
    dev = forward_mode(moe, inp, KERNEL).cpu()
    pin = lambda t: t.cpu().pin_memory()
    px, psf, pidx, pw = pin(inp.x), pin(inp.x_sf), pin(inp.topk_idx), pin(inp.topk_w)
    T, H = dev.shape
    for mode in (IN_FFN, native.COMBINE_AUTO):
        moe.set_option(native.OPT_COMBINE_MODE, mode)
        o = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        moe.forward_host(px, psf, pidx, pw, out=o)
        assert torch.equal(bits(dev), bits(o))
        big = torch.empty(T * H + 1, dtype=torch.bfloat16).pin_memory()
        odd = big[1:].view(T, H)
        moe.forward_host(px, psf, pidx, pw, out=odd)
        assert torch.equal(bits(dev), bits(odd))
        page = moe.forward_host(inp.x.cpu(), inp.x_sf.cpu(), inp.topk_idx.cpu(), inp.topk_w.cpu(),
                                out=torch.empty(T, H, dtype=torch.bfloat16))
        assert torch.equal(bits(dev), bits(page))
    assert moe.get_error() == 0
    moe.close()


def test_widest_route_32_slots():
    """topk = 32 (the largest routed-slot count, the full width of a token's slot mask; four
    rounds of eight plane loads in the reduce) with skipped slots: both combine modes against
    the oracle on every token, and bit-identical to each other."""
    T = 128
    wl = Workload("in-ffn-k32", T=T, H=256, I=128, E=40, topk=32, R=2, skip_frac=0.1, seed=84)
    moe, inp = layer(wl)
    ref = oracle_ref(inp, np.arange(T))
    outs = []
    for mode in (KERNEL, IN_FFN):
        out = forward_mode(moe, inp, mode)
        rel = rel_l2(out, ref)
        assert np.all(rel <= TOL), rel.max()
        outs.append(out.clone())
    assert torch.equal(bits(outs[0]), bits(outs[1]))
    moe.close()
