"""GPU parity of the fused MoE layer against the CPU oracle, through the C ABI.

Integers are compared bit-exactly: per-expert counts, per-(expert, source) counts,
expert block offsets, the round-robin source sequence of every expert, the multiset of
(expert, source, token, slot) entries (slot order inside a source comes from atomics,
so it is compared after sorting), the index-table entry each pool row was read from,
and the gathered row bytes and scales.  Floats use the per-token relative L2 bound
||out - ref|| / ||ref|| <= 2e-2 on every compared token.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_persistent_warp_gb300 import FusedMoE, MoeError
from combine_persistent_warp_gb300 import native
from combine_persistent_warp_gb300.workloads import WORKLOADS, Workload, make_inputs
from conftest import block_cover_tokens, blocks_of_tokens

pytestmark = pytest.mark.gpu

TOL = 2e-2
# tokens compared against the oracle per workload: all of them (tiny, decode), else a seeded
# sample plus a cover of the pool (at least one row in every M-block of every expert)
SAMPLES = {"tiny": None, "decode": None, "prefill": 12, "skewed": 12, "large": 12}


def rel_l2(got_bf16: torch.Tensor, ref: np.ndarray) -> np.ndarray:
    g = got_bf16.float().cpu().numpy()
    den = np.linalg.norm(ref, axis=1)
    num = np.linalg.norm(g - ref, axis=1)
    return np.where(den > 0, num / np.maximum(den, 1e-30), num)


class Case:
    def __init__(self, name: str):
        torch.cuda.set_device(0)
        self.inp = make_inputs(name, device="cuda")
        self.wl = self.inp.wl
        wl = self.wl
        self.moe = FusedMoE(wl.E, wl.H, wl.I, wl.topk, wl.R).reserve(wl.T)
        self.moe.load_weights(self.inp.w_gate_up, self.inp.sf_gate_up, self.inp.w_down,
                              self.inp.sf_down)
        self.out = self.moe.forward(self.inp.x, self.inp.x_sf, self.inp.topk_idx, self.inp.topk_w)
        torch.cuda.synchronize()
        self.status = self.moe.get_error()
        self.host = oracle.HostInputs.from_inputs(self.inp)

    def sample_tokens(self, n):
        T = self.wl.T
        if n is None or n >= T:
            return np.arange(T)
        rng = np.random.default_rng(1234)
        picks = set(rng.choice(T, n - 2, replace=False).tolist()) | {0, T - 1}
        skipped = np.nonzero((self.host.idx < 0).any(axis=1))[0]
        if skipped.size:
            picks.add(int(skipped[0]))
        return np.array(sorted(picks))


_cases = {}


def case(name) -> Case:
    if name not in _cases:      # all five workloads fit in HBM together (~12 GB)
        _cases[name] = Case(name)
    return _cases[name]


def check_routing(c: Case):
    wl, moe, h = c.wl, c.moe, c.host
    E, R, K, T = wl.E, wl.R, wl.topk, wl.T
    Tsrc = T // R
    dbg = moe.debug_routing(T)
    counts, recv, bad = oracle.route_counts(h.idx, E, R)
    assert not bad
    assert np.array_equal(dbg["counts"], counts)
    assert np.array_equal(dbg["recv"], recv)
    BM = dbg["block_m"]
    off = oracle.block_offsets(counts, BM)
    assert np.array_equal(dbg["block_offset"], off)
    assert dbg["P"] == off[-1] * BM
    meta = dbg["meta"].astype(np.int64)
    table = moe.debug_buffer("table")
    pool_x = moe.debug_buffer("pool_x")
    pool_sf = moe.debug_buffer("pool_sf")
    gpu_keys = []
    for e in range(E):
        n = int(counts[e])
        if n == 0:
            continue
        rows = off[e] * BM + np.arange(n)
        m = meta[rows]
        src, slot = oracle.round_robin(recv[e])
        assert np.array_equal(m[:, 0], src), f"round-robin source order of expert {e}"
        # the row came from the table entry at (e, source, slot) of that round-robin step
        tok_in_src = m[:, 1] - m[:, 0] * Tsrc
        assert np.array_equal(table[e, src, slot], tok_in_src * K + m[:, 2])
        assert np.array_equal(pool_x[rows], h.x[m[:, 1]])
        assert np.array_equal(pool_sf[:, rows], h.x_sf[m[:, 1]].T)
        gpu_keys.append(((e * R + m[:, 0]) * T + m[:, 1]) * K + m[:, 2])
    gpu_keys = np.sort(np.concatenate(gpu_keys)) if gpu_keys else np.zeros(0, np.int64)
    ref = oracle.route_multiset(h.idx, E, R)
    ref_keys = np.sort(np.array([((e * R + r) * T + t) * K + kk for (e, r), v in ref.items() for t, kk in v],
                                np.int64))
    assert np.array_equal(gpu_keys, ref_keys)
    return dbg


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_routing_bit_exact(name):
    c = case(name)
    assert c.status == 0
    check_routing(c)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_output_parity(name):
    c = case(name)
    assert c.status == 0
    dbg = c.moe.debug_routing(c.wl.T)
    toks = block_cover_tokens(dbg, extra=c.sample_tokens(SAMPLES[name]).tolist())
    assert blocks_of_tokens(dbg, toks) == set(range(int(dbg["block_offset"][-1])))
    _, ref, bad = oracle.forward_tokens(c.host, toks)
    assert not bad
    rel = rel_l2(c.out[torch.as_tensor(toks, device=c.out.device)], ref)
    assert np.all(rel <= TOL), f"max per-token rel L2 {rel.max():.3e} at token {toks[rel.argmax()]}"


@pytest.mark.parametrize("name", ["tiny", "decode", "large"])
def test_swiglu_requant_stage(name):
    """Sampled pool rows of the gate_up GEMM + SwiGLU + 1x128 requant vs the oracle."""
    c = case(name)
    dbg = c.moe.debug_routing(c.wl.T)
    act = c.moe.debug_buffer("act")
    act_sf = c.moe.debug_buffer("act_sf")
    h = c.host
    BM, off, meta = dbg["block_m"], dbg["block_offset"], dbg["meta"]
    rng = np.random.default_rng(7)
    experts = np.nonzero(dbg["counts"])[0]
    for e in rng.choice(experts, min(4, experts.size), replace=False):
        n = int(dbg["counts"][e])
        for i in sorted({0, n - 1, int(rng.integers(n))}):
            row = off[e] * BM + i
            t = int(meta[row, 1])
            _, hq, hsf = oracle.expert_ffn(h.x[t], h.x_sf[t], h.w1[e], h.s1[e], h.w2[e], h.s2[e])
            ref = oracle.e4m3_decode(hq) * np.repeat(hsf.astype(np.float64), 128)
            got = oracle.e4m3_decode(act[row]) * np.repeat(act_sf[:, row].astype(np.float64), 128)
            assert np.linalg.norm(got - ref) <= 1e-2 * np.linalg.norm(ref)
            assert (act[row] == hq).mean() >= 0.97
            assert np.allclose(act_sf[:, row], hsf, rtol=1e-4)


# ----------------------------------------------------------------- edge cases -------
def tiny_layer(T_max=64, E=8, H=256, I=128, k=2, R=2, seed=21):
    wl = Workload("edge", T=T_max, H=H, I=I, E=E, topk=k, R=R, seed=seed)
    inp = make_inputs(wl, device="cuda")
    moe = FusedMoE(E, H, I, k, R).reserve(T_max)
    moe.load_weights(inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down)
    return moe, inp


def run_and_compare(moe, inp, idx, w, T):
    x, xs = inp.x[:T].contiguous(), inp.x_sf[:T].contiguous()
    out = moe.forward(x, xs, idx, w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    h = oracle.HostInputs(x, xs, idx, w, inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down)
    _, ref, _ = oracle.forward_tokens(h, np.arange(T))
    rel = rel_l2(out, ref)
    assert np.all(rel <= TOL), rel.max()
    return out, ref


@pytest.mark.parametrize("H", [384, 640])
def test_hidden_size_odd_multiple_of_128(H):
    """H = 3 or 5 x 128: the down GEMM's last 256-column tile covers 128 real columns (its
    other half runs on zero weight rows and stores nothing); every token against the oracle,
    with a Zipf-skewed routing so experts hold several M-blocks and a partly filled last one."""
    T = 384
    wl = Workload("odd-h", T=T, H=H, I=256, E=6, topk=3, R=4, routing="zipf", zipf_s=1.1, skip_frac=0.05,
                  seed=70 + H)
    inp = make_inputs(wl, device="cuda")
    moe = FusedMoE(wl.E, H, wl.I, wl.topk, wl.R).reserve(T)
    moe.load_weights(inp.w_gate_up, inp.sf_gate_up, inp.w_down, inp.sf_down)
    assert moe.info().H == H
    out, _ = run_and_compare(moe, inp, inp.topk_idx, inp.topk_w, T)
    assert out.shape == (T, H)


def test_empty_batch():
    moe, inp = tiny_layer()
    e = torch.empty(0, 256, dtype=torch.uint8, device="cuda")
    out = moe.forward(e, torch.empty(0, 2, device="cuda"), torch.empty(0, 2, dtype=torch.int64, device="cuda"),
                      torch.empty(0, 2, device="cuda"))
    assert out.shape == (0, 256) and moe.get_error() == 0


def test_all_slots_skipped_gives_zero():
    moe, inp = tiny_layer()
    idx = torch.full((64, 2), -1, dtype=torch.int64, device="cuda")
    out = moe.forward(inp.x, inp.x_sf, idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    assert not torch.any(out.float() != 0)
    dbg = moe.debug_routing(64)
    assert dbg["counts"].sum() == 0 and dbg["P"] == 0


def test_ragged_batch_and_single_hot_expert():
    moe, inp = tiny_layer(T_max=160)
    T = 158                                     # 79 tokens per source, not a tile multiple
    idx = inp.topk_idx[:T].clone()
    idx[:, 0] = 3                               # expert 3 receives every token
    idx[:, 1] = torch.where(idx[:, 1] == 3, torch.full_like(idx[:, 1], -1), idx[:, 1])
    w = inp.topk_w[:T].contiguous()
    run_and_compare(moe, inp, idx.contiguous(), w, T)
    dbg = moe.debug_routing(T)
    assert dbg["counts"][3] == T
    assert dbg["block_offset"][4] - dbg["block_offset"][3] == -(-T // dbg["block_m"])


def test_repeat_is_deterministic_and_stats_accumulate():
    moe, inp = tiny_layer(seed=5)
    a = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w).clone()
    b = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    counts, _, _ = oracle.route_counts(inp.topk_idx, 8, 2)
    assert np.array_equal(moe.cumulative_expert_rows(), 2 * counts.astype(np.uint64))


def test_host_entry_point_matches_device_entry_point():
    """Host-buffer entry point: pinned inputs read in place and pinned output written in
    place, pageable buffers through copies, a misaligned pinned output through the staging
    buffer, and the asynchronous variant with two forwards in flight: all equal the device
    entry point bit for bit."""
    moe, inp = tiny_layer(seed=9)
    dev = moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w).cpu()
    torch.cuda.synchronize()
    pin = lambda t: t.cpu().pin_memory()
    px, psf, pidx, pw = pin(inp.x), pin(inp.x_sf), pin(inp.topk_idx), pin(inp.topk_w)
    host = moe.forward_host(px, psf, pidx, pw)
    assert torch.equal(dev.view(torch.int16), host.view(torch.int16))
    pageable = moe.forward_host(inp.x.cpu(), inp.x_sf.cpu(), inp.topk_idx.cpu(), inp.topk_w.cpu(),
                                out=torch.empty(64, 256, dtype=torch.bfloat16))
    assert torch.equal(dev.view(torch.int16), pageable.view(torch.int16))
    big = torch.empty(64 * 256 + 1, dtype=torch.bfloat16).pin_memory()
    odd = big[1:].view(64, 256)                      # 2-byte offset: not 16-byte aligned
    moe.forward_host(px, psf, pidx, pw, out=odd)
    assert torch.equal(dev.view(torch.int16), odd.view(torch.int16))
    # asynchronous: a second batch (other routing) enqueued before the first has finished
    idx2 = torch.flip(inp.topk_idx, dims=[1]).contiguous()
    w2 = torch.flip(inp.topk_w, dims=[1]).contiguous()
    dev2 = moe.forward(inp.x, inp.x_sf, idx2, w2).cpu()
    torch.cuda.synchronize()
    o1 = torch.empty(64, 256, dtype=torch.bfloat16).pin_memory()
    o2 = torch.empty(64, 256, dtype=torch.bfloat16).pin_memory()
    pidx2, pw2 = pin(idx2), pin(w2)
    moe.forward_host(px, psf, pidx, pw, out=o1, wait=False)
    moe.forward_host(px, psf, pidx2, pw2, out=o2, wait=False)
    assert moe.get_error() == 0                      # synchronizes the stream
    assert torch.equal(dev.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(dev2.view(torch.int16), o2.view(torch.int16))


def test_capacity_and_shape_errors():
    moe, inp = tiny_layer(T_max=32)
    with pytest.raises(MoeError) as ei:
        big = make_inputs("tiny", device="cuda")
        moe.forward(big.x, big.x_sf, big.topk_idx, big.topk_w)        # 64 > 32 reserved
    assert ei.value.code == 3
    with pytest.raises(MoeError) as ei:
        moe.forward(inp.x[:31], inp.x_sf[:31], inp.topk_idx[:31], inp.topk_w[:31])   # T % R
    assert ei.value.code == 1


def test_bad_index_is_reported_then_recovers():
    moe, inp = tiny_layer()
    idx = inp.topk_idx.clone()
    idx[5, 1] = 8                                # == E
    moe.forward(inp.x, inp.x_sf, idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 6
    run_and_compare(moe, inp, inp.topk_idx, inp.topk_w, 64)


def test_slot_overflow_is_reported_then_recovers():
    moe, inp = tiny_layer()
    idx = torch.zeros(64, 2, dtype=torch.int64, device="cuda")   # same expert twice per token
    moe.forward(inp.x, inp.x_sf, idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 8
    run_and_compare(moe, inp, inp.topk_idx, inp.topk_w, 64)


def test_barrier_timeout_is_reported_then_recovers():
    moe, inp = tiny_layer()
    moe.set_option(native.OPT_TIMEOUT_NS, 20_000_000)
    moe.set_option(native.OPT_DEBUG_SKIP_BARRIER, 1)
    moe.forward(inp.x, inp.x_sf, inp.topk_idx, inp.topk_w)
    torch.cuda.synchronize()
    assert moe.get_error() == 7
    # the sticky word blocks forwards until it has been read; after that, normal again
    moe.set_option(native.OPT_DEBUG_SKIP_BARRIER, 0)
    moe.set_option(native.OPT_TIMEOUT_NS, 2_000_000_000)
    run_and_compare(moe, inp, inp.topk_idx, inp.topk_w, 64)


# ----------------------------------------------------------------- FFN kernel mode -----
def test_multi_block_experts_and_mode_values():
    """Experts with 1-3 M-blocks (odd counts among them), every token against the oracle;
    MOE_OPT_FFN_MODE takes 0 (automatic) and 1 (one CTA per tile), the same kernel, and
    refuses anything else."""
    T = 1024
    moe, inp = tiny_layer(T_max=T, E=8, H=256, I=256, k=2, R=2, seed=33)
    counts, _, _ = oracle.route_counts(inp.topk_idx, 8, 2)
    blocks = -(-counts.astype(np.int64) // 128)
    assert np.any(blocks % 2 == 1) and np.any(blocks >= 2)
    outs = []
    for mode in (0, 1):
        moe.set_option(native.OPT_FFN_MODE, mode)
        out, _ = run_and_compare(moe, inp, inp.topk_idx, inp.topk_w, T)
        outs.append(out.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    for bad in (-1, 2):
        with pytest.raises(MoeError) as ei:
            moe.set_option(native.OPT_FFN_MODE, bad)
        assert ei.value.code == 1
