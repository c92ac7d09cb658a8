"""Pins of the CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to a worked example printed on the pages, to a
library routine (torch's FP8 / bf16 casts, numpy matmul), to a closed form, or to a
brute-force enumeration, so that a dropped term, a wrong index or a transposed operand
in the oracle fails here.
"""
import itertools

import numpy as np
import pytest
import torch

from conftest import OCP_E2M1, fp8_twin_of_mxfp4, golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ------------------------------------------------------------------ FP8 E4M3 ------
def torch_e4m3_value(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def torch_e4m3_encode(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_mod.e4m3_decode(codes)
    ref = torch_e4m3_value(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_library_in_range(oracle_mod):
    rng = np.random.default_rng(0)
    mag = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 200_000))
    v = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    v = np.concatenate([v, np.float32([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10])])
    assert np.array_equal(oracle_mod.e4m3_encode(v), torch_e4m3_encode(v))


def test_e4m3_encode_midpoints_round_to_even(oracle_mod):
    vals = oracle_mod.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)   # exact in fp32
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)
    enc = oracle_mod.e4m3_encode(mids)
    lo = np.arange(0x7E, dtype=np.uint8)
    expect = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(enc, expect)
    assert np.array_equal(enc, torch_e4m3_encode(mids))
    assert np.array_equal(oracle_mod.e4m3_encode(-mids), expect | 0x80)


def test_e4m3_encode_saturates(oracle_mod):
    v = np.float32([449.0, 464.0, 479.0, 480.0, 1e6, np.inf, -500.0, -np.inf])
    assert oracle_mod.e4m3_encode(v).tolist() == [0x7E] * 6 + [0xFE] * 2
    assert oracle_mod.e4m3_encode(np.float32([np.nan])).tolist() == [0x7F]


def test_bf16_rne_matches_library(oracle_mod):
    rng = np.random.default_rng(1)
    v = rng.standard_normal(100_000).astype(np.float32) * np.float32(37.0)
    bits = v.view(np.uint32)
    ties = ((bits & 0xFFFF0000) | 0x8000).view(np.float32)          # exact halfway cases
    allv = np.concatenate([v, ties, np.float32([0.0, -0.0, 1e38, -3.4e38])])
    ref = torch.from_numpy(allv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle_mod.bf16_rne(allv), ref)


# ------------------------------------------------------------------ routing -------
def test_packed_claim_worked_example(oracle_mod):
    g = dict(golden("packed_claim_3_2.txt"))
    counts = [int(c) for c in g["counts"]]
    starts, word = oracle_mod.packed_claim(counts)
    assert starts.tolist() == [int(s) for s in g["starts"]]
    assert word >> 32 == int(g["final_high"][0])
    assert word & 0xFFFFFFFF == int(g["final_low"][0])


def test_packed_claim_intervals_tile(oracle_mod):
    rng = np.random.default_rng(2)
    for _ in range(50):
        counts = rng.integers(0, 40, rng.integers(1, 30))
        starts, word = oracle_mod.packed_claim(counts)
        assert word >> 32 == counts.size and word & 0xFFFFFFFF == counts.sum()
        covered = np.zeros(int(counts.sum()), np.int32)
        for s, c in zip(starts, counts):
            covered[s:s + c] += 1
        assert np.all(covered == 1)


def test_round_robin_worked_example(oracle_mod):
    rows = golden("round_robin_3_5_2.txt")
    recv = [int(v) for v in dict(rows)["recv"]]
    src, slot = oracle_mod.round_robin(recv)
    for key, vals in rows:
        if key == "page_group":
            lo, hi = int(vals[0]), int(vals[1])
            srcs = {int(v) for v in vals[2].split(",")}
            slots = {int(v) for v in vals[3].split(",")}
            got = set(zip(src[lo:hi].tolist(), slot[lo:hi].tolist()))
            assert got == set(itertools.product(srcs, slots))
        elif key == "page_position":
            p, s, sl = map(int, vals)
            assert oracle_mod.round_robin_one(recv, p) == (s, sl)
            assert (src[p], slot[p]) == (s, sl)
    d = dict(rows)
    assert src.tolist() == [int(v) for v in d["reading_src"]]
    assert slot.tolist() == [int(v) for v in d["reading_slot"]]


def _peel_by_rounds(recv):
    """Enumerate the rounds literally: every active source emits one row per step."""
    rem = list(recv)
    nxt = [0] * len(recv)
    out = []
    while any(rem):
        active = [r for r, v in enumerate(rem) if v > 0]
        L = min(rem[r] for r in active)
        for _ in range(L):
            for r in active:
                out.append((r, nxt[r]))
                nxt[r] += 1
        for r in active:
            rem[r] -= L
    return out


def test_round_robin_brute_force_small(oracle_mod):
    for R in range(1, 5):
        for recv in itertools.product(range(6), repeat=R):
            if sum(recv) == 0:
                continue
            src, slot = oracle_mod.round_robin(recv)
            pairs = list(zip(src.tolist(), slot.tolist()))
            assert pairs == _peel_by_rounds(recv), recv
            # a permutation of {(r, s) : s < recv[r]}
            assert sorted(pairs) == [(r, s) for r in range(R) for s in range(recv[r])]


def test_block_offsets_worked_example(oracle_mod):
    g = dict(golden("segments_100_10_30.txt"))
    counts = [int(c) for c in g["counts"]]
    assert np.cumsum([0] + counts).tolist() == [int(v) for v in g["range_starts"]]
    assert oracle_mod.block_offsets(counts, 128).tolist() == [int(v) for v in g["offsets_bm128"]]
    assert oracle_mod.block_offsets(counts, 64).tolist() == [int(v) for v in g["offsets_bm64"]]


def test_block_offsets_closed_form(oracle_mod):
    rng = np.random.default_rng(3)
    for BM in (32, 64, 128):
        c = rng.integers(0, 1000, 40)
        off = oracle_mod.block_offsets(c, BM)
        assert off.tolist() == np.concatenate([[0], np.cumsum(-(-c // BM))]).tolist()


def test_route_counts_vs_bincount(oracle_mod):
    from combine_persistent_warp_gb300.workloads import make_routing
    T, E, k, R = 512, 16, 4, 4
    idx, _ = make_routing(T, E, k, seed=5, skip_frac=0.1)
    counts, recv, bad = oracle_mod.route_counts(idx, E, R)
    assert not bad
    valid = idx >= 0
    assert counts.tolist() == torch.bincount(idx[valid], minlength=E).tolist()
    src = (torch.arange(T)[:, None] // (T // R)).expand(T, k)
    ref = torch.bincount((idx * R + src)[valid], minlength=E * R).view(E, R)
    assert recv.tolist() == ref.tolist()
    bad_idx = idx.clone()
    bad_idx[3, 1] = E
    assert oracle_mod.route_counts(bad_idx, E, R)[2]
    bad_idx[3, 1] = -2
    assert oracle_mod.route_counts(bad_idx, E, R)[2]


def test_route_multiset_hand_example(oracle_mod):
    """Index-table grouping ("Mega-MoE 内核代码导读：从 Dispatch 到 WGMMA 的融合流水线" §4.3: an
    entry of token t's slot k goes to table[expert][source of t]) on a batch small enough to
    write out: T=4 tokens in R=2 sources of 2, top-2 over E=3 experts, -1 skipped."""
    idx = np.array([[0, 2], [2, -1], [1, 0], [-1, 2]], np.int64)
    got = oracle_mod.route_multiset(idx, 3, 2)
    want = {(0, 0): [(0, 0)], (0, 1): [(2, 1)], (1, 0): [], (1, 1): [(2, 0)],
            (2, 0): [(0, 1), (1, 0)], (2, 1): [(3, 1)]}
    assert got == want


def test_route_multiset_brute_force(oracle_mod):
    """Every valid (token, slot) appears exactly once, under its own expert and its token's
    source, and the group sizes equal the C oracle's per-(expert, source) counts."""
    from combine_persistent_warp_gb300.workloads import make_routing
    T, E, k, R = 96, 7, 3, 4
    idx, _ = make_routing(T, E, k, seed=8, skip_frac=0.15)
    a = idx.numpy()
    got = oracle_mod.route_multiset(idx, E, R)
    _, recv, _ = oracle_mod.route_counts(idx, E, R)
    seen = []
    for (e, r), v in got.items():
        assert len(v) == recv[e, r]
        for t, kk in v:
            assert a[t, kk] == e and t // (T // R) == r
            seen.append((t, kk))
    assert sorted(seen) == [(t, kk) for t in range(T) for kk in range(k) if a[t, kk] >= 0]


# ------------------------------------------------------------------ numerics ------
def _tiny_inputs(E=4, H=256, I=128, T=8, k=2, seed=11):
    from combine_persistent_warp_gb300 import workloads as W
    idx, w = W.make_routing(T, E, k, seed=seed)
    x, xs = W.make_activations(T, H, seed=seed)
    w1, s1, w2, s2 = W.make_weights(E, H, I, seed=seed)
    return x, xs, idx, w, w1, s1, w2, s2


def _dequant(codes, scale, rb, cb):
    v = torch_e4m3_value(codes.numpy())
    return v * np.kron(scale.numpy().astype(np.float64), np.ones((rb, cb)))


def _np_pow2_ceil(v):
    """Smallest power of two >= v via numpy's frexp (v = m * 2^e, m in [0.5, 1))."""
    v = np.asarray(v, np.float32)
    m, e = np.frexp(v)
    return np.where(m == 0.5, v, np.ldexp(np.float32(1.0), e)).astype(np.float32)


def _dense_ffn_library(x_row, xs_row, w1, s1, w2, s2, pow2=False):
    """One expert via numpy matmuls and torch FP8 casts (the single-expert special case)."""
    I = w2.shape[1]
    dx = _dequant(x_row[None, :], xs_row[None, :], 1, 128)[0]
    gu = _dequant(w1, s1, 128, 128) @ dx
    g, u = gu[:I], gu[I:]
    h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32).reshape(-1, 128)
    sf = (np.maximum(np.abs(h).max(axis=1), np.float32(1e-4)) / np.float32(448.0)).astype(np.float32)
    if pow2:
        sf = _np_pow2_ceil(sf)
    q = torch_e4m3_encode(h / sf[:, None])
    hd = (torch_e4m3_value(q) * sf[:, None].astype(np.float64)).reshape(-1)
    y = _dequant(w2, s2, 128, 128) @ hd
    return y, q.reshape(-1), sf


def test_expert_ffn_matches_dense_library_chain(oracle_mod):
    x, xs, idx, w, w1, s1, w2, s2 = _tiny_inputs(H=384, I=256)
    for t, e in [(0, 0), (3, 2), (7, 3)]:
        y, hq, hsf = oracle_mod.expert_ffn(x[t], xs[t], w1[e], s1[e], w2[e], s2[e])
        y_ref, q_ref, sf_ref = _dense_ffn_library(x[t], xs[t], w1[e], s1[e], w2[e], s2[e])
        assert np.array_equal(hsf, sf_ref)
        assert (hq == q_ref).mean() >= 0.995
        assert np.linalg.norm(y - y_ref) <= 1e-6 * np.linalg.norm(y_ref)


def test_pow2_ceil_closed_forms(oracle_mod):
    assert oracle_mod.pow2_ceil(3.0) == 4.0
    assert oracle_mod.pow2_ceil(4.0) == 4.0
    assert oracle_mod.pow2_ceil(0.3) == 0.5
    assert oracle_mod.pow2_ceil(2.0 ** -20) == 2.0 ** -20
    assert oracle_mod.pow2_ceil(float(np.nextafter(np.float32(2.0 ** -20), np.float32(1)))) == 2.0 ** -19
    assert oracle_mod.pow2_ceil(float(np.float32(1e-4) / np.float32(448))) == 2.0 ** -22


def test_pow2_ceil_defining_inequalities(oracle_mod):
    rng = np.random.default_rng(5)
    for q in (10.0 ** rng.uniform(-7, 3, 400)).astype(np.float32):
        sf = np.float32(oracle_mod.pow2_ceil(float(q)))
        m, _ = np.frexp(sf)
        assert m == 0.5 and sf >= q and sf / 2 < q


def test_expert_ffn_pow2_rule_matches_dense_chain(oracle_mod):
    """With the power-of-two rule the re-quantisation scales are the smallest powers of two
    >= the fp32-rule quotients (numpy frexp arithmetic) and the whole expert matches the
    numpy chain with that rule."""
    x, xs, idx, w, w1, s1, w2, s2 = _tiny_inputs(H=384, I=256)
    try:
        oracle_mod.set_scale_rule("pow2")
        for t, e in [(0, 0), (5, 1), (7, 3)]:
            y, hq, hsf = oracle_mod.expert_ffn(x[t], xs[t], w1[e], s1[e], w2[e], s2[e])
            y_ref, q_ref, sf_ref = _dense_ffn_library(x[t], xs[t], w1[e], s1[e], w2[e], s2[e], pow2=True)
            assert np.array_equal(hsf, sf_ref)
            assert (hq == q_ref).mean() >= 0.995
            assert np.linalg.norm(y - y_ref) <= 1e-6 * np.linalg.norm(y_ref)
            # tight: every group's largest code magnitude is at least 448/2 (below it the
            # next smaller power of two would have been enough)
            mags = np.abs(torch_e4m3_value(hq.reshape(-1, 128)))
            assert np.all(mags.max(axis=1) >= 224) and np.all(mags.max(axis=1) <= 448)
    finally:
        oracle_mod.set_scale_rule("fp32")


def test_forward_single_expert_is_dense_ffn(oracle_mod):
    x, xs, _, _, w1, s1, w2, s2 = _tiny_inputs(E=3)
    T = x.shape[0]
    idx = torch.full((T, 1), 1, dtype=torch.int64)
    w = torch.ones(T, 1)
    h = oracle_mod.HostInputs(x, xs, idx, w, w1, s1, w2, s2)
    bits, f32, bad = oracle_mod.forward_tokens(h, np.arange(T))
    assert not bad
    for t in range(T):
        y_ref, _, _ = _dense_ffn_library(x[t], xs[t], w1[1], s1[1], w2[1], s2[1])
        assert np.linalg.norm(f32[t] - y_ref) <= 1e-5 * np.linalg.norm(y_ref)
        ref_bits = torch.from_numpy(y_ref.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
        assert (bits[t] == ref_bits.numpy().view(np.uint16)).mean() > 0.99


def test_combine_worked_example(oracle_mod):
    g = dict(golden("combine_073_027.txt"))
    t = int(g["token"][0])
    e_a, e_b = (int(v) for v in g["experts"])
    w_a, w_b = (float(v) for v in g["weights"])
    x, xs, idx, w, w1, s1, w2, s2 = _tiny_inputs(E=8, T=4, k=2)
    idx[t] = torch.tensor([e_a, e_b])
    w[t] = torch.tensor([w_a, w_b])
    h = oracle_mod.HostInputs(x, xs, idx, w, w1, s1, w2, s2)
    bits, f32, _ = oracle_mod.forward_tokens(h, [t])
    ya, _, _ = oracle_mod.expert_ffn(x[t], xs[t], w1[e_a], s1[e_a], w2[e_a], s2[e_a])
    yb, _, _ = oracle_mod.expert_ffn(x[t], xs[t], w1[e_b], s1[e_b], w2[e_b], s2[e_b])
    wa, wb = np.float32(w_a), np.float32(w_b)
    expect = (float(wa) * ya + float(wb) * yb).astype(np.float32)
    assert np.array_equal(f32[0], expect)
    assert np.array_equal(bits[0], oracle_mod.bf16_rne(expect))


def test_zero_down_weights_give_zero(oracle_mod):
    x, xs, idx, w, w1, s1, w2, s2 = _tiny_inputs()
    w2 = torch.zeros_like(w2)
    h = oracle_mod.HostInputs(x, xs, idx, w, w1, s1, w2, s2)
    bits, f32, _ = oracle_mod.forward_tokens(h, np.arange(x.shape[0]))
    assert not np.any(f32) and not np.any(bits & 0x7FFF)


def test_identical_experts_make_routing_irrelevant(oracle_mod):
    x, xs, idx, w, w1, s1, w2, s2 = _tiny_inputs(E=4, k=2)
    for t in (w1, s1, w2, s2):
        t[:] = t[0:1]
    h1 = oracle_mod.HostInputs(x, xs, idx, w, w1, s1, w2, s2)
    idx2 = torch.flip(idx, dims=[1]).clone()
    idx2[:, 0] = (idx2[:, 0] + 1) % 4
    idx2[:, 1] = torch.where(idx2[:, 1] == idx2[:, 0], (idx2[:, 1] + 1) % 4, idx2[:, 1])
    h2 = oracle_mod.HostInputs(x, xs, idx2, w, w1, s1, w2, s2)
    n = np.arange(x.shape[0])
    _, f1, _ = oracle_mod.forward_tokens(h1, n)
    _, f2, _ = oracle_mod.forward_tokens(h2, n)
    assert np.allclose(f1, f2, rtol=1e-6, atol=1e-9)


def test_linear_in_gate_weights(oracle_mod):
    x, xs, idx, w, w1, s1, w2, s2 = _tiny_inputs()
    n = np.arange(x.shape[0])
    _, f1, _ = oracle_mod.forward_tokens(oracle_mod.HostInputs(x, xs, idx, w, w1, s1, w2, s2), n)
    _, f2, _ = oracle_mod.forward_tokens(oracle_mod.HostInputs(x, xs, idx, 2 * w, w1, s1, w2, s2), n)
    assert np.array_equal(f2, 2 * f1)


def test_skipped_slots_and_empty_tokens(oracle_mod):
    x, xs, idx, w, w1, s1, w2, s2 = _tiny_inputs()
    idx[2] = -1
    idx[5, 1] = -1
    h = oracle_mod.HostInputs(x, xs, idx, w, w1, s1, w2, s2)
    bits, f32, bad = oracle_mod.forward_tokens(h, [2, 5])
    assert not bad and not np.any(f32[0])
    y, _, _ = oracle_mod.expert_ffn(x[5], xs[5], w1[idx[5, 0]], s1[idx[5, 0]], w2[idx[5, 0]], s2[idx[5, 0]])
    assert np.array_equal(f32[1], (float(w[5, 0]) * y).astype(np.float32))


def test_forward_tiny_matches_independent_numpy_restatement(oracle_mod):
    """The whole tiny batch (64 tokens, 8 experts, top-2, 2 sources) against a second,
    independent float64 restatement of the layer: torch's FP8 and bf16 casts, numpy matmuls
    per (token, slot) expert FFN, and the top-k sum in fp32 in ascending slot order."""
    from combine_persistent_warp_gb300.workloads import make_inputs
    inp = make_inputs("tiny")
    h = oracle_mod.HostInputs.from_inputs(inp)
    bits, out32, bad = oracle_mod.forward_tokens(h, np.arange(h.T))
    assert not bad
    ref = np.zeros((h.T, h.H), np.float32)
    for t in range(h.T):
        acc = np.zeros(h.H, np.float32)
        for kk in range(h.k):
            e = int(h.idx[t, kk])
            if e < 0:
                continue
            y = _dense_ffn_library(inp.x[t], inp.x_sf[t], inp.w_gate_up[e], inp.sf_gate_up[e],
                                   inp.w_down[e], inp.sf_down[e])[0].astype(np.float32)
            acc = (acc + np.float32(h.w[t, kk]) * y).astype(np.float32)
        ref[t] = acc
    ref_bits = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    rel = np.linalg.norm(out32 - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert rel.max() <= 1e-3            # room for a rare one-step FP8 requant flip
    assert (bits == ref_bits).mean() >= 0.99


# ------------------------------------------------------------------ MXFP4 weights ----


def test_e2m1_decode_all_codes(oracle_mod):
    got = oracle_mod.e2m1_decode(np.arange(16, dtype=np.uint8))
    want = np.array(OCP_E2M1 + [-v for v in OCP_E2M1])
    assert np.array_equal(got, want)
    assert np.signbit(got[8]) and not np.signbit(got[0])


def test_e8m0_decode(oracle_mod):
    b = np.array([0, 1, 100, 126, 127, 128, 200, 254], np.uint8)
    assert np.array_equal(oracle_mod.e8m0_decode(b), np.ldexp(1.0, b.astype(int) - 127))
    assert np.isnan(oracle_mod.e8m0_decode(np.array([255], np.uint8))[0])


def _mxfp4_case(E=3, H=256, I=128, seed=5, span=4):
    """Random MXFP4 expert weights: uniform codes, per-32 scale bytes 120 + [0, span]."""
    g = torch.Generator().manual_seed(seed)
    def one(N, K):
        packed = torch.randint(0, 256, (E, N, K // 2), generator=g, dtype=torch.int64).to(torch.uint8)
        sf = (120 + torch.randint(0, span + 1, (E, N, K // 32), generator=g)).to(torch.uint8)
        return packed, sf
    return one(2 * I, H) + one(H, I)


def test_mxfp4_layer_equals_its_fp8_twin(oracle_mod):
    """Every output of the layer with MXFP4 weights (random codes, per-32 scales varying
    within each 128x128 block) is bit-identical to the layer with the FP8 twin weights:
    the oracle's nibble order, scale index and per-expert strides all enter."""
    from combine_persistent_warp_gb300 import workloads as W
    E, H, I, T, k = 3, 256, 128, 12, 2
    w1, s1, w2, s2 = _mxfp4_case(E, H, I)
    t1 = [fp8_twin_of_mxfp4(w1[e], s1[e]) for e in range(E)]
    t2 = [fp8_twin_of_mxfp4(w2[e], s2[e]) for e in range(E)]
    f1, g1 = torch.stack([a for a, _ in t1]), torch.stack([b for _, b in t1])
    f2, g2 = torch.stack([a for a, _ in t2]), torch.stack([b for _, b in t2])
    idx, w = W.make_routing(T, E, k, seed=3)
    x, xs = W.make_activations(T, H, seed=3, scales="pow2")
    h4 = oracle_mod.HostInputs(x, xs, idx, w, w1, s1, w2, s2, weights="mxfp4")
    h8 = oracle_mod.HostInputs(x, xs, idx, w, f1, g1, f2, g2)
    for rule in ("fp32", "pow2"):
        oracle_mod.set_scale_rule(rule)
        try:
            b4, o4, bad4 = oracle_mod.forward_tokens(h4, np.arange(T))
            b8, o8, bad8 = oracle_mod.forward_tokens(h8, np.arange(T))
        finally:
            oracle_mod.set_scale_rule("fp32")
        assert not bad4 and not bad8
        assert np.array_equal(o4, o8) and np.array_equal(b4, b8)
        assert np.abs(o4).max() > 0


def test_mxfp4_single_element_weights(oracle_mod):
    """Gate, up and down weights each with one non-zero element: the expert output is that
    element's closed form, so a swapped nibble or a wrong scale index moves it."""
    H, I = 256, 128
    x = torch.zeros(H, dtype=torch.uint8)
    xs = torch.ones(H // 128)
    c0 = 37                                   # odd column: the high nibble of byte 18
    x[c0] = 0x38                              # e4m3 1.0
    w1 = torch.zeros(2 * I, H // 2, dtype=torch.uint8)
    s1 = torch.full((2 * I, H // 32), 127, dtype=torch.uint8)
    n0 = 5
    w1[n0, c0 // 2] = 0x3 << 4                # gate (n0, c0) = code 3 = 1.5
    w1[I + n0, c0 // 2] = 0x6 << 4            # up (n0, c0) = code 6 = 4.0
    s1[n0, c0 // 32] = 129                    # x 4
    s1[I + n0, c0 // 32] = 126                # x 0.5
    w2 = torch.zeros(H, I // 2, dtype=torch.uint8)
    s2 = torch.full((H, I // 32), 127, dtype=torch.uint8)
    r0 = 200
    w2[r0, n0 // 2] = 0xD << 4 if n0 % 2 else 0xD   # down (r0, n0) = code 13 = -3.0
    s2[r0, n0 // 32] = 128                    # x 2
    y, hq, hsf = oracle_mod.expert_ffn(x, xs, w1, s1, w2, s2, weights="mxfp4")
    g, u = 1.5 * 4.0, 4.0 * 0.5
    hval = np.float32(g / (1.0 + np.exp(-g)) * u)
    sf = np.float32(hval / np.float32(448.0))
    hd = torch.tensor([float(hval / sf)]).to(torch.float8_e4m3fn).double().item() * float(sf)
    want = np.zeros(H)
    want[r0] = hd * -3.0 * 2.0
    assert np.allclose(y, want, rtol=0, atol=1e-12) and y[r0] != 0


def test_bf16_plane_mode_matches_numpy_restatement(oracle_mod):
    """Diagnostic combine mode: out[t] = bf16(fp32 sum over ascending k of bf16(fp32(w_k y_k)))
    with y_k the (pinned) expert outputs; restated with torch's bf16 casts and numpy fp32
    adds, bit for bit, on the tiny batch (skipped slots included)."""
    from combine_persistent_warp_gb300.workloads import Workload, make_inputs
    inp = make_inputs(Workload("plane", T=16, H=256, I=128, E=4, topk=3, R=2, seed=21, skip_frac=0.1))
    h = oracle_mod.HostInputs.from_inputs(inp)
    oracle_mod.set_plane_bf16(True)
    try:
        bits, out32, _ = oracle_mod.forward_tokens(h, np.arange(h.T))
    finally:
        oracle_mod.set_plane_bf16(False)
    to_bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()
    for t in range(h.T):
        acc = np.zeros(h.H, np.float32)
        for kk in range(h.k):
            e = int(h.idx[t, kk])
            if e < 0:
                continue
            y, _, _ = oracle_mod.expert_ffn(h.x[t], h.x_sf[t], h.w1[e], h.s1[e], h.w2[e], h.s2[e])
            acc = (acc + to_bf16((np.float64(h.w[t, kk]) * y).astype(np.float32))).astype(np.float32)
        want = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(bits[t], want), t
        assert np.array_equal(out32[t], acc), t
    # default mode unchanged: the double sum
    b2, o2, _ = oracle_mod.forward_tokens(h, np.arange(h.T))
    assert not np.array_equal(o2, out32)


def _mxfp4_dequant(packed, sf):
    """[N][K/2] packed E2M1 + [N][K/32] E8M0 -> float64 [N][K] from the OCP element table."""
    p = packed.numpy().astype(np.int64)
    codes = np.empty((p.shape[0], 2 * p.shape[1]), np.int64)
    codes[:, 0::2], codes[:, 1::2] = p & 0xF, p >> 4
    mags = np.array(OCP_E2M1)
    v = np.where(codes >= 8, -mags[codes & 7], mags[codes & 7])
    return v * np.ldexp(1.0, np.repeat(sf.numpy().astype(np.int64) - 127, 32, axis=1))


def test_forward_tiny_mxfp4_matches_independent_numpy_restatement(oracle_mod):
    """The tiny batch with MXFP4 weights (generator's OCP conversion) against a second
    restatement: OCP-table dequantisation, numpy fp64 matmuls, torch FP8 casts for the
    power-of-two requant, the top-k sum in fp32 ascending k."""
    from combine_persistent_warp_gb300.workloads import make_inputs
    inp = make_inputs("tiny-mxfp4")
    h = oracle_mod.HostInputs.from_inputs(inp)
    assert h.weights == "mxfp4"
    oracle_mod.set_scale_rule("pow2")
    try:
        bits, out32, bad = oracle_mod.forward_tokens(h, np.arange(h.T))
    finally:
        oracle_mod.set_scale_rule("fp32")
    assert not bad
    I = h.I
    W1 = [_mxfp4_dequant(inp.w_gate_up[e], inp.sf_gate_up[e]) for e in range(h.E)]
    W2 = [_mxfp4_dequant(inp.w_down[e], inp.sf_down[e]) for e in range(h.E)]
    ref = np.zeros((h.T, h.H), np.float32)
    for t in range(h.T):
        dx = _dequant(inp.x[t][None, :], inp.x_sf[t][None, :], 1, 128)[0]
        acc = np.zeros(h.H, np.float32)
        for kk in range(h.k):
            e = int(h.idx[t, kk])
            if e < 0:
                continue
            gu = W1[e] @ dx
            hv = (gu[:I] / (1.0 + np.exp(-gu[:I])) * gu[I:]).astype(np.float32).reshape(-1, 128)
            sf = _np_pow2_ceil(np.maximum(np.abs(hv).max(axis=1), np.float32(1e-4)) / np.float32(448.0))
            q = torch_e4m3_encode(hv / sf[:, None])
            hd = (torch_e4m3_value(q) * sf[:, None].astype(np.float64)).reshape(-1)
            y = (W2[e] @ hd).astype(np.float32)
            acc = (acc + np.float32(h.w[t, kk]) * y).astype(np.float32)
        ref[t] = acc
    rel = np.linalg.norm(out32 - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert rel.max() <= 1e-3
