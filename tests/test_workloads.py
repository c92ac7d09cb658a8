"""Synthetic workload recipe checks (CPU only)."""
import numpy as np
import torch

from combine_persistent_warp_gb300 import workloads as W


def test_routing_without_replacement_and_normalised():
    idx, w = W.make_routing(256, 32, 8, seed=1)
    assert idx.shape == (256, 8) and idx.dtype == torch.int64
    for row in idx.tolist():
        assert len(set(row)) == 8
    assert torch.allclose(w.sum(1), torch.ones(256), atol=1e-6)


def test_skewed_routing_shape():
    wl = W.WORKLOADS["skewed"]
    idx, w = W.make_routing(wl.T, wl.E, wl.topk, seed=wl.seed, routing=wl.routing,
                            zipf_s=wl.zipf_s, skip_frac=wl.skip_frac)
    skipped = (idx == -1).float().mean().item()
    assert abs(skipped - 0.05) < 1e-3
    # without replacement an expert gets at most T rows, i.e. at most E/topk times the mean
    ratio = W.skew_ratio(idx, wl.E)
    assert 5.0 < ratio <= wl.E / wl.topk + 1e-9


def test_quantisers_roundtrip_within_fp8_error():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(4, 512, generator=g)
    q, sf = W.quantize_1x128(x)
    back = q.view(torch.float8_e4m3fn).float().view(4, 4, 128) * sf[:, :, None]
    assert torch.allclose(back.view(4, 512), x, rtol=0.07, atol=1e-6)
    w = torch.randn(256, 384, generator=g) * 0.02
    q, sf = W.quantize_128x128(w)
    assert sf.shape == (2, 3)
    back = q.view(torch.float8_e4m3fn).float().view(2, 128, 3, 128) * sf[:, None, :, None]
    assert torch.allclose(back.reshape(256, 384), w, rtol=0.07, atol=1e-6)


def test_make_inputs_shapes():
    inp = W.make_inputs("tiny")
    wl = inp.wl
    assert inp.x.shape == (wl.T, wl.H) and inp.x.dtype == torch.uint8
    assert inp.x_sf.shape == (wl.T, wl.H // 128)
    assert inp.w_gate_up.shape == (wl.E, 2 * wl.I, wl.H)
    assert inp.sf_gate_up.shape == (wl.E, 2 * wl.I // 128, wl.H // 128)
    assert inp.w_down.shape == (wl.E, wl.H, wl.I)
    assert inp.sf_down.shape == (wl.E, wl.H // 128, wl.I // 128)
    again = W.make_inputs("tiny")
    assert torch.equal(inp.x, again.x) and torch.equal(inp.topk_idx, again.topk_idx)


def test_quantize_mxfp4_scale_rule_and_error_bound():
    """MXFP4 synthesis: each 32-run's scale is 2^(floor(log2 amax) - 2), the decoded values
    (oracle decoders) lie within half an E2M1 step of v (saturated runs: within 2 X), and the
    packing puts element 2j in the low nibble."""
    import oracle
    from combine_persistent_warp_gb300.workloads import quantize_mxfp4
    g = torch.Generator().manual_seed(9)
    w = torch.randn(64, 256, generator=g) * 0.02
    w[3, :32] = 0.0                                   # an all-zero run
    packed, sf = quantize_mxfp4(w)
    assert packed.shape == (64, 128) and sf.shape == (64, 8)
    amax = w.view(64, 8, 32).abs().amax(dim=2).double().numpy()
    ex = sf.numpy().astype(np.int64) - 127
    nz = amax > 0
    assert np.array_equal(ex[nz], (np.floor(np.log2(amax[nz])) - 2).astype(np.int64))
    assert ex[3, 0] == -127
    p = packed.numpy()
    codes = np.stack([p & 0xF, p >> 4], axis=2).reshape(64, 256)
    X = np.repeat(np.ldexp(1.0, ex), 32, axis=1)
    q = oracle.e2m1_decode(codes) * X
    err = np.abs(q - w.double().numpy())
    # E2M1 steps: 0.5 up to 2, 1 up to 4, 2 up to 6; |v|/X < 8 always
    a = np.abs(w.double().numpy()) / X
    bound = np.where(a <= 2, 0.25, np.where(a <= 4, 0.5, np.where(a <= 6, 1.0, 2.0))) * X
    assert np.all(err <= bound + 1e-18)
