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
