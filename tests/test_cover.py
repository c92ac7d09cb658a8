"""The test helper that picks compared tokens so that every M-block of the pool holds a row of
one of them (used by the full-size GPU parity tests), checked on CPU on routing results the
oracle builds for the five batch shapes."""
import numpy as np
import pytest

import oracle
from combine_persistent_warp_gb300.workloads import WORKLOADS, make_routing
from conftest import block_cover_tokens, blocks_of_tokens


def oracle_routing(wl, BM=128):
    """What moe_debug_routing reports, from the oracle: counts, block offsets and the pool
    rows' {source, token, slot} (the slot order inside one source is free; ascending here)."""
    idx, _ = make_routing(wl.T, wl.E, wl.topk, seed=wl.seed, routing=wl.routing, zipf_s=wl.zipf_s,
                          skip_frac=wl.skip_frac)
    counts, recv, _ = oracle.route_counts(idx, wl.E, wl.R)
    off = oracle.block_offsets(counts, BM)
    groups = oracle.route_multiset(idx, wl.E, wl.R)
    meta = np.full((int(off[-1]) * BM, 3), 0xFFFFFFFF, np.uint32)   # padding rows: garbage
    for e in range(wl.E):
        if counts[e] == 0:
            continue
        src, slot = oracle.round_robin(recv[e])
        rows = int(off[e]) * BM + np.arange(int(counts[e]))
        for row, r, sl in zip(rows, src, slot):
            t, kk = groups[(e, int(r))][int(sl)]
            meta[row] = (r, t, kk)
    return {"counts": counts, "recv": recv, "block_offset": off, "meta": meta, "block_m": BM}


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_cover_reaches_every_block(name):
    wl = WORKLOADS[name]
    dbg = oracle_routing(wl)
    toks = block_cover_tokens(dbg, extra=[0, wl.T - 1])
    nblk = int(dbg["block_offset"][-1])
    assert blocks_of_tokens(dbg, toks) == set(range(nblk))
    assert {0, wl.T - 1} <= set(toks.tolist())
    # each token holds at most topk rows, so at least nblk / topk tokens are needed; the
    # greedy cover stays well below one token per block
    assert len(toks) >= nblk / wl.topk
    assert len(toks) <= max(2 + nblk // 2, 4)


def test_cover_ignores_padding_rows():
    wl = WORKLOADS["tiny"]
    dbg = oracle_routing(wl)
    toks = block_cover_tokens(dbg)
    assert all(0 <= t < wl.T for t in toks.tolist())
