import os
import sys

import numpy as np
import torch

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden(name):
    """Parse a tests/golden fixture: '#' lines are comments, others 'key v1 v2 ...'."""
    rows = []
    with open(os.path.join(ROOT, "tests", "golden", name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.append((key, vals))
    return rows


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.lib()
    return oracle


# OCP Microscaling Formats (MX) v1.0, FP4 E2M1 element: the eight magnitudes of codes 0..7
# (bit 3 is the sign); E8M0 scale bytes are 2^(b-127) with 0xFF = NaN.
OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def fp8_twin_of_mxfp4(packed, sf):
    """An FP8 weight with the same element values as an MXFP4 one ([N][K/2] packed, [N][K/32]
    E8M0): per 128x128 block the scale 2^m with m the block's smallest scale exponent, and
    e4m3 codes (torch's cast) of value / 2^m, exact while each block's exponents span <= 6."""
    p = packed.numpy().astype(np.int64)
    N = p.shape[0]
    codes = np.empty((N, 2 * p.shape[1]), np.int64)
    codes[:, 0::2] = p & 0xF
    codes[:, 1::2] = p >> 4
    mags = np.array(OCP_E2M1)
    val = np.where(codes >= 8, -mags[codes & 7], mags[codes & 7])
    ex = sf.numpy().astype(np.int64) - 127                       # [N][K/32]
    val = val * np.ldexp(1.0, np.repeat(ex, 32, axis=1))
    K = val.shape[1]
    m = ex.reshape(N // 128, 128, K // 128, 4).min(axis=(1, 3))   # [N/128][K/128]
    assert (ex.reshape(N // 128, 128, K // 128, 4).max(axis=(1, 3)) - m).max() <= 6
    scale = np.ldexp(1.0, m).astype(np.float32)
    q = val / np.kron(scale.astype(np.float64), np.ones((128, 128)))
    c8 = torch.from_numpy(q).to(torch.float8_e4m3fn)
    assert np.array_equal(c8.to(torch.float64).numpy(), q)        # exact twin
    return c8.view(torch.uint8), torch.from_numpy(scale)


def _rows_by_token(dbg):
    """(token, M-block) of every valid pool row of the last forward (padding rows left out)."""
    BM, off, counts, meta = dbg["block_m"], dbg["block_offset"], dbg["counts"], dbg["meta"]
    toks, blks = [np.zeros(0, np.int64)], [np.zeros(0, np.int64)]
    for e in range(counts.size):
        n = int(counts[e])
        if n:
            r = int(off[e]) * BM + np.arange(n)
            toks.append(meta[r, 1].astype(np.int64))
            blks.append(r // BM)
    return np.concatenate(toks), np.concatenate(blks)


def block_cover_tokens(dbg, extra=()):
    """Tokens whose routed rows, together, fall in every M-block of the pool of the last
    forward (dbg = FusedMoE.debug_routing()): every M-block of every expert, the last partly
    filled block of each and the blocks of the last wave included, holds at least one row of
    a returned token.  Greedy: for each block not yet covered, the token among its rows that
    covers the most uncovered blocks.  The `extra` tokens are part of the result (sorted)."""
    tok, blk = _rows_by_token(dbg)
    nblk = int(dbg["block_offset"][-1])
    by_tok = {}
    for t, b in zip(tok.tolist(), blk.tolist()):
        by_tok.setdefault(t, []).append(b)
    by_tok = {t: np.array(v, np.int64) for t, v in by_tok.items()}
    by_blk = {}
    for t, b in zip(tok.tolist(), blk.tolist()):
        by_blk.setdefault(b, set()).add(t)
    covered = np.zeros(nblk, bool)
    chosen = set(int(t) for t in extra)
    for t in chosen:
        if t in by_tok:
            covered[by_tok[t]] = True
    for b in range(nblk):
        if covered[b]:
            continue
        best = max(sorted(by_blk[b]), key=lambda t: int((~covered[by_tok[t]]).sum()))
        covered[by_tok[best]] = True
        chosen.add(best)
    assert covered.all()
    return np.array(sorted(chosen), np.int64)


def blocks_of_tokens(dbg, tokens):
    """M-blocks holding at least one valid row of `tokens` (to check a cover)."""
    tok, blk = _rows_by_token(dbg)
    return set(blk[np.isin(tok, np.asarray(tokens, np.int64))].tolist())
