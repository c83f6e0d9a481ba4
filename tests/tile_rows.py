"""Rows (tokens) that full-size parity tests compare against the oracle.

The prefill GEMMs tile the tokens in 128-row tiles; the CTA-pair engine runs
tiles 2p and 2p + 1 together, the even one in the CTA that issues the MMAs and
the odd one in its peer. A bug tied to one tile, one CTA of a pair or the rows
past a pair's first tile shows only in rows of that tile, so the samples here
take rows from EVERY tile: its first and last row and seeded rows between them.
Rows are independent through the MLP block and the projections, so the
oracle evaluates only the sampled rows.
"""
from __future__ import annotations

import numpy as np


def tile_rows(T: int, per_tile: int = 4, seed: int = 0, tile: int = 128) -> np.ndarray:
    """Sorted unique rows: the first and last row of every `tile`-row tile of a
    T-row batch (the last, partial tile included) and per_tile - 2 seeded rows
    strictly inside each tile."""
    rng = np.random.default_rng(seed)
    out = []
    for lo in range(0, T, tile):
        hi = min(T, lo + tile)
        out += [lo, hi - 1]
        inner = np.arange(lo + 1, hi - 1)
        k = min(max(per_tile - 2, 0), inner.size)
        if k:
            out += rng.choice(inner, k, replace=False).tolist()
    return np.unique(np.asarray(out, dtype=np.int64))


def moe_tile_tokens(expert_ids: np.ndarray, per_tile: int = 2, tile: int = 128, seed: int = 0) -> np.ndarray:
    """Tokens whose routed rows fall in every 128-row tile of the grouped expert GEMMs.

    The block sorts the routed (token, slot) entries by expert, keeping entry order
    (token * k + slot) within an expert, and starts each expert's rows on a tile
    boundary; the entries of tile c of expert e are that expert's entries
    [128 c, 128 c + 128). Takes the first and last entry of each such tile and
    per_tile - 2 seeded ones between them, and returns their tokens."""
    rng = np.random.default_rng(seed)
    ids = np.asarray(expert_ids)
    k = ids.shape[1]
    flat = ids.reshape(-1)
    toks = []
    for e in np.unique(flat):
        ent = np.nonzero(flat == e)[0]
        for lo in range(0, ent.size, tile):
            chunk = ent[lo:lo + tile]
            pick = [chunk[0], chunk[-1]]
            if chunk.size > 2 and per_tile > 2:
                pick += rng.choice(chunk[1:-1], min(per_tile - 2, chunk.size - 2), replace=False).tolist()
            toks += [int(p) // k for p in pick]
    return np.unique(np.asarray(toks, dtype=np.int64))
