"""Brute-force tile classification (test infrastructure only).

The column-wise representation lets a kernel skip work wherever the mask is
empty of visible entries ("FlashMask: Efficient and Rich Mask Extension of
FlashAttention", abstract: kernel optimisations that eliminate unnecessary
computation by exploiting mask sparsity). Over the materialised mask, each
T x T tile (query block r, key block c) gets one exact label:

  TILE_NONE    = 0   no entry of the tile is masked
  TILE_PARTIAL = 1   some entries masked, some visible
  TILE_FULL    = 2   every entry masked (the tile is skipped)

and each key block gets the min and max of each boundary vector over its
columns, in the order (min LTS, max LTS, min LTE, max LTE, min UTS, max UTS,
min UTE, max UTE). Absent upper vectors count as all zero.
"""
from __future__ import annotations

import numpy as np

from .attention import visible

TILE_NONE, TILE_PARTIAL, TILE_FULL = 0, 1, 2


def tile_labels(N: int, lts, lte, uts, ute, causal: bool, T: int = 128, row_blocks=None):
    """uint8 labels [Tr, Tc] for one mask head (rows not in ``row_blocks`` are 255)."""
    Tr = (N + T - 1) // T
    Tc = Tr
    lab = np.full((Tr, Tc), 255, dtype=np.uint8)
    for r in (range(Tr) if row_blocks is None else row_blocks):
        rows = np.arange(r * T, min((r + 1) * T, N))
        vis = visible(rows, N, lts, lte, uts, ute, causal)
        for c in range(Tc):
            blk = vis[:, c * T:(c + 1) * T]
            if blk.all():
                lab[r, c] = TILE_NONE
            elif not blk.any():
                lab[r, c] = TILE_FULL
            else:
                lab[r, c] = TILE_PARTIAL
    return lab


def key_block_minmax(N: int, lts, lte, uts, ute, T: int = 128) -> np.ndarray:
    """int32 [Tc, 8] per-key-block min/max of the four vectors."""
    Tc = (N + T - 1) // T
    zero = np.zeros(N, dtype=np.int64)
    vecs = [np.asarray(lts, np.int64), np.asarray(lte, np.int64),
            zero if uts is None else np.asarray(uts, np.int64),
            zero if ute is None else np.asarray(ute, np.int64)]
    out = np.empty((Tc, 8), dtype=np.int32)
    for c in range(Tc):
        for n, vv in enumerate(vecs):
            blk = vv[c * T:(c + 1) * T]
            out[c, 2 * n] = blk.min()
            out[c, 2 * n + 1] = blk.max()
    return out
