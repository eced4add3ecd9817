"""Effective (unmasked) FLOP accounting for the benchmark.

Work is counted only over visible (unmasked) score entries, in the
FlashAttention-family convention: per visible entry 4*d FLOPs forward (Q K^T
and P V) and 10*d backward (S recompute, dP, dV, dK, dQ), 14*d in total.

The visible count of a key column is N minus the size of the union of the
rows it masks ([0, j) when causal, [LTS, LTE), [UTS, UTE), each clamped to
[0, N]); the union of three intervals is measured by inclusion-exclusion.
"""
from __future__ import annotations

import numpy as np

FWD_PER_ENTRY = 4   # times d
BWD_PER_ENTRY = 10  # times d


def _clamp(s, e, N):
    s = np.clip(np.asarray(s, np.int64), 0, N)
    e = np.clip(np.asarray(e, np.int64), 0, N)
    e = np.maximum(e, s)  # empty when start >= end
    return s, e


def visible_per_column(N: int, lts, lte, uts, ute, causal: bool) -> np.ndarray:
    """int64 [N]: number of visible query rows of each key column (one mask head)."""
    j = np.arange(N, dtype=np.int64)
    zero = np.zeros(N, np.int64)
    iv = [_clamp(zero, j if causal else zero, N), _clamp(lts, lte, N)]
    iv.append(_clamp(zero, zero, N) if uts is None else _clamp(uts, ute, N))

    def length(s, e):
        return np.maximum(e - s, 0)

    def inter(a, b):
        return np.maximum(a[0], b[0]), np.minimum(a[1], b[1])

    A, Bv, C = iv
    union = (length(*A) + length(*Bv) + length(*C)
             - length(*inter(A, Bv)) - length(*inter(A, C)) - length(*inter(Bv, C))
             + length(*inter(inter(A, Bv), C)))
    return N - union


def visible_pairs(mask, H: int) -> int:
    """Visible (query, key) pairs summed over every (batch, head)."""
    B, Hm, N = mask.lts.shape
    total = 0
    for b in range(B):
        for hm in range(Hm):
            g = lambda a: None if a is None else a[b, hm]
            per_head = int(visible_per_column(N, g(mask.lts), g(mask.lte), g(mask.uts), g(mask.ute),
                                              mask.causal).sum())
            total += per_head * (H // Hm)
    return total


def effective_flops(mask, H: int, d: int) -> dict:
    nnz = visible_pairs(mask, H)
    return {"nnz": nnz, "fwd": FWD_PER_ENTRY * d * nnz, "bwd": BWD_PER_ENTRY * d * nnz,
            "total": (FWD_PER_ENTRY + BWD_PER_ENTRY) * d * nnz}
