"""Dense masks built straight from each family's definition (test infrastructure only).

None of these reads a boundary vector: each writes visible(i, j) from what the
mask family means ("FlashMask-3", abstract: document, prefix-LM,
share-question, sliding-window and block-sparse masks). Equality with the mask
decoded from the boundary vectors pins the encoding.
"""
from __future__ import annotations

import numpy as np


def _doc_ids(lengths) -> np.ndarray:
    return np.repeat(np.arange(len(lengths)), lengths)


def _ij(N: int, rows):
    rows = np.arange(N) if rows is None else np.asarray(rows)
    return rows[:, None], np.arange(N)[None, :], rows


def causal(N: int, rows=None) -> np.ndarray:
    """Row i sees key j iff j <= i."""
    i, j, _ = _ij(N, rows)
    return j <= i


def causal_document(lengths, rows=None) -> np.ndarray:
    """Row i sees key j iff both lie in the same document and j <= i."""
    doc = _doc_ids(lengths)
    N = len(doc)
    i, j, r = _ij(N, rows)
    return (doc[r][:, None] == doc[None, :]) & (j <= i)


def bidirectional_document(lengths, rows=None) -> np.ndarray:
    """Row i sees key j iff both lie in the same document (no causal order)."""
    doc = _doc_ids(lengths)
    N = len(doc)
    _, _, r = _ij(N, rows)
    return doc[r][:, None] == doc[None, :]


def block_causal(N: int, block: int, rows=None) -> np.ndarray:
    """Row i sees key j iff j's block is not after i's block."""
    i, j, _ = _ij(N, rows)
    return (j // block) <= (i // block)


def block_sparse(N: int, block: int, runs, rows=None) -> np.ndarray:
    """Block-level visibility expanded to elements: query block r sees key
    block c iff a_c <= r <= b_c, with runs = (a, b) listed per key block."""
    a, b = (np.asarray(x) for x in runs)
    nb = len(a)
    r_blk = np.arange(nb)[:, None]
    vis_blocks = (a[None, :] <= r_blk) & (r_blk <= b[None, :])  # [query block, key block]
    dense = np.kron(vis_blocks, np.ones((block, block), bool))[:N, :N]
    return dense if rows is None else dense[np.asarray(rows)]


def share_question(q_len: int, answers, rows=None) -> np.ndarray:
    """Question rows see the question causally; an answer row sees the whole
    question before it and its own answer causally, never another answer."""
    N = q_len + int(sum(answers))
    seg = np.concatenate([np.zeros(q_len, int), 1 + _doc_ids(answers)])  # 0 = question
    i, j, r = _ij(N, rows)
    same = seg[r][:, None] == seg[None, :]
    key_is_q = (seg == 0)[None, :]
    return (j <= i) & (same | key_is_q)


def window_prefix(N: int, window: int, prefix: int, rows=None) -> np.ndarray:
    """Global bidirectional prefix plus a causal window of ``window`` keys
    (diagonal included) outside it."""
    i, j, _ = _ij(N, rows)
    prefix_key = j < prefix
    in_window = (j <= i) & (j > i - window)
    return prefix_key | in_window


def visible_pairs_window_prefix(N: int, window: int, prefix: int) -> int:
    """Visible-pair count of ``window_prefix`` from its definition, row by row
    (a closed form per row, so it also works at N = 131072)."""
    i = np.arange(N, dtype=np.int64)
    lo = np.maximum(i - window + 1, prefix)  # window keys outside the prefix
    win = np.maximum(i - lo + 1, 0)
    return int((prefix + win).sum())


def visible_pairs_document(lengths) -> int:
    """Causal document mask: each document of length L has L(L+1)/2 pairs."""
    return int(sum(L * (L + 1) // 2 for L in lengths))


def visible_pairs_share_question(q_len: int, answers) -> int:
    """Question: causal triangle; each answer of length L sees the question
    (q_len per row) plus its own causal triangle."""
    return int(q_len * (q_len + 1) // 2 + sum(L * q_len + L * (L + 1) // 2 for L in answers))
