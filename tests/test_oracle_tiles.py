"""Pins the brute-force tile classifier: hand-worked labels, closed-form counts
and labels reduced from the independently built dense masks."""
import numpy as np
import pytest

from mask_aware_exact_gb300 import workloads as W
from oracle import masks_independent as MI
from oracle import tiles as TL


def labels_from_dense(vis, T=128):
    """Reduce a dense visibility matrix to tile labels by reshaping (a second,
    independent route to the same three-way label)."""
    N = vis.shape[0]
    t = vis.reshape(N // T, T, N // T, T)
    allv = t.all(axis=(1, 3))
    anyv = t.any(axis=(1, 3))
    return np.where(allv, TL.TILE_NONE, np.where(anyv, TL.TILE_PARTIAL, TL.TILE_FULL)).astype(np.uint8)


def head(spec):
    g = lambda a: None if a is None else a[0, 0]
    return g(spec.lts), g(spec.lte), g(spec.uts), g(spec.ute)


def test_hand_worked_causal_256():
    N = 256
    s = W.causal_bounds(1, 1, N)
    lab = TL.tile_labels(N, *head(s), True)
    assert lab.tolist() == [[TL.TILE_PARTIAL, TL.TILE_FULL], [TL.TILE_NONE, TL.TILE_PARTIAL]]


def test_hand_worked_document_256():
    # docs [163, 54, 39]: rows 128..255 see keys 0..127 only where the row is in
    # doc 0 (rows 128..162) -> tile (1,0) partial; tile (0,1) is above the diagonal
    w = W.workload(0)
    lab = TL.tile_labels(w.N, *head(w.mask), True)
    assert lab.tolist() == [[TL.TILE_PARTIAL, TL.TILE_FULL], [TL.TILE_PARTIAL, TL.TILE_PARTIAL]]


def test_causal_counts_closed_form():
    N, T = 8192, 128
    Tr = N // T
    lab = TL.tile_labels(N, *head(W.causal_bounds(1, 1, N)), True)
    assert (lab == TL.TILE_FULL).sum() == Tr * (Tr - 1) // 2
    assert (lab == TL.TILE_NONE).sum() == Tr * (Tr - 1) // 2
    assert (lab == TL.TILE_PARTIAL).sum() == Tr
    assert np.all(np.diag(lab) == TL.TILE_PARTIAL)


@pytest.mark.parametrize("idx", [0, 3])
def test_labels_match_independent_dense_reduction(idx):
    w = W.workload(idx)
    p = w.mask.params
    if w.mask.family == "document":
        vis = MI.causal_document(p["lengths"])
    else:
        vis = MI.share_question(p["question"], p["answers"])
    assert np.array_equal(TL.tile_labels(w.N, *head(w.mask), True), labels_from_dense(vis))


def test_window_prefix_reduced_labels():
    N = 4096
    spec = W.window_prefix_bounds(1, 1, N, 1024, 512)
    vis = MI.window_prefix(N, 1024, 512)
    assert np.array_equal(TL.tile_labels(N, *head(spec), False), labels_from_dense(vis))


def test_random_bounds_labels_match_dense_reduction():
    for seed in range(4):
        N = 512
        spec = W.random_bounds(1, 1, N, seed % 2 == 0, seed)
        from oracle.attention import visible
        vis = visible(np.arange(N), N, *head(spec), spec.causal)
        assert np.array_equal(TL.tile_labels(N, *head(spec), spec.causal), labels_from_dense(vis))


def test_minmax_hand_worked():
    N = 256
    lts = np.arange(N)[::-1].copy()
    lte = np.full(N, 7)
    mm = TL.key_block_minmax(N, lts, lte, None, None)
    assert mm.tolist() == [[128, 255, 7, 7, 0, 0, 0, 0], [0, 127, 7, 7, 0, 0, 0, 0]]


def test_minmax_hand_worked_upper_vectors():
    # distinct, non-trivial values in all four vectors so that every one of
    # the eight columns (min/max of LTS, LTE, UTS, UTE) has its own hand value
    N = 256
    j = np.arange(N)
    lts = 2 * j            # block 0: 0..254,   block 1: 256..510
    lte = 1000 - j         # block 0: 873..1000, block 1: 745..872
    uts = j                # block 0: 0..127,   block 1: 128..255
    ute = N - j            # block 0: 129..256, block 1: 1..128
    mm = TL.key_block_minmax(N, lts, lte, uts, ute)
    assert mm.tolist() == [[0, 254, 873, 1000, 0, 127, 129, 256],
                           [256, 510, 745, 872, 128, 255, 1, 128]]


def test_minmax_short_last_block():
    # N = 200: the second key block holds keys 128..199 only
    N = 200
    j = np.arange(N)
    mm = TL.key_block_minmax(N, j + 5, 3 * j, N - j, np.full(N, 9))
    assert mm.tolist() == [[5, 132, 0, 381, 73, 200, 9, 9],
                           [133, 204, 384, 597, 1, 72, 9, 9]]
