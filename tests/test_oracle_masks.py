"""Pins the mask decoding (boundary vectors -> dense mask) against dense masks
written straight from each family's definition."""
import numpy as np
import pytest

from mask_aware_exact_gb300 import workloads as W
from oracle import masks_independent as MI
from oracle.attention import visible


def decoded(spec, rows, b=0, hm=0):
    g = lambda a: None if a is None else a[b, hm]
    return visible(rows, spec.N, g(spec.lts), g(spec.lte), g(spec.uts), g(spec.ute), spec.causal)


def compare_blocked(spec, indep, block=1024, rows_iter=None):
    N = spec.N
    for s in (rows_iter if rows_iter is not None else range(0, N, block)):
        rows = np.arange(s, min(s + block, N))
        assert np.array_equal(decoded(spec, rows), indep(rows)), f"rows {s}.."


def test_workload_recipes_match_stated_lengths():
    # Lengths the recipes produce with seed 0 (document cuts, uniform lengths, answers).
    assert W.workload(0).mask.params["lengths"] == [163, 54, 39]
    assert W.workload(2).mask.params["lengths"] == [7045, 5404, 4438, 2584, 2876, 826, 1089,
                                                     638, 1858, 6010]
    assert W.workload(3).mask.params["answers"] == [6281, 1545, 2624, 1838]
    assert sum(W.workload(2).mask.params["lengths"]) == 32768
    assert min(W.workload(2).mask.params["lengths"][:-1]) >= 512


def test_document_small():
    w = W.workload(0)
    compare_blocked(w.mask, lambda r: MI.causal_document(w.mask.params["lengths"], r))


def test_causal():
    w = W.workload(1)
    compare_blocked(w.mask, lambda r: MI.causal(w.N, r))


def test_causal_literal_visible_interval_reading():
    # The workload text describes plain causal as "LTS = column index, LTE = N";
    # read as the VISIBLE rows [j, N) of column j, that is the causal mask this
    # encoding (causal flag, empty intervals) decodes to.
    N = 512
    spec = W.causal_bounds(1, 1, N)
    j = np.arange(N)
    lit_start, lit_end = j, np.full(N, N)
    i = np.arange(N)[:, None]
    literal_visible = (lit_start[None, :] <= i) & (i < lit_end[None, :])
    assert np.array_equal(decoded(spec, np.arange(N)), literal_visible)


def test_document_large():
    w = W.workload(2)
    compare_blocked(w.mask, lambda r: MI.causal_document(w.mask.params["lengths"], r),
                    block=512, rows_iter=range(0, w.N, 4096))


def test_share_question():
    w = W.workload(3)
    p = w.mask.params
    compare_blocked(w.mask, lambda r: MI.share_question(p["question"], p["answers"], r),
                    block=512, rows_iter=range(0, w.N, 2048))
    # every answer row sees the whole question, never an earlier answer
    qa = MI.share_question(p["question"], p["answers"], np.array([p["question"] + p["answers"][0]]))
    assert qa[0, :p["question"]].all() and not qa[0, p["question"] + p["answers"][0] + 1:].any()


def test_window_prefix_reduced_full():
    # same family at N = 16384 compared in full
    spec = W.window_prefix_bounds(1, 1, 16384, 4096, 2048)
    compare_blocked(spec, lambda r: MI.window_prefix(16384, 4096, 2048, r), block=1024)


def test_window_prefix_full_size_sampled():
    w = W.workload(4)
    rows_iter = [0, 1024, 2048 - 256, 2048, 4096, 6143, 65536, w.N - 512]
    compare_blocked(w.mask, lambda r: MI.window_prefix(w.N, 4096, 2048, r), block=256,
                    rows_iter=rows_iter)
    # 4096 window keys (diagonal included) plus the 2048-token prefix per late row
    row = decoded(w.mask, np.array([100000]))[0]
    assert row.sum() == 4096 + 2048


@pytest.mark.parametrize("idx,expected", [(0, 15631), (2, 77679895), (3, 84779251)])
def test_visible_pair_counts_closed_form(idx, expected):
    w = W.workload(idx)
    p = w.mask.params
    if w.mask.family == "document":
        assert MI.visible_pairs_document(p["lengths"]) == expected
    else:
        assert MI.visible_pairs_share_question(p["question"], p["answers"]) == expected


def test_visible_pairs_window_prefix_closed_form():
    # the per-row closed form agrees with a dense count on a reduced instance ...
    N = 8192
    assert MI.visible_pairs_window_prefix(N, 1024, 512) == int(MI.window_prefix(N, 1024, 512).sum())
    # ... and gives the full-size count
    assert MI.visible_pairs_window_prefix(131072, 4096, 2048) == 788531200


def test_decoded_count_matches_closed_form_small():
    from oracle.attention import visible_count
    w = W.workload(0)
    m = w.mask
    assert visible_count(w.N, m.lts[0, 0], m.lte[0, 0], None, None, True) == 15631


@pytest.mark.parametrize("lengths", [[5, 7, 1, 20], [100, 28], [300, 37, 129, 1]])
def test_bidirectional_document(lengths):
    spec = W.bidirectional_document_bounds(1, 1, lengths)
    compare_blocked(spec, lambda r: MI.bidirectional_document(lengths, r), block=64)


@pytest.mark.parametrize("N,block", [(256, 128), (333, 128), (200, 64), (100, 7)])
def test_block_causal(N, block):
    spec = W.block_causal_bounds(1, 1, N, block)
    compare_blocked(spec, lambda r: MI.block_causal(N, block, r), block=64)


def test_stack_heads_decodes_each_head():
    # per-head masks: head hm of the stack decodes to the hm-th family's mask
    N = 200
    parts = [W.document_bounds(1, 1, [120, 80]), W.causal_bounds(1, 1, N)]
    spec = W.stack_heads(parts)
    rows = np.arange(N)
    assert np.array_equal(decoded(spec, rows, hm=0), MI.causal_document([120, 80], rows))
    assert np.array_equal(decoded(spec, rows, hm=1), MI.causal(N, rows))


@pytest.mark.parametrize("N,block,seed", [(640, 64, 0), (1024, 128, 1), (700, 96, 2),
                                          (300, 128, 3)])
def test_block_sparse(N, block, seed):
    spec = W.block_sparse_bounds(1, 1, N, block, seed)
    runs = spec.params["runs"]
    compare_blocked(spec, lambda r: MI.block_sparse(N, block, runs, r), block=128)
    # the runs themselves: each contains its diagonal block; block 0 is global
    a, b = runs
    assert a[0] == 0 and b[0] == len(a) - 1
    assert all(a[c] <= c <= b[c] for c in range(len(a)))
    # the pattern is not a plain causal / banded one: some key block is hidden
    # from some query block above and below its run
    assert any(x > 0 for x in a[1:]) and any(y < len(a) - 1 for y in b[1:])
