"""The benchmark's visible-pair counter against the oracle's dense count and the
families' closed forms."""
import numpy as np
import pytest

from mask_aware_exact_gb300 import flops as F
from mask_aware_exact_gb300 import workloads as W
from oracle import masks_independent as MI
from oracle.attention import visible


@pytest.mark.parametrize("seed", range(8))
def test_random_bounds_match_dense_count(seed):
    N = 256
    spec = W.random_bounds(1, 1, N, causal=seed % 2 == 0, seed=seed, upper=seed % 3 != 0)
    g = lambda a: None if a is None else a[0, 0]
    dense = visible(np.arange(N), N, g(spec.lts), g(spec.lte), g(spec.uts), g(spec.ute), spec.causal)
    per_col = F.visible_per_column(N, g(spec.lts), g(spec.lte), g(spec.uts), g(spec.ute), spec.causal)
    assert np.array_equal(per_col, dense.sum(axis=0))


def test_workload_counts():
    w = W.workload(2)
    assert F.visible_pairs(w.mask, 1) == MI.visible_pairs_document(w.mask.params["lengths"])
    w = W.workload(3)
    p = w.mask.params
    assert F.visible_pairs(w.mask, 1) == 2 * MI.visible_pairs_share_question(p["question"], p["answers"])
    w = W.workload(4)
    assert F.visible_pairs(w.mask, 1) == MI.visible_pairs_window_prefix(w.N, 4096, 2048)
    w = W.workload(1)
    assert F.visible_pairs(w.mask, 16) == 4 * 16 * (8192 * 8193 // 2)
    f = F.effective_flops(W.workload(2).mask, 32, 128)
    assert f["total"] == 14 * 128 * f["nnz"] and f["nnz"] == 32 * 77679895
