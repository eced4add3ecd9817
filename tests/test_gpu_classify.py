"""GPU tile classification vs brute-force tile enumeration on the materialised
mask: labels and per-key-block min/max bit-exact; lists and orders valid."""
import numpy as np
import pytest

from mask_aware_exact_gb300 import workloads as W
from oracle import tiles as TL

from gpu_common import need_gpu

pytestmark = pytest.mark.gpu


def gpu_classify(fm, spec):
    mask = fm.DeviceMask.from_spec(spec)
    ws = fm.alloc_workspace(spec.B, spec.Hm, spec.Hm, spec.N, 64, for_bwd=False)
    fm.flashmask_classify(mask, spec.B, spec.N, ws)
    st, site = fm.flashmask_check_status(ws)
    assert st == fm.FM_OK, (st, site)
    return fm.read_classification(ws, spec.B, spec.Hm, spec.N)


def check_consistency(c, b, hm):
    """Lists, counts and orders are consistent with the labels (valid, complete)."""
    lab = c["labels"][b, hm]
    Tr, Tc = lab.shape
    assert np.array_equal(c["labels_t"][b, hm], lab.T)
    for r in range(Tr):
        keep = np.nonzero(lab[r] != TL.TILE_FULL)[0]
        n = c["row_count"][b, hm, r]
        assert n == len(keep)
        lst = c["row_list"][b, hm, r, :n]
        assert np.array_equal(lst >> 2, keep) and np.array_equal(lst & 3, lab[r, keep])
    for cc in range(Tc):
        keep = np.nonzero(lab[:, cc] != TL.TILE_FULL)[0]
        n = c["col_count"][b, hm, cc]
        assert n == len(keep)
        lst = c["col_list"][b, hm, cc, :n]
        assert np.array_equal(lst >> 2, keep) and np.array_equal(lst & 3, lab[keep, cc])
    for key, cnt in (("row_order", c["row_count"][b, hm]), ("col_order", c["col_count"][b, hm])):
        order = c[key][b, hm]
        assert sorted(order.tolist()) == list(range(len(order)))  # a permutation
        assert np.all(np.diff(cnt[order]) <= 0)                  # longest first


def oracle_labels(spec, b, hm, row_blocks=None):
    g = lambda a: None if a is None else a[b, hm]
    return TL.tile_labels(spec.N, g(spec.lts), g(spec.lte), g(spec.uts), g(spec.ute), spec.causal,
                          row_blocks=row_blocks)


def oracle_minmax(spec, b, hm):
    g = lambda a: None if a is None else a[b, hm]
    return TL.key_block_minmax(spec.N, g(spec.lts), g(spec.lte), g(spec.uts), g(spec.ute))


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_classify_workloads(idx):
    # every (query block, key block) label of every workload, the 128K one
    # included (1024 x 1024 tiles), against brute force over the dense mask
    fm = need_gpu()
    w = W.workload(idx)
    spec = w.mask
    c = gpu_classify(fm, spec)
    for b in range(spec.B):
        ref = oracle_labels(spec, b, 0)
        got = c["labels"][b, 0]
        assert np.array_equal(got, ref), f"labels differ ({w.name}, b={b})"
        assert np.array_equal(c["minmax"][b, 0], oracle_minmax(spec, b, 0))
        check_consistency(c, b, 0)


def test_classify_closed_form_counts():
    # causal N = 8192: Tr(Tr-1)/2 FULL, Tr PARTIAL, Tr(Tr-1)/2 NONE
    fm = need_gpu()
    c = gpu_classify(fm, W.workload(1).mask)
    lab = c["labels"][0, 0]
    Tr = lab.shape[0]
    assert (lab == TL.TILE_FULL).sum() == Tr * (Tr - 1) // 2
    assert (lab == TL.TILE_PARTIAL).sum() == Tr
    assert (lab == TL.TILE_NONE).sum() == Tr * (Tr - 1) // 2


@pytest.mark.parametrize("seed", range(6))
def test_classify_random_bounds(seed):
    # adversarial bounds: empty / reversed intervals, values at 0 and N and
    # beyond, overlapping LT / UT, several batches and mask heads
    fm = need_gpu()
    N = [256, 512, 1024, 384, 640, 128][seed]
    B, Hm = (1 + seed % 2), (1 + seed % 3)
    spec = W.random_bounds(B, Hm, N, causal=seed % 2 == 0, seed=100 + seed, upper=seed != 3)
    c = gpu_classify(fm, spec)
    for b in range(B):
        for hm in range(Hm):
            assert np.array_equal(c["labels"][b, hm], oracle_labels(spec, b, hm))
            assert np.array_equal(c["minmax"][b, hm], oracle_minmax(spec, b, hm))
            check_consistency(c, b, hm)


def test_classify_extreme_bounds():
    # int32 extremes must act as if clamped to [0, N]
    fm = need_gpu()
    N = 512
    lts = np.full((1, 1, N), np.iinfo(np.int32).min, np.int32)
    lte = np.full((1, 1, N), np.iinfo(np.int32).max, np.int32)
    lte[0, 0, ::3] = 200  # some columns masked only for rows [0, 200)
    spec = W.MaskSpec("extreme", False, lts, lte, None, None)
    c = gpu_classify(fm, spec)
    assert np.array_equal(c["labels"][0, 0], oracle_labels(spec, 0, 0))
    assert np.array_equal(c["minmax"][0, 0], oracle_minmax(spec, 0, 0))


@pytest.mark.parametrize("N,seed", [(130, 0), (300, 1), (777, 2), (1000, 3), (64, 4), (1, 5)])
def test_classify_ragged_lengths(N, seed):
    # N not a multiple of 128: the last row and key blocks are short and the
    # labels are exact over the entries that exist
    fm = need_gpu()
    B, Hm = 1 + seed % 2, 1 + seed % 3
    spec = W.random_bounds(B, Hm, N, causal=seed % 2 == 0, seed=500 + seed, upper=True)
    c = gpu_classify(fm, spec)
    Tr = (N + 127) // 128
    assert c["labels"].shape[-1] == Tr
    for b in range(B):
        for hm in range(Hm):
            assert np.array_equal(c["labels"][b, hm], oracle_labels(spec, b, hm))
            assert np.array_equal(c["minmax"][b, hm], oracle_minmax(spec, b, hm))
            check_consistency(c, b, hm)


@pytest.mark.parametrize("N,block,seed", [(4096, 128, 0), (3000, 96, 1), (2048, 64, 2)])
def test_classify_block_sparse(N, block, seed):
    # block-sparse runs (FULL tiles above and below each key block's run)
    fm = need_gpu()
    spec = W.block_sparse_bounds(2, 1, N, block, seed)
    c = gpu_classify(fm, spec)
    for b in range(2):
        assert np.array_equal(c["labels"][b, 0], oracle_labels(spec, b, 0))
        assert np.array_equal(c["minmax"][b, 0], oracle_minmax(spec, b, 0))
        check_consistency(c, b, 0)
