"""Per-rank mask localisation on the GPU against the global dense mask sliced to
the rank's rows (the plain definition of the local problem: the chunk's query
rows against every key)."""
import numpy as np
import pytest

from mask_aware_exact_gb300 import workloads as W
from oracle.attention import visible

from gpu_common import need_gpu

pytestmark = pytest.mark.gpu


def dense_rows(spec, b, hm, rows):
    g = lambda a: None if a is None else a[b, hm]
    return visible(rows, spec.N, g(spec.lts), g(spec.lte), g(spec.uts), g(spec.ute), spec.causal)


def local_dense(loc, b, hm, rows, N):
    h = lambda t: None if t is None else t[b, hm].cpu().numpy()
    return visible(np.arange(rows), N, h(loc.lts), h(loc.lte), h(loc.uts), h(loc.ute), False)


SPECS = {
    "causal": lambda: W.causal_bounds(2, 1, 700),
    "document": lambda: W.document_bounds(1, 2, [150, 333, 217]),
    "window_prefix": lambda: W.window_prefix_bounds(1, 1, 1000, 300, 96),
    "share_question": lambda: W.share_question_bounds(2, 1, 256, [200, 180, 300]),
    "bidirectional_document": lambda: W.bidirectional_document_bounds(1, 1, [90, 400, 210]),
    "random_noncausal": lambda: W.random_bounds(2, 2, 640, causal=False, seed=3, upper=True),
}


@pytest.mark.parametrize("kind", sorted(SPECS))
def test_localized_chunks_match_dense_slices(kind):
    fm = need_gpu()
    spec = SPECS[kind]()
    N = spec.N
    mask = fm.DeviceMask.from_spec(spec)
    B, Hm = spec.lts.shape[:2]
    # chunks of a 4-rank assignment, dual-chunk style (rank r holds chunk r
    # and chunk 7 - r of 8), plus a ragged one
    edges = np.linspace(0, N, 9).astype(int)
    chunks = [(edges[i], edges[i + 1] - edges[i]) for i in range(8)] + [(N - 77, 77), (0, N)]
    for row0, rows in chunks:
        loc, inexact = fm.flashmask_localize(mask, B, N, int(row0), int(rows))
        assert not inexact, (kind, row0, rows)
        for b in range(B):
            for hm in range(Hm):
                want = dense_rows(spec, b, hm, np.arange(row0, row0 + rows))
                got = local_dense(loc, b, hm, rows, N)
                assert np.array_equal(got, want), (kind, row0, rows, b, hm)


def test_causal_with_detached_upper_interval_is_flagged():
    # causal, plus an upper interval starting below the diagonal part of the
    # chunk: not representable with one upper interval, so it must be flagged
    fm = need_gpu()
    N = 256
    lts = np.full((1, 1, N), N, np.int32)
    lte = lts.copy()
    uts = np.full((1, 1, N), 200, np.int32)
    ute = np.full((1, 1, N), 220, np.int32)
    spec = W.MaskSpec("detached", True, lts, lte, uts, ute)
    loc, inexact = fm.flashmask_localize(fm.DeviceMask.from_spec(spec), 1, N, 0, N)
    assert inexact
