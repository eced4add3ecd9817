"""Per-rank mask localisation: argument checks on the host (no CUDA call)."""
import ctypes

import pytest

from mask_aware_exact_gb300 import build as BLD
from mask_aware_exact_gb300 import flashmask as fm

FAKE = 1 << 20


@pytest.fixture(scope="module")
def lib():
    BLD.build()
    return fm.load()


def call(lib, row0=0, rows=128, N=256, mask=None, out=FAKE):
    m = mask if mask is not None else fm._FmMask(FAKE, FAKE, None, None, 1, 1)
    return lib.flashmask_localize(ctypes.byref(m), 1, N, row0, rows, out, FAKE, FAKE, FAKE, None,
                                  None)


def test_localize_argument_errors(lib):
    assert call(lib, row0=-1) == fm.FM_ERR_INVALID_ARG
    assert call(lib, rows=0) == fm.FM_ERR_INVALID_ARG
    assert call(lib, row0=200, rows=100) == fm.FM_ERR_INVALID_ARG   # past N
    assert call(lib, out=None) == fm.FM_ERR_INVALID_ARG
    assert call(lib, mask=fm._FmMask(FAKE, None, None, None, 1, 1)) == fm.FM_ERR_INVALID_ARG
    assert call(lib, mask=fm._FmMask(FAKE, FAKE, None, FAKE, 1, 1)) == fm.FM_ERR_INVALID_ARG
    assert call(lib, N=0, rows=1) == fm.FM_ERR_UNSUPPORTED
