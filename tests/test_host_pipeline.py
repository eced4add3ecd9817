"""Host-buffer pipeline (flashmask_fwd_bwd_host): workspace sizing and the
argument checks that refuse bad calls on the host, before any CUDA call."""
import ctypes

import pytest

from mask_aware_exact_gb300 import build as BLD
from mask_aware_exact_gb300 import flashmask as fm

FAKE = 1 << 20  # a 256-aligned non-null address; validation fails before it is used


@pytest.fixture(scope="module")
def lib():
    BLD.build()
    return fm.load()


def test_host_workspace_bytes(lib):
    # three slots, each holding 8 bf16 chunk tensors plus the chunk's workspace
    n = fm.flashmask_host_workspace_bytes(1, 32, 1, 32768, 128, 4)
    chunk_tensor = 4 * 32768 * 128 * 2
    assert n >= 3 * (8 * chunk_tensor + fm.flashmask_workspace_bytes(1, 4, 1, 32768, 128, True))
    assert n < 3 * (8 * chunk_tensor + fm.flashmask_workspace_bytes(1, 4, 1, 32768, 128, True)) \
        + 3 * (5 << 20)
    # chunks must divide H and align with the mask-head groups
    assert fm.flashmask_host_workspace_bytes(1, 32, 1, 32768, 128, 5) == 0
    assert fm.flashmask_host_workspace_bytes(1, 6, 3, 1024, 64, 3) == 0   # groups of 2, chunk 3
    assert fm.flashmask_host_workspace_bytes(1, 6, 3, 1024, 64, 2) > 0
    assert fm.flashmask_host_workspace_bytes(1, 6, 3, 1024, 64, 6) > 0
    assert fm.flashmask_host_workspace_bytes(1, 6, 3, 0, 64, 2) == 0      # N
    assert fm.flashmask_host_workspace_bytes(1, 6, 3, 1000, 64, 2) > 0    # ragged N
    assert fm.flashmask_host_workspace_bytes(1, 6, 3, 1024, 96, 2) == 0   # d


def call(lib, q=FAKE, mask=None, B=1, H=4, N=256, d=64, scale=0.125, ws=FAKE, ws_bytes=1 << 40,
         chunk=2):
    m = mask if mask is not None else fm._FmMask(FAKE, FAKE, None, None, 1, 1)
    return lib.flashmask_fwd_bwd_host(q, FAKE, FAKE, FAKE, ctypes.byref(m), B, H, N, d, scale, FAKE,
                                      FAKE, FAKE, FAKE, FAKE, ws, ws_bytes, chunk, None)


def test_host_pipeline_argument_errors(lib):
    assert call(lib, q=None) == fm.FM_ERR_INVALID_ARG
    assert call(lib, scale=float("inf")) == fm.FM_ERR_INVALID_ARG
    assert call(lib, mask=fm._FmMask(FAKE, FAKE, FAKE, None, 1, 1)) == fm.FM_ERR_INVALID_ARG
    assert call(lib, chunk=3) == fm.FM_ERR_UNSUPPORTED
    assert call(lib, chunk=0) == fm.FM_ERR_UNSUPPORTED
    assert call(lib, d=80) == fm.FM_ERR_UNSUPPORTED
    assert call(lib, ws=None) == fm.FM_ERR_WORKSPACE
    assert call(lib, ws=FAKE + 64) == fm.FM_ERR_WORKSPACE
    assert call(lib, ws_bytes=1000) == fm.FM_ERR_WORKSPACE
