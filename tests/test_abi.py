"""The C ABI library builds, loads, exports every entry point include/flashmask.h
declares, and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

from mask_aware_exact_gb300 import build as B
from mask_aware_exact_gb300 import flashmask as fm

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "flashmask.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return fm.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flashmask_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(fm.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(6):
        assert fm.flashmask_status_string(s)
    assert fm.flashmask_status_string(99) == "unknown status"


def test_workspace_sizes(lib):
    # classification only, then with the backward's fp32 scratch
    f = fm.flashmask_workspace_bytes(1, 32, 1, 32768, 128, False)
    b = fm.flashmask_workspace_bytes(1, 32, 1, 32768, 128, True)
    BHN = 32 * 32768
    assert b - f >= BHN * 4 * 2 + BHN * 128 * 4
    assert f >= 256 * 256 * 2  # two label tables
    for bad in [(1, 32, 1, 32768, 96), (1, 32, 3, 1024, 128), (0, 1, 1, 128, 64),
                (1, 1, 1, 0, 64), (1, 1, 1, -128, 64), (1, 1, 1, (1 << 21) + 1, 64)]:
        assert fm.flashmask_workspace_bytes(*bad, True) == 0
    # the longest supported sequence (FM_MAX_SEQLEN = 2^21) is accepted
    assert fm.flashmask_workspace_bytes(1, 1, 1, 1 << 21, 64, False) > 0
    # a sequence length that is not a multiple of 128: the tables cover
    # ceil(N / 128) blocks and the backward arrays are padded to 128 rows
    L = fm.flashmask_workspace_layout(1, 2, 1, 1000, 64, True)
    assert L.kv_part - L.dq_accum == 2 * 1024 * 64 * 4
    # split key blocks: E = min(Tc, 16) = 8 per head, three parts' fp32 dV, dK rows
    assert L.kv_sync - L.kv_part == 2 * 8 * 3 * 2 * 128 * 64 * 4
    assert L.total - L.kv_sync == 2 * 8 * 8 * 4  # 8 int32 per split block
    assert L.labels_t - L.labels >= 8 * 8


def test_workspace_layout_regions_disjoint(lib):
    L = fm.flashmask_workspace_layout(2, 8, 2, 1024, 64, True)
    offs = [L.status, L.minmax, L.labels, L.labels_t, L.row_count, L.row_list, L.row_order,
            L.col_count, L.col_list, L.col_order, L.lse2, L.delta, L.dq_accum, L.kv_part,
            L.kv_sync, L.total]
    assert offs == sorted(offs) and len(set(offs)) == len(offs)
    assert all(o % 256 == 0 for o in offs)
    Tr = 1024 // 128
    assert L.labels_t - L.labels >= 2 * 2 * Tr * Tr
    assert L.kv_part - L.dq_accum == 2 * 8 * 1024 * 64 * 4
    assert L.kv_sync - L.kv_part == 2 * 8 * 8 * 3 * 2 * 128 * 64 * 4


FAKE = 1 << 20  # a 256-aligned non-null address; validation fails before it is used


def call_fwd(lib, q=FAKE, B_=1, H=2, N=256, d=64, scale=0.125, ws=FAKE, ws_bytes=1 << 30,
             mask=None, Hm=1):
    m = mask if mask is not None else fm._FmMask(FAKE, FAKE, None, None, Hm, 1)
    return lib.flashmask_fwd(q, FAKE, FAKE, ctypes.byref(m), B_, H, N, d, scale, FAKE, FAKE, ws,
                             ws_bytes, 0, None)


def test_fwd_argument_errors(lib):
    assert call_fwd(lib, q=None) == fm.FM_ERR_INVALID_ARG
    assert call_fwd(lib, q=FAKE + 8) == fm.FM_ERR_INVALID_ARG            # misaligned
    assert call_fwd(lib, scale=float("nan")) == fm.FM_ERR_INVALID_ARG
    assert call_fwd(lib, scale=-1.0) == fm.FM_ERR_INVALID_ARG
    assert call_fwd(lib, d=96) == fm.FM_ERR_UNSUPPORTED
    assert call_fwd(lib, N=0) == fm.FM_ERR_UNSUPPORTED
    assert call_fwd(lib, H=3, Hm=2) == fm.FM_ERR_UNSUPPORTED
    assert call_fwd(lib, ws=None) == fm.FM_ERR_WORKSPACE
    assert call_fwd(lib, ws=FAKE + 16) == fm.FM_ERR_WORKSPACE
    assert call_fwd(lib, ws_bytes=100) == fm.FM_ERR_WORKSPACE
    half = fm._FmMask(FAKE, FAKE, FAKE, None, 1, 1)  # uts without ute
    assert call_fwd(lib, mask=half) == fm.FM_ERR_INVALID_ARG
    nolts = fm._FmMask(None, FAKE, None, None, 1, 1)
    assert call_fwd(lib, mask=nolts) == fm.FM_ERR_INVALID_ARG


def test_bwd_and_classify_argument_errors(lib):
    m = fm._FmMask(FAKE, FAKE, None, None, 1, 1)
    args = [FAKE] * 6
    # workspace sized for the forward only is too small for the backward
    fwd_ws = fm.flashmask_workspace_bytes(1, 2, 1, 256, 64, False)
    st = lib.flashmask_bwd(*args, ctypes.byref(m), 1, 2, 256, 64, 0.125, FAKE, FAKE, FAKE, FAKE,
                           fwd_ws, 0, None)
    assert st == fm.FM_ERR_WORKSPACE
    st = lib.flashmask_bwd(*args[:5], None, ctypes.byref(m), 1, 2, 256, 64, 0.125, FAKE, FAKE,
                           FAKE, FAKE, 1 << 30, 0, None)
    assert st == fm.FM_ERR_INVALID_ARG
    assert lib.flashmask_classify(None, 1, 256, FAKE, 1 << 30, None) == fm.FM_ERR_INVALID_ARG
    assert lib.flashmask_classify(ctypes.byref(m), 1, 0, FAKE, 1 << 30, None) == fm.FM_ERR_UNSUPPORTED
    assert lib.flashmask_classify(ctypes.byref(m), 1, 256, FAKE, 8, None) == fm.FM_ERR_WORKSPACE
    assert lib.flashmask_workspace_layout(1, 2, 1, 256, 64, 1, None) == fm.FM_ERR_INVALID_ARG
    assert lib.flashmask_check_status(None, None, None) == fm.FM_ERR_WORKSPACE


def test_selftest_argument_errors(lib):
    assert lib.flashmask_selftest_timeout(None, 256, 10_000_000, 1, None) == fm.FM_ERR_WORKSPACE
    assert lib.flashmask_selftest_timeout(FAKE, 8, 10_000_000, 1, None) == fm.FM_ERR_WORKSPACE
    assert lib.flashmask_selftest_timeout(FAKE, 256, 10, 1, None) == fm.FM_ERR_INVALID_ARG
    assert lib.flashmask_selftest_timeout(FAKE, 256, 10_000_000, 0, None) == fm.FM_ERR_INVALID_ARG
    assert lib.flashmask_selftest_timeout(FAKE, 256, 3_000_000_000, 1, None) == fm.FM_ERR_INVALID_ARG
