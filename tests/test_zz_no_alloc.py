"""The allocation-free forward (flashmask_fwd_noalloc) against the workspace
forward (flashmask_fwd): same inputs, outputs equal within the parity
tolerances, on two calls in a row that reuse the library's fixed scratch; the
first call is also compared with the fp64 oracle directly.

The file name sorts last so that the GPU test also runs after every other test
of the suite, when the scratch and the CUDA context have seen other work."""
import ctypes

import numpy as np
import pytest
import torch

from mask_aware_exact_gb300 import build as BLD
from mask_aware_exact_gb300 import flashmask as fm
from mask_aware_exact_gb300 import workloads as W

from gpu_common import TOL_LSE, TOL_O, check_forward, need_gpu, to_np

FAKE = 1 << 20  # a 256-aligned non-null address; validation fails before it is used


def call_noalloc(lib, q, k, v, m, B, H, N, d, scale, o, lse, stream):
    return lib.flashmask_fwd_noalloc(q, k, v, ctypes.byref(m), B, H, N, d, scale, o, lse, stream)


def test_noalloc_rejects_on_host():
    # shapes whose tables exceed the fixed scratch, and bad arguments, are
    # refused before any CUDA call (this runs without a GPU)
    BLD.build()
    lib = fm.load()
    m = fm._FmMask(FAKE, FAKE, None, None, 1, 1)
    big = fm.flashmask_workspace_bytes(2, 8, 1, 131072, 128, False)
    assert big > lib_scratch_bytes()
    assert call_noalloc(lib, FAKE, FAKE, FAKE, m, 2, 8, 131072, 128, 0.1, FAKE, FAKE,
                        None) == fm.FM_ERR_WORKSPACE
    assert call_noalloc(lib, None, FAKE, FAKE, m, 1, 2, 256, 64, 0.1, FAKE, FAKE,
                        None) == fm.FM_ERR_INVALID_ARG
    assert call_noalloc(lib, FAKE + 8, FAKE, FAKE, m, 1, 2, 256, 64, 0.1, FAKE, FAKE,
                        None) == fm.FM_ERR_INVALID_ARG
    assert call_noalloc(lib, FAKE, FAKE, FAKE, m, 1, 2, 256, 96, 0.1, FAKE, FAKE,
                        None) == fm.FM_ERR_UNSUPPORTED
    # the largest single-sequence shape of the 128K window workload fits
    assert fm.flashmask_workspace_bytes(1, 8, 1, 131072, 128, False) <= lib_scratch_bytes()


def lib_scratch_bytes():
    # FM_NOALLOC_SCRATCH_BYTES as include/flashmask.h defines it
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                       "flashmask.h")
    mo = re.search(r"#define\s+FM_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", open(hdr).read())
    return int(mo.group(1)) << int(mo.group(2))


def workspace_forward(q, k, v, mask):
    B, H, N, d = q.shape
    ws = fm.alloc_workspace(B, H, mask.Hm, N, d, for_bwd=False)
    o, lse = fm.flashmask_fwd(q, k, v, mask, ws)
    st, site = fm.flashmask_check_status(ws)
    assert st == fm.FM_OK, (st, site)
    return to_np(o), to_np(lse)


def noalloc_forward(lib, q, k, v, mask):
    B, H, N, d = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    m = mask.c_struct()
    st = call_noalloc(lib, q.data_ptr(), k.data_ptr(), v.data_ptr(), m, B, H, N, d, d ** -0.5,
                      o.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == fm.FM_OK, fm.flashmask_status_string(st)
    torch.cuda.synchronize()
    return to_np(o), to_np(lse)


def assert_close(got, ref, what):
    o, lse = got
    o_ref, lse_ref = ref
    assert np.abs(o - o_ref).max() <= TOL_O, what
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), what
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref)), what
    if fin.any():
        assert np.abs(lse[fin] - lse_ref[fin]).max() <= TOL_LSE, what


CASES = [
    # (mask, B, H, N, d, seed): a ragged document mask with d = 128, then two
    # mask heads with upper intervals and fully masked rows at d = 64, so the
    # second shape reuses scratch left by the first
    ("document", 1, 4, 768, 128, 1),
    ("random", 2, 4, 640, 64, 2),
]


def make_case(kind, B, H, N, d, seed):
    if kind == "document":
        spec = W.document_bounds(B, 1, [300, 129, 211, 128])
    else:
        spec = W.random_bounds(B, 2, N, causal=True, seed=40 + seed, upper=True)
    q, k, v, _ = W.make_qkv(B, H, N, d, seed)
    return spec, q, k, v


@pytest.mark.gpu
def test_noalloc_matches_workspace_forward_twice():
    need_gpu()
    lib = fm.load()
    from oracle import attention as A
    for case in CASES:
        spec, q_h, k_h, v_h = make_case(*case)
        q, k, v = q_h.cuda(), k_h.cuda(), v_h.cuda()
        mask = fm.DeviceMask.from_spec(spec)
        ref = workspace_forward(q, k, v, mask)
        first = noalloc_forward(lib, q, k, v, mask)
        second = noalloc_forward(lib, q, k, v, mask)
        assert_close(first, ref, f"{case} first call")
        assert_close(second, ref, f"{case} second call")
        # and the first call straight against the fp64 oracle
        o_ref, lse_ref = A.forward(q_h, k_h, v_h, spec, q.shape[-1] ** -0.5)
        check_forward(first[0], first[1], o_ref, lse_ref, f"{case} vs oracle")
