"""Failure detection on the GPU without a fault: a wait that can never complete
gives up after its time limit, the failure reaches the host through the
workspace status word, the other CTAs stop waiting as soon as they see it, and
the context stays usable for real work afterwards."""
import math
import time

import numpy as np
import pytest
import torch

from mask_aware_exact_gb300 import workloads as W
from oracle import attention as A

from gpu_common import check_forward, need_gpu, run_path, to_np

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    fm = need_gpu()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    # CTA 0 gives up after 20 ms; 63 others wait with the library's 2 s limit
    # and must leave as soon as CTA 0's failure is in the status word
    fm.flashmask_selftest_timeout(ws, 20_000_000, ctas=64)
    st, site = fm.flashmask_check_status(ws)
    elapsed = time.perf_counter() - t0
    assert st == fm.FM_ERR_TIMEOUT and site == 301, (st, site)
    assert 0.015 < elapsed < 1.0, elapsed
    # the status word was cleared by the read
    assert fm.flashmask_check_status(ws) == (fm.FM_OK, 0)
    # the context is still good: a full forward and backward on the small workload
    w = W.workload(0)
    q, k, v, do = W.make_qkv(w.B, w.H, w.N, w.d, w.seed)
    out = run_path(fm, q, k, v, do, w.mask)
    o_ref, lse_ref = A.forward(q, k, v, w.mask, 1 / math.sqrt(w.d))
    check_forward(to_np(out["o"]), to_np(out["lse"]), o_ref, lse_ref, "after self-test")


def test_uninitialised_status_word_is_reported_and_cleared():
    # A workspace that was not allocated zeroed: the documented way to make it
    # usable is one flashmask_check_status(), which reports what the status
    # word held (as a timeout with that detail) and clears it. No kernel runs
    # on the poisoned word.
    fm = need_gpu()
    w = W.workload(0)
    ws = torch.empty(fm.flashmask_workspace_bytes(w.B, w.H, 1, w.N, w.d, True),
                     dtype=torch.uint8, device="cuda")
    ws[:16].copy_(torch.tensor(np.array([0x7f, 0x12345, 0, 0], np.int32).view(np.uint8)))
    st, site = fm.flashmask_check_status(ws)
    assert (st, site) == (fm.FM_ERR_TIMEOUT, 0x12345)
    assert fm.flashmask_check_status(ws) == (fm.FM_OK, 0)
    q, k, v, do = W.make_qkv(w.B, w.H, w.N, w.d, w.seed)
    mask = fm.DeviceMask.from_spec(w.mask)
    o, lse = fm.flashmask_fwd(q.cuda(), k.cuda(), v.cuda(), mask, ws)
    assert fm.flashmask_check_status(ws) == (fm.FM_OK, 0)
    o_ref, lse_ref = A.forward(q, k, v, w.mask, 1 / math.sqrt(w.d))
    check_forward(to_np(o), to_np(lse), o_ref, lse_ref, "after clearing")
