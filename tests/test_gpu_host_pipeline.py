"""The host-buffer pipeline against the fp64 oracle and against the device-buffer
path: every chunking gives the same O, LSE, dK, dV as the device path (the
kernels are deterministic apart from the order of the dQ reductions) and all
outputs meet the parity tolerances."""
import math

import numpy as np
import pytest
import torch

from mask_aware_exact_gb300 import workloads as W
from oracle import attention as A

from gpu_common import TOL_O, check_forward, check_grad, need_gpu, run_path, to_np

pytestmark = pytest.mark.gpu


def host_run(fm, q, k, v, do, spec, chunk, scale=None):
    B, H, N, d = q.shape
    hq, hk, hv, hdo = (x.contiguous().pin_memory() for x in (q, k, v, do))
    mask = fm.HostMask.from_spec(spec)
    ws = fm.alloc_host_workspace(B, H, mask.Hm, N, d, chunk)
    return fm.flashmask_fwd_bwd_host(hq, hk, hv, hdo, mask, ws, chunk, scale=scale)


CASES = [
    # (B, H, Hm, N, d, chunks, mask kind)
    (2, 4, 2, 384, 64, (1, 2, 4), "random"),
    (1, 6, 3, 640, 128, (2, 6), "document"),
    (1, 2, 1, 256, 64, (1, 2), "workload0"),
    (2, 4, 1, 333, 128, (2,), "random"),
    (1, 8, 1, 512, 64, (2, 4), "random"),
]


def make_spec(kind, B, Hm, N):
    if kind == "random":
        return W.random_bounds(B, Hm, N, causal=True, seed=77 + N, upper=True)
    if kind == "document":
        lengths = [200, 37, 300, 103]
        spec = W.document_bounds(B, 1, lengths)
        rep = lambda a: None if a is None else np.repeat(a, Hm, axis=1)
        return W.MaskSpec(spec.family, spec.causal, rep(spec.lts), rep(spec.lte), rep(spec.uts),
                          rep(spec.ute))
    return W.workload(0).mask


@pytest.mark.parametrize("case", range(len(CASES)))
def test_host_pipeline_matches_device_path_and_oracle(case):
    fm = need_gpu()
    B, H, Hm, N, d, chunks, kind = CASES[case]
    spec = make_spec(kind, B, Hm, N)
    q, k, v, do = W.make_qkv(B, H, N, d, seed=case)
    ref = run_path(fm, q, k, v, do, spec)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = A.forward(q, k, v, spec, scale)
    dq_ref, dk_ref, dv_ref = A.backward(q, k, v, do, spec, scale)
    for chunk in chunks:
        o, lse, dq, dk, dv = host_run(fm, q, k, v, do, spec, chunk)
        for name, got, dev in (("o", o, ref["o"]), ("lse", lse, ref["lse"]), ("dk", dk, ref["dk"]),
                               ("dv", dv, ref["dv"])):
            assert torch.equal(got, dev.cpu()), f"{name} differs from the device path, chunk {chunk}"
        assert (dq.float() - ref["dq"].float().cpu()).abs().max().item() <= TOL_O
        what = f"host pipeline chunk {chunk}"
        check_forward(to_np(o), to_np(lse), o_ref, lse_ref, what)
        check_grad("Q", to_np(dq), dq_ref, what)
        check_grad("K", to_np(dk), dk_ref, what)
        check_grad("V", to_np(dv), dv_ref, what)


def test_host_pipeline_twice_and_unpinned():
    # two calls in a row reuse the per-device streams; pageable host memory
    # is correct too (its copies just do not overlap)
    fm = need_gpu()
    B, H, N, d = 1, 4, 512, 64
    spec = W.causal_bounds(B, 1, N)
    q, k, v, do = W.make_qkv(B, H, N, d, seed=9)
    mask = fm.HostMask.from_spec(spec, pin=False)
    ws = fm.alloc_host_workspace(B, H, 1, N, d, 1)
    a = fm.flashmask_fwd_bwd_host(q, k, v, do, mask, ws, 1)
    b = fm.flashmask_fwd_bwd_host(q, k, v, do, mask, ws, 1)
    for x, y in zip(a, b):
        assert torch.allclose(x.float(), y.float(), atol=TOL_O)
    o_ref, lse_ref = A.forward(q, k, v, spec, 1 / math.sqrt(d))
    check_forward(to_np(a[0]), to_np(a[1]), o_ref, lse_ref, "unpinned")
