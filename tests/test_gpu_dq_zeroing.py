"""The dQ accumulator's life cycle. The forward zeroes it when its workspace is
sized for the backward, and the backward preprocess of the same shape then
skips that pass. The cases fill the accumulator (and dQ) with NaN first, so a
zeroing or a write that nobody did shows up as NaN or a wrong dQ; dQ, dK and
dV are compared with the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

from mask_aware_exact_gb300 import workloads as W
from oracle import attention as A

from gpu_common import check_grad, need_gpu, to_np

pytestmark = pytest.mark.gpu

B, H, N, D = 1, 2, 1000, 128  # ragged: 8 query blocks, the last one short


def _setup(fm, seed=3):
    spec = W.document_bounds(B, 1, [300, 450, 250])
    q, k, v, do = W.make_qkv(B, H, N, D, seed=seed)
    dev = [x.cuda() for x in (q, k, v, do)]
    mask = fm.DeviceMask.from_spec(spec)
    return spec, (q, k, v, do), dev, mask


def _poison_accumulator(fm, ws, Hm):
    lay = fm.flashmask_workspace_layout(B, H, Hm, N, D, True)
    npad = -(-N // 128) * 128
    n = B * H * npad * D * 4
    ws[lay.dq_accum:lay.dq_accum + n].view(torch.float32).fill_(float("nan"))


def _status_tag(ws):
    return int(ws[:16].view(torch.int32)[3].item())


def _backward(fm, dev, o, lse, mask, ws):
    qd, kd, vd, dod = dev
    dq = torch.full_like(qd, float("nan"))
    dk, dv = (torch.empty_like(qd) for _ in range(2))
    fm.flashmask_bwd_preprocess(o, lse, dod, mask.Hm, ws)
    fm.flashmask_bwd_main(qd, kd, vd, dod, mask, ws, dk, dv)
    fm.flashmask_bwd_finalize(dq, mask.Hm, ws)
    return dq, dk, dv


def _check(host, spec, grads, what):
    q, k, v, do = host
    ref = A.backward(q, k, v, do, spec, 1 / math.sqrt(D))
    for name, g, r in zip("QKV", grads, ref):
        x = to_np(g)
        assert np.isfinite(x).all(), f"{what}: d{name} not finite"
        check_grad(name, x, r, what)


def test_forward_zeroes_accumulator_for_the_backward():
    fm = need_gpu()
    spec, host, dev, mask = _setup(fm)
    qd, kd, vd, _ = dev
    ws = fm.alloc_workspace(B, H, mask.Hm, N, D, for_bwd=True)
    fm.flashmask_classify(mask, B, N, ws)
    _poison_accumulator(fm, ws, mask.Hm)
    o, lse = fm.flashmask_fwd(qd, kd, vd, mask, ws, ws_classified=True)
    torch.cuda.synchronize()
    assert _status_tag(ws) != 0, "the forward leaves its tag"
    lay = fm.flashmask_workspace_layout(B, H, mask.Hm, N, D, True)
    npad = -(-N // 128) * 128
    acc = ws[lay.dq_accum:lay.dq_accum + B * H * npad * D * 4].view(torch.float32)
    assert bool((acc == 0).all()), "every accumulator row is zeroed by the forward"
    grads = _backward(fm, dev, o, lse, mask, ws)
    _check(host, spec, grads, "forward-zeroed accumulator")
    torch.cuda.synchronize()
    assert _status_tag(ws) == 0, "the backward main kernel clears the tag"
    st, site = fm.flashmask_check_status(ws)
    assert st == fm.FM_OK, (st, site)


def test_second_backward_zeroes_again():
    # two backward passes after one forward: the second preprocess must zero
    fm = need_gpu()
    spec, host, dev, mask = _setup(fm, seed=4)
    qd, kd, vd, _ = dev
    ws = fm.alloc_workspace(B, H, mask.Hm, N, D, for_bwd=True)
    o, lse = fm.flashmask_fwd(qd, kd, vd, mask, ws)
    first = _backward(fm, dev, o, lse, mask, ws)
    second = _backward(fm, dev, o, lse, mask, ws)
    _check(host, spec, second, "second backward")
    d = (second[0].float() - first[0].float()).abs().max().item()
    assert d <= 1e-2 * first[0].float().abs().max().item()


def test_forward_only_workspace_leaves_zeroing_to_the_preprocess():
    # forward with its own forward-sized workspace, backward with another one
    # whose accumulator holds NaN: the tag does not match, so it is zeroed
    fm = need_gpu()
    spec, host, dev, mask = _setup(fm, seed=5)
    qd, kd, vd, _ = dev
    ws_f = fm.alloc_workspace(B, H, mask.Hm, N, D, for_bwd=False)
    o, lse = fm.flashmask_fwd(qd, kd, vd, mask, ws_f)
    torch.cuda.synchronize()
    assert _status_tag(ws_f) == 0
    ws_b = fm.alloc_workspace(B, H, mask.Hm, N, D, for_bwd=True)
    fm.flashmask_classify(mask, B, N, ws_b)
    _poison_accumulator(fm, ws_b, mask.Hm)
    grads = _backward(fm, dev, o, lse, mask, ws_b)
    _check(host, spec, grads, "separate backward workspace")


def test_fp8_forward_clears_the_tag():
    # the FP8 operands overlap a backward layout's accumulator: after an FP8
    # forward on the same workspace the preprocess must zero it again
    fm = need_gpu()
    spec, host, dev, mask = _setup(fm, seed=6)
    qd, kd, vd, _ = dev
    nbytes = max(fm.flashmask_workspace_bytes(B, H, mask.Hm, N, D, True),
                 fm.flashmask_fwd_fp8_workspace_bytes(B, H, mask.Hm, N))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    o, lse = fm.flashmask_fwd(qd, kd, vd, mask, ws)
    torch.cuda.synchronize()
    assert _status_tag(ws) != 0
    fm.flashmask_fwd_fp8(qd, kd, vd, mask, ws)
    torch.cuda.synchronize()
    assert _status_tag(ws) == 0
    _poison_accumulator(fm, ws, mask.Hm)
    grads = _backward(fm, dev, o, lse, mask, ws)
    _check(host, spec, grads, "after an FP8 forward")


def test_unseen_query_blocks_get_zero_dq():
    # rows [256, 512) see no key at all: their query blocks (2 and 3) have no
    # non-FULL tile, and their dQ must still come out exactly 0
    fm = need_gpu()
    lts = np.full((B, 1, N), 256, np.int32)
    lte = np.full((B, 1, N), 512, np.int32)
    spec = W.MaskSpec("causal_hole", True, lts, lte, None, None)
    q, k, v, do = W.make_qkv(B, H, N, D, seed=8)
    dev = [x.cuda() for x in (q, k, v, do)]
    mask = fm.DeviceMask.from_spec(spec)
    ws = fm.alloc_workspace(B, H, mask.Hm, N, D, for_bwd=True)
    o, lse = fm.flashmask_fwd(dev[0], dev[1], dev[2], mask, ws)
    grads = _backward(fm, dev, o, lse, mask, ws)
    dq = to_np(grads[0])
    assert np.all(dq[:, :, 256:512] == 0)
    _check((q, k, v, do), spec, grads, "query blocks without visible keys")
