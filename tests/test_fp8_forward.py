"""The FP8 (e4m3) forward against the oracle.

Three checks, from the tightest down:
  1. the quantised operands the call leaves in its workspace (e4m3 codes of Q,
     K and V^T, fp32 scales) equal oracle.fp8's element by element;
  2. with the oracle run on those dequantised operands, LSE agrees to the bf16
     path's tolerance (it carries no P rounding) and every element of O stays
     within the bound of rounding c P to e4m3 (c = 28, the scale the FP8
     forward applies to P; relative step 2^-4): for row i
     |O_i - O'_i| <= (2^-4 + 2^-9) (P'|V'|)_i + 2^-10 / c (vis|V'|)_i
     + 2^-8 |O'_i| + 1e-5, where primes mark the oracle on dequantised
     operands; the terms are P's rounding, P's e4m3 subnormal floor (absolute
     2^-10 / c), bf16 output rounding, and 2^-9 for fp32-level error of the
     tensor-core sums;
  3. against the exact oracle on the original bf16 inputs O's relative
     Frobenius error stays below 0.1: the three roundings (Q K^T inputs, P, V)
     each contribute about 2^-4 / sqrt(3) ~ 0.036 RMS relative error.
Fully masked rows keep the exact convention (O = 0, LSE = -inf).
The argument checks run without a GPU."""
import ctypes
import math

import numpy as np
import pytest
import torch

from mask_aware_exact_gb300 import flashmask as fm
from mask_aware_exact_gb300 import workloads as W
from oracle import attention as A
from oracle import fp8 as F

from gpu_common import TOL_LSE, head_bounds, need_gpu, rel_fro, to_np

FAKE = 1 << 20  # a 256-aligned non-null address; validation fails before it is used
TOL_FP8_REL = 0.1
P_SCALE = 28.0  # the FP8 forward rounds P * 28 to e4m3 (include/flashmask.h)
TABLE = F.e4m3_table()


@pytest.fixture(scope="module")
def lib():
    from mask_aware_exact_gb300 import build
    build.build()
    return fm.load()


def call(lib, q=FAKE, d=128, N=256, ws=FAKE, ws_bytes=1 << 30, mask=None, scale=0.125):
    m = mask if mask is not None else fm._FmMask(FAKE, FAKE, None, None, 1, 1)
    return lib.flashmask_fwd_fp8(q, FAKE, FAKE, ctypes.byref(m), 1, 2, N, d, scale, FAKE, FAKE,
                                 ws, ws_bytes, 0, None)


def test_fp8_argument_errors(lib):
    assert call(lib, d=64) == fm.FM_ERR_UNSUPPORTED
    assert call(lib, N=0) == fm.FM_ERR_UNSUPPORTED
    assert call(lib, q=None) == fm.FM_ERR_INVALID_ARG
    assert call(lib, q=FAKE + 8) == fm.FM_ERR_INVALID_ARG
    assert call(lib, scale=float("nan")) == fm.FM_ERR_INVALID_ARG
    assert call(lib, ws=FAKE + 16) == fm.FM_ERR_WORKSPACE
    need = fm.flashmask_fwd_fp8_workspace_bytes(1, 2, 1, 256)
    assert call(lib, ws_bytes=need - 1) == fm.FM_ERR_WORKSPACE
    assert fm.flashmask_fwd_fp8_workspace_bytes(1, 2, 1, 0) == 0
    assert fm.flashmask_fwd_fp8_workspace_bytes(1, 3, 2, 256) == 0  # H % Hm != 0


@pytest.mark.parametrize("B,H,Hm,N", [(1, 2, 1, 256), (2, 4, 2, 333), (1, 32, 1, 32768)])
def test_fp8_layout(lib, B, H, Hm, N):
    L = fm.flashmask_fwd_fp8_layout(B, H, Hm, N)
    Tr = (N + 127) // 128
    assert L.fwd_total == fm.flashmask_workspace_bytes(B, H, Hm, N, 128, False)
    regions = [(L.q8, B * H * N * 128), (L.k8, B * H * N * 128), (L.vt8, B * H * 128 * 128 * Tr),
               (L.qscale, B * H * Tr * 4), (L.kscale, B * H * Tr * 4), (L.vscale, B * H * 4)]
    end = L.fwd_total
    for off, n in regions:
        assert off % 256 == 0 and off >= end
        end = off + n
    assert L.total >= end and L.total == fm.flashmask_fwd_fp8_workspace_bytes(B, H, Hm, N)


def run_fp8(q, k, v, spec):
    B, H, N, d = q.shape
    mask = fm.DeviceMask.from_spec(spec)
    ws = fm.alloc_fp8_workspace(B, H, mask.Hm, N)
    o, lse = fm.flashmask_fwd_fp8(q.cuda(), k.cuda(), v.cuda(), mask, ws)
    st, site = fm.flashmask_check_status(ws)
    assert st == fm.FM_OK, f"device status {st} at site {site}"
    return o, lse, fm.read_fp8_operands(ws, B, H, mask.Hm, N)


def check_operands(ops, q, k, v, heads):
    q8, k8, vt8, qs, ks, vs = (x.cpu().numpy() for x in ops)
    N = q.shape[2]
    out = {}
    for (b, h) in heads:
        cq, sq, dq_ = F.quantize_rows(q[b, h].float().numpy())
        ck, sk, dk_ = F.quantize_rows(k[b, h].float().numpy())
        cv, sv, dv_ = F.quantize_head(v[b, h].float().numpy())
        assert np.array_equal(qs[b, h], sq), (b, h)
        assert np.array_equal(ks[b, h], sk), (b, h)
        assert vs[b, h] == sv, (b, h)
        assert np.array_equal(TABLE[q8[b, h]], cq), (b, h)
        assert np.array_equal(TABLE[k8[b, h]], ck), (b, h)
        vt = TABLE[vt8[b, h]]
        assert np.array_equal(vt[:, :N], cv.T), (b, h)
        assert np.all(vt[:, N:] == 0), (b, h)
        out[(b, h)] = (dq_, dk_, dv_)
    return out


def check_outputs(o, lse, q, k, v, spec, deq, rows=None, what=""):
    H = q.shape[1]
    N, d = q.shape[2], q.shape[3]
    scale = 1 / math.sqrt(d)
    errs = []
    for (b, h), (dq_, dk_, dv_) in deq.items():
        lts, lte, uts, ute = head_bounds(spec, b, h, H)
        r = np.arange(N) if rows is None else rows
        og, lg = to_np(o[b, h])[r], to_np(lse[b, h])[r]
        o_q, lse_q = A.forward_head(dq_, dk_, dv_, lts, lte, uts, ute, spec.causal, scale, rows=r)
        pv_abs, _ = A.forward_head(dq_, dk_, np.abs(dv_), lts, lte, uts, ute, spec.causal, scale,
                                   rows=r)
        vis_abs = A.visible(r, N, lts, lte, uts, ute, spec.causal).astype(np.float64) @ np.abs(dv_)
        fin = np.isfinite(lse_q)
        assert np.all(np.isneginf(lg[~fin])) and np.all(og[~fin] == 0), what
        assert np.array_equal(np.isfinite(lg), fin), what
        if fin.any():
            e_l = np.abs(lg[fin] - lse_q[fin]).max()
            assert e_l <= TOL_LSE, f"{what} {(b, h)} max|LSE - LSE'| = {e_l}"
        bound = ((2.0 ** -4 + 2.0 ** -9) * pv_abs + 2.0 ** -10 / P_SCALE * vis_abs
                 + 2.0 ** -8 * np.abs(o_q) + 1e-5)
        excess = np.abs(og - o_q) - bound
        assert excess.max() <= 0, f"{what} {(b, h)} O outside the P-rounding bound by {excess.max()}"
        o_ref, _ = A.forward_head(q[b, h], k[b, h], v[b, h], lts, lte, uts, ute, spec.causal,
                                  scale, rows=r)
        e = rel_fro(og, o_ref)
        errs.append(e)
        assert e <= TOL_FP8_REL, f"{what} {(b, h)} rel_fro(O - O_exact) = {e}"
    return errs


CASES = {
    "causal": lambda B, N: W.causal_bounds(B, 1, N),
    "document": lambda B, N: W.document_bounds(B, 1, [N // 3, 77, N - N // 3 - 77]),
    "random_upper": lambda B, N: W.random_bounds(B, 2, N, causal=False, seed=91, upper=True),
    "share_question": lambda B, N: W.share_question_bounds(
        B, 1, N // 4, [N // 4, N // 8, N - N // 4 - N // 4 - N // 8]),
}


@pytest.mark.gpu
@pytest.mark.parametrize("N", [640, 333])
@pytest.mark.parametrize("kind", list(CASES))
def test_fp8_forward_small(kind, N):
    need_gpu()
    B, H = 2, 2
    spec = CASES[kind](B, N)
    q, k, v, _ = W.make_qkv(B, H, N, 128, seed=11)
    o, lse, ops = run_fp8(q, k, v, spec)
    heads = [(b, h) for b in range(B) for h in range(H)]
    deq = check_operands(ops, q, k, v, heads)
    errs = check_outputs(o, lse, q, k, v, spec, deq, what=f"{kind} N={N}")
    print(f"fp8 {kind} N={N}: rel_fro(O - O_exact) max {max(errs):.4f}")


@pytest.mark.gpu
def test_fp8_scaled_inputs_and_outliers():
    # large and tiny magnitudes per block and a few outliers: the block scales
    # keep every block's largest element at 448
    need_gpu()
    B, H, N = 1, 2, 512
    q, k, v, _ = W.make_qkv(B, H, N, 128, seed=5)
    q = (q.float() * 20.0).to(torch.bfloat16)
    k = (k.float() * 0.01).to(torch.bfloat16)
    k[0, 0, 300, 7] = 3.0
    v[0, 1, 5, 100] = 40.0
    spec = W.causal_bounds(B, 1, N)
    o, lse, ops = run_fp8(q, k, v, spec)
    deq = check_operands(ops, q, k, v, [(0, 0), (0, 1)])
    check_outputs(o, lse, q, k, v, spec, deq, what="scaled")


@pytest.mark.gpu
def test_fp8_full_size_document_sampled():
    # the 32K document workload in full, sampled query rows checked
    need_gpu()
    w = W.workload(2)
    q, k, v, _ = W.make_qkv(w.B, w.H, w.N, w.d, w.seed)
    o, lse, ops = run_fp8(q, k, v, w.mask)
    heads = [(0, 0), (0, 31)]
    deq = check_operands(ops, q, k, v, heads)
    rows = np.concatenate([np.arange(r * 128, r * 128 + 128) for r in (0, 55, 56, 200, 255)])
    errs = check_outputs(o, lse, q, k, v, w.mask, deq, rows=rows, what=w.name)
    print(f"fp8 {w.name}: rel_fro(O - O_exact) max {max(errs):.4f}")
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
