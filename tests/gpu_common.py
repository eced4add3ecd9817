"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
binding and compare against the fp64 oracle with the stated tolerances."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from mask_aware_exact_gb300 import workloads as W

# tolerances of the method's parity bar
TOL_O = 1e-2       # max |O - O_ref|
TOL_LSE = 1e-3     # max |LSE - LSE_ref| over rows with a visible key
TOL_GRAD = 2e-2    # ||dX - dX_ref||_F / ||dX_ref||_F for X in {Q, K, V}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mask_aware_exact_gb300 import build
    build.build()
    from mask_aware_exact_gb300 import flashmask as fm
    fm.load()
    return fm


def run_path(fm, q, k, v, do, spec, scale=None, bwd=True):
    """Classify + forward (+ backward) on the GPU. Inputs are CPU bf16 tensors."""
    dev = "cuda"
    B, H, N, d = q.shape
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    mask = fm.DeviceMask.from_spec(spec)
    ws = fm.alloc_workspace(B, H, mask.Hm, N, d, for_bwd=bwd)
    fm.flashmask_classify(mask, B, N, ws)
    o, lse = fm.flashmask_fwd(qd, kd, vd, mask, ws, scale=scale, ws_classified=True)
    out = {"o": o, "lse": lse, "ws": ws, "mask": mask}
    if bwd:
        dq, dk, dv = fm.flashmask_bwd(qd, kd, vd, o, lse, dod, mask, ws, scale=scale,
                                      ws_classified=True)
        out.update(dq=dq, dk=dk, dv=dv)
    st, site = fm.flashmask_check_status(ws)
    assert st == fm.FM_OK, f"device status {st} at site {site}"
    return out


def to_np(x):
    return x.detach().float().cpu().numpy().astype(np.float64)


def rel_fro(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / nb if nb > 0 else np.linalg.norm(a)


def check_forward(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    err_o = np.abs(o_gpu - o_ref).max()
    fin = np.isfinite(lse_ref)
    err_l = np.abs(lse_gpu[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert err_o <= TOL_O, f"{what} max|O-O_ref| = {err_o}"
    assert err_l <= TOL_LSE, f"{what} max|LSE-LSE_ref| = {err_l}"
    # fully masked rows: O = 0 and LSE = -inf exactly
    assert np.all(np.isneginf(lse_gpu[~fin])), f"{what} fully masked rows must have LSE=-inf"
    assert np.all(o_gpu[~fin] == 0), f"{what} fully masked rows must have O=0"
    return err_o, err_l


def check_grad(name, g, ref, what=""):
    e = rel_fro(g, ref)
    assert e <= TOL_GRAD, f"{what} rel_fro(d{name}) = {e}"
    return e


def head_bounds(spec, b, h, H):
    hm = h // (H // spec.Hm)
    g = lambda a: None if a is None else a[b, hm]
    return g(spec.lts), g(spec.lte), g(spec.uts), g(spec.ute)
