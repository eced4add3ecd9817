"""Thin ctypes binding over libflashmask.so (include/flashmask.h).

Argument marshalling only: each function checks dtypes, devices and
contiguity of the torch tensors it is given, passes their device pointers and
the current CUDA stream to the C entry point of the same name, and raises on a
non-OK status. Every step of the computation runs in the library's kernels;
there is no fallback path. If the library is missing the import of the
binding still works but the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libflashmask.so")

FM_OK, FM_ERR_INVALID_ARG, FM_ERR_UNSUPPORTED, FM_ERR_CUDA, FM_ERR_TIMEOUT, FM_ERR_WORKSPACE = range(6)
FM_TILE = 128
FM_TILE_NONE, FM_TILE_PARTIAL, FM_TILE_FULL = 0, 1, 2


class _FmMask(ctypes.Structure):
    _fields_ = [("lts", ctypes.c_void_p), ("lte", ctypes.c_void_p), ("uts", ctypes.c_void_p),
                ("ute", ctypes.c_void_p), ("Hm", ctypes.c_int), ("causal", ctypes.c_int)]


class FmWsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "minmax", "labels", "labels_t", "row_count", "row_list", "row_order",
                 "col_count", "col_list", "col_order", "lse2", "delta", "dq_accum", "kv_part",
                 "kv_sync", "total")]


class FmFp8Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("fwd_total", "q8", "k8", "vt8", "qscale", "kscale", "vscale", "total")]


EXPORTED = ("flashmask_workspace_bytes", "flashmask_workspace_layout", "flashmask_classify",
            "flashmask_fwd", "flashmask_bwd", "flashmask_bwd_preprocess", "flashmask_bwd_main",
            "flashmask_bwd_finalize", "flashmask_fwd_noalloc", "flashmask_host_workspace_bytes",
            "flashmask_fwd_bwd_host", "flashmask_localize", "flashmask_selftest_timeout",
            "flashmask_fwd_fp8_workspace_bytes", "flashmask_fwd_fp8_layout", "flashmask_fwd_fp8",
            "flashmask_check_status", "flashmask_status_string")

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the library (once) and declares the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with mask_aware_exact_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.flashmask_workspace_bytes.argtypes = [i, i, i, i, i, i]
    L.flashmask_workspace_bytes.restype = sz
    L.flashmask_workspace_layout.argtypes = [i, i, i, i, i, i, ctypes.POINTER(FmWsLayout)]
    L.flashmask_workspace_layout.restype = i
    L.flashmask_classify.argtypes = [ctypes.POINTER(_FmMask), i, i, vp, sz, vp]
    L.flashmask_classify.restype = i
    L.flashmask_fwd.argtypes = [vp, vp, vp, ctypes.POINTER(_FmMask), i, i, i, i, f, vp, vp, vp, sz,
                                i, vp]
    L.flashmask_fwd.restype = i
    L.flashmask_bwd.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.POINTER(_FmMask), i, i, i, i, f, vp,
                                vp, vp, vp, sz, i, vp]
    L.flashmask_bwd.restype = i
    L.flashmask_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, i, vp, sz, vp]
    L.flashmask_bwd_preprocess.restype = i
    L.flashmask_bwd_main.argtypes = [vp, vp, vp, vp, ctypes.POINTER(_FmMask), i, i, i, i, f, vp, vp,
                                     vp, sz, vp]
    L.flashmask_bwd_main.restype = i
    L.flashmask_bwd_finalize.argtypes = [i, i, i, i, i, f, vp, vp, sz, vp]
    L.flashmask_bwd_finalize.restype = i
    L.flashmask_fwd_noalloc.argtypes = [vp, vp, vp, ctypes.POINTER(_FmMask), i, i, i, i, f, vp, vp,
                                        vp]
    L.flashmask_fwd_noalloc.restype = i
    L.flashmask_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i]
    L.flashmask_fwd_fp8_workspace_bytes.restype = sz
    L.flashmask_fwd_fp8_layout.argtypes = [i, i, i, i, ctypes.POINTER(FmFp8Layout)]
    L.flashmask_fwd_fp8_layout.restype = i
    L.flashmask_fwd_fp8.argtypes = [vp, vp, vp, ctypes.POINTER(_FmMask), i, i, i, i, f, vp, vp, vp,
                                    sz, i, vp]
    L.flashmask_fwd_fp8.restype = i
    L.flashmask_host_workspace_bytes.argtypes = [i, i, i, i, i, i]
    L.flashmask_host_workspace_bytes.restype = sz
    L.flashmask_fwd_bwd_host.argtypes = [vp, vp, vp, vp, ctypes.POINTER(_FmMask), i, i, i, i, f, vp,
                                         vp, vp, vp, vp, vp, sz, i, vp]
    L.flashmask_fwd_bwd_host.restype = i
    L.flashmask_localize.argtypes = [ctypes.POINTER(_FmMask), i, i, i, i, vp, vp, vp, vp, vp, vp]
    L.flashmask_localize.restype = i
    L.flashmask_selftest_timeout.argtypes = [vp, sz, ctypes.c_longlong, i, vp]
    L.flashmask_selftest_timeout.restype = i
    L.flashmask_check_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
    L.flashmask_check_status.restype = i
    L.flashmask_status_string.argtypes = [i]
    L.flashmask_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


class FlashMaskError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().flashmask_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def _check(status: int, where: str):
    if status != FM_OK:
        raise FlashMaskError(status, where)


def _stream_ptr(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


@dataclass
class DeviceMask:
    """Boundary vectors on the device (int32 [B, Hm, N]) plus Hm and the causal flag."""

    lts: torch.Tensor
    lte: torch.Tensor
    uts: torch.Tensor | None
    ute: torch.Tensor | None
    causal: bool

    @property
    def Hm(self) -> int:
        return self.lts.shape[1]

    @staticmethod
    def from_spec(spec, device="cuda") -> "DeviceMask":
        t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)
        return DeviceMask(t(spec.lts), t(spec.lte), t(spec.uts), t(spec.ute), bool(spec.causal))

    def c_struct(self) -> _FmMask:
        for v in (self.lts, self.lte, self.uts, self.ute):
            if v is not None:
                if v.dtype != torch.int32 or not v.is_cuda or not v.is_contiguous():
                    raise ValueError("mask vectors must be contiguous int32 CUDA tensors")
        p = lambda v: None if v is None else v.data_ptr()
        return _FmMask(p(self.lts), p(self.lte), p(self.uts), p(self.ute), self.Hm, int(self.causal))


def _bf16(x: torch.Tensor, name: str):
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous() or x.dim() != 4:
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor [B, H, N, d]")


def flashmask_workspace_bytes(B, H, Hm, N, d, for_bwd=True) -> int:
    return int(load().flashmask_workspace_bytes(B, H, Hm, N, d, int(bool(for_bwd))))


def flashmask_workspace_layout(B, H, Hm, N, d, for_bwd=True) -> FmWsLayout:
    out = FmWsLayout()
    _check(load().flashmask_workspace_layout(B, H, Hm, N, d, int(bool(for_bwd)), ctypes.byref(out)),
           "flashmask_workspace_layout")
    return out


def alloc_workspace(B, H, Hm, N, d, for_bwd=True, device="cuda") -> torch.Tensor:
    n = flashmask_workspace_bytes(B, H, Hm, N, d, for_bwd)
    if n == 0:
        raise FlashMaskError(FM_ERR_UNSUPPORTED, "flashmask_workspace_bytes")
    ws = torch.zeros(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def flashmask_classify(mask: DeviceMask, B: int, N: int, ws: torch.Tensor, stream=None):
    m = mask.c_struct()
    _check(load().flashmask_classify(ctypes.byref(m), B, N, ws.data_ptr(), ws.numel(),
                                     _stream_ptr(stream)), "flashmask_classify")


def flashmask_fwd(q, k, v, mask: DeviceMask, ws, scale=None, o=None, lse=None, ws_classified=False,
                  stream=None):
    """Returns (O bf16 [B,H,N,d], LSE fp32 [B,H,N])."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _bf16(t, n)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    m = mask.c_struct()
    _check(load().flashmask_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(m), B, H, N,
                                d, scale, o.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(),
                                int(bool(ws_classified)), _stream_ptr(stream)), "flashmask_fwd")
    return o, lse


def flashmask_fwd_fp8_workspace_bytes(B, H, Hm, N) -> int:
    return load().flashmask_fwd_fp8_workspace_bytes(B, H, Hm, N)


def flashmask_fwd_fp8_layout(B, H, Hm, N) -> FmFp8Layout:
    out = FmFp8Layout()
    _check(load().flashmask_fwd_fp8_layout(B, H, Hm, N, ctypes.byref(out)),
           "flashmask_fwd_fp8_layout")
    return out


def read_fp8_operands(ws, B, H, Hm, N):
    """The e4m3 operands and scales the last FP8 forward left in `ws`, as torch
    tensors on its device: q8, k8 uint8 [B,H,N,128], vt8 uint8 [B,H,128,Npad],
    qscale, kscale fp32 [B,H,Tr], vscale fp32 [B,H]."""
    L = flashmask_fwd_fp8_layout(B, H, Hm, N)
    Tr = (N + 127) // 128
    Npad = 128 * Tr

    def part(off, n):
        return ws[off:off + n]
    q8 = part(L.q8, B * H * N * 128).view(B, H, N, 128)
    k8 = part(L.k8, B * H * N * 128).view(B, H, N, 128)
    vt8 = part(L.vt8, B * H * 128 * Npad).view(B, H, 128, Npad)
    qs = part(L.qscale, B * H * Tr * 4).view(torch.float32).view(B, H, Tr)
    ks = part(L.kscale, B * H * Tr * 4).view(torch.float32).view(B, H, Tr)
    vs = part(L.vscale, B * H * 4).view(torch.float32).view(B, H)
    return q8, k8, vt8, qs, ks, vs


def alloc_fp8_workspace(B, H, Hm, N, device="cuda") -> torch.Tensor:
    n = flashmask_fwd_fp8_workspace_bytes(B, H, Hm, N)
    if n == 0:
        raise FlashMaskError(FM_ERR_UNSUPPORTED, "flashmask_fwd_fp8_workspace_bytes")
    ws = torch.zeros(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def flashmask_fwd_fp8(q, k, v, mask: DeviceMask, ws, scale=None, o=None, lse=None,
                      ws_classified=False, stream=None):
    """FP8 (e4m3) forward of bf16 Q, K, V with d = 128; returns (O bf16, LSE fp32)
    like flashmask_fwd. `ws` comes from alloc_fp8_workspace."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _bf16(t, n)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    m = mask.c_struct()
    _check(load().flashmask_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(m), B, H,
                                    N, d, scale, o.data_ptr(), lse.data_ptr(), ws.data_ptr(),
                                    ws.numel(), int(bool(ws_classified)), _stream_ptr(stream)),
           "flashmask_fwd_fp8")
    return o, lse


def flashmask_bwd(q, k, v, o, lse, do, mask: DeviceMask, ws, scale=None, dq=None, dk=None, dv=None,
                  ws_classified=False, stream=None):
    """Returns (dQ, dK, dV) bf16 [B,H,N,d]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _bf16(t, n)
    if lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [B, H, N]")
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    m = mask.c_struct()
    _check(load().flashmask_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), do.data_ptr(), ctypes.byref(m), B, H, N, d, scale,
                                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                                ws.numel(), int(bool(ws_classified)), _stream_ptr(stream)),
           "flashmask_bwd")
    return dq, dk, dv


def flashmask_bwd_preprocess(o, lse, do, Hm: int, ws, stream=None):
    _bf16(o, "o")
    _bf16(do, "do")
    B, H, N, d = o.shape
    _check(load().flashmask_bwd_preprocess(o.data_ptr(), lse.data_ptr(), do.data_ptr(), B, H, Hm, N,
                                           d, ws.data_ptr(), ws.numel(), _stream_ptr(stream)),
           "flashmask_bwd_preprocess")


def flashmask_bwd_main(q, k, v, do, mask: DeviceMask, ws, dk, dv, scale=None, stream=None):
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (do, "do"), (dk, "dk"), (dv, "dv")):
        _bf16(t, n)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    m = mask.c_struct()
    _check(load().flashmask_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                     ctypes.byref(m), B, H, N, d, scale, dk.data_ptr(),
                                     dv.data_ptr(), ws.data_ptr(), ws.numel(),
                                     _stream_ptr(stream)), "flashmask_bwd_main")


def flashmask_bwd_finalize(dq, Hm: int, ws, scale=None, stream=None):
    _bf16(dq, "dq")
    B, H, N, d = dq.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(load().flashmask_bwd_finalize(B, H, Hm, N, d, scale, dq.data_ptr(), ws.data_ptr(),
                                         ws.numel(), _stream_ptr(stream)), "flashmask_bwd_finalize")


def flashmask_check_status(ws: torch.Tensor, stream=None) -> tuple[int, int]:
    """(status, failure site) after synchronising the stream; clears the word."""
    detail = ctypes.c_int(0)
    st = load().flashmask_check_status(ws.data_ptr(), _stream_ptr(stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def flashmask_status_string(status: int) -> str:
    return load().flashmask_status_string(status).decode()


def read_classification(ws: torch.Tensor, B: int, Hm: int, N: int) -> dict:
    """Copies the classification regions of a workspace to host numpy arrays."""
    L = flashmask_workspace_layout(B, Hm, Hm, N, 64, False)
    Tr = Tc = (N + FM_TILE - 1) // FM_TILE
    h = ws[:L.total].cpu().numpy()

    def region(off, count, dtype, shape):
        return h[off:off + count * np.dtype(dtype).itemsize].view(dtype).reshape(shape).copy()

    return {
        "minmax": region(L.minmax, B * Hm * Tc * 8, np.int32, (B, Hm, Tc, 8)),
        "labels": region(L.labels, B * Hm * Tr * Tc, np.uint8, (B, Hm, Tr, Tc)),
        "labels_t": region(L.labels_t, B * Hm * Tc * Tr, np.uint8, (B, Hm, Tc, Tr)),
        "row_count": region(L.row_count, B * Hm * Tr, np.int32, (B, Hm, Tr)),
        "row_list": region(L.row_list, B * Hm * Tr * Tc, np.int32, (B, Hm, Tr, Tc)),
        "row_order": region(L.row_order, B * Hm * Tr, np.int32, (B, Hm, Tr)),
        "col_count": region(L.col_count, B * Hm * Tc, np.int32, (B, Hm, Tc)),
        "col_list": region(L.col_list, B * Hm * Tc * Tr, np.int32, (B, Hm, Tc, Tr)),
        "col_order": region(L.col_order, B * Hm * Tc, np.int32, (B, Hm, Tc)),
    }


def flashmask_fwd_noalloc(q, k, v, mask: DeviceMask, o, lse, scale=None, stream=None):
    """Forward into caller-provided O and LSE with no workspace and no allocation.

    The tables live in the library's fixed scratch array, so calls that may
    overlap on the GPU must be serialised by the caller, and the first call on
    a device must come before any stream capture. Shapes whose tables do not fit
    raise FlashMaskError with FM_ERR_WORKSPACE."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _bf16(t, n)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    m = mask.c_struct()
    _check(load().flashmask_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(m),
                                        B, H, N, d, scale, o.data_ptr(), lse.data_ptr(),
                                        _stream_ptr(stream)), "flashmask_fwd_noalloc")
    return o, lse


# ---------------------------------------------------------------- host buffers
@dataclass
class HostMask:
    """Boundary vectors in host memory (contiguous int32 [B, Hm, N] CPU tensors,
    page-locked when made by from_spec) plus the causal flag."""

    lts: torch.Tensor
    lte: torch.Tensor
    uts: torch.Tensor | None
    ute: torch.Tensor | None
    causal: bool

    @property
    def Hm(self) -> int:
        return self.lts.shape[1]

    @staticmethod
    def from_spec(spec, pin=True) -> "HostMask":
        def t(a):
            if a is None:
                return None
            x = torch.from_numpy(np.ascontiguousarray(a, np.int32))
            return x.pin_memory() if pin else x
        return HostMask(t(spec.lts), t(spec.lte), t(spec.uts), t(spec.ute), bool(spec.causal))

    def c_struct(self) -> _FmMask:
        for v in (self.lts, self.lte, self.uts, self.ute):
            if v is not None:
                if v.dtype != torch.int32 or v.is_cuda or not v.is_contiguous():
                    raise ValueError("host mask vectors must be contiguous int32 CPU tensors")
        p = lambda v: None if v is None else v.data_ptr()
        return _FmMask(p(self.lts), p(self.lte), p(self.uts), p(self.ute), self.Hm, int(self.causal))


def flashmask_host_workspace_bytes(B, H, Hm, N, d, chunk_heads) -> int:
    return int(load().flashmask_host_workspace_bytes(B, H, Hm, N, d, chunk_heads))


def alloc_host_workspace(B, H, Hm, N, d, chunk_heads, device="cuda") -> torch.Tensor:
    n = flashmask_host_workspace_bytes(B, H, Hm, N, d, chunk_heads)
    if n == 0:
        raise FlashMaskError(FM_ERR_UNSUPPORTED, "flashmask_host_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def flashmask_fwd_bwd_host(q, k, v, do, mask: HostMask, dev_ws, chunk_heads, scale=None,
                           out=None, stream=None):
    """Forward and backward between host tensors (bf16 [B,H,N,d], page-locked for
    the copies to overlap). Returns (O, LSE, dQ, dK, dV) on the host; `out` may
    hold preallocated host tensors in that order. Blocks until the results are
    in host memory."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (do, "do")):
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous bf16 CPU tensor")
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        pin = q.is_pinned()
        mk = lambda shape, dt: torch.empty(shape, dtype=dt, pin_memory=pin)
        out = (mk(q.shape, torch.bfloat16), mk((B, H, N), torch.float32), mk(q.shape, torch.bfloat16),
               mk(q.shape, torch.bfloat16), mk(q.shape, torch.bfloat16))
    o, lse, dq, dk, dv = out
    m = mask.c_struct()
    _check(load().flashmask_fwd_bwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                         ctypes.byref(m), B, H, N, d, scale, o.data_ptr(),
                                         lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                         dev_ws.data_ptr(), dev_ws.numel(), int(chunk_heads),
                                         _stream_ptr(stream)), "flashmask_fwd_bwd_host")
    return o, lse, dq, dk, dv


def flashmask_localize(mask: DeviceMask, B: int, N: int, row0: int, rows: int, stream=None):
    """Boundary vectors of the local problem of a rank holding query rows
    [row0, row0 + rows): returns (DeviceMask with causal=False, inexact flag as
    a bool). Synchronises the stream to read the flag."""
    dev = mask.lts.device
    shape = (B, mask.Hm, N)
    out = [torch.empty(shape, dtype=torch.int32, device=dev) for _ in range(4)]
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    m = mask.c_struct()
    _check(load().flashmask_localize(ctypes.byref(m), B, N, int(row0), int(rows), out[0].data_ptr(),
                                     out[1].data_ptr(), out[2].data_ptr(), out[3].data_ptr(),
                                     flag.data_ptr(), _stream_ptr(stream)), "flashmask_localize")
    return DeviceMask(out[0], out[1], out[2], out[3], False), bool(flag.item())


def flashmask_selftest_timeout(ws: torch.Tensor, limit_ns: int, ctas: int = 1, stream=None):
    """Queues the bounded-wait self-test (see include/flashmask.h)."""
    _check(load().flashmask_selftest_timeout(ws.data_ptr(), ws.numel(), int(limit_ns), int(ctas),
                                             _stream_ptr(stream)), "flashmask_selftest_timeout")
