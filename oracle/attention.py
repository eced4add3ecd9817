"""fp64 dense-mask attention, forward and backward (test infrastructure only).

Definitions followed ("FlashMask: Efficient and Rich Mask Extension of
FlashAttention", abstract: exact attention under a column-wise sparse mask;
"FlashMask-3", abstract: four query-axis boundary vectors per key column;
"FlashAttention-3", abstract, and "FlashAttention" README: the exact attention
the tiled kernels reproduce):

  visible(i, j) = not [ (causal and j > i) or LTS_j <= i < LTE_j or UTS_j <= i < UTE_j ]
  s_ij   = scale * <q_i, k_j>
  m_i    = max over visible j of s_ij
  l_i    = sum over visible j of exp(s_ij - m_i)
  P_ij   = exp(s_ij - m_i) / l_i   (visible),  0 (masked)
  O_i    = sum_j P_ij v_j
  LSE_i  = m_i + ln l_i
  A row with no visible key has O_i = 0, LSE_i = -inf and contributes nothing
  to any gradient.

  dV_j  = sum_i P_ij dO_i
  dP_ij = <dO_i, v_j>
  D_i   = <dO_i, O_i>
  dS_ij = P_ij (dP_ij - D_i)
  dQ_i  = scale * sum_j dS_ij k_j
  dK_j  = scale * sum_i dS_ij q_i

The mask is materialised one block of rows at a time (a [rows, N] boolean
array); that is the only departure from "build the N x N mask", and it changes
no value. Each row block sees every key, so its softmax is complete.
"""
from __future__ import annotations

import numpy as np

ROW_BLOCK = 256


def _f64(x) -> np.ndarray:
    """fp64 copy of an array or a torch tensor (bf16 tensors are widened exactly)."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return x.detach().to(torch.float64).cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def visible(rows, N: int, lts, lte, uts, ute, causal: bool) -> np.ndarray:
    """Dense visibility [len(rows), N] for one mask head, from the boundary vectors.

    ``uts``/``ute`` may be None (no upper interval)."""
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(N, dtype=np.int64)[None, :]
    masked = (np.asarray(lts, np.int64)[None, :] <= i) & (i < np.asarray(lte, np.int64)[None, :])
    if uts is not None:
        masked |= (np.asarray(uts, np.int64)[None, :] <= i) & (i < np.asarray(ute, np.int64)[None, :])
    if causal:
        masked |= j > i
    return ~masked


def forward_head(q, k, v, lts, lte, uts, ute, causal: bool, scale: float, rows=None,
                 block: int = ROW_BLOCK):
    """O [R, d] and LSE [R] (natural log) for one (batch, head), fp64.

    q, k, v: [N, d]; bounds: [N] for this head's mask head; ``rows`` selects
    which query rows to compute (all by default)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    N = k.shape[0]
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.zeros((len(rows), v.shape[1]))
    LSE = np.empty(len(rows))
    for s in range(0, len(rows), block):
        r = rows[s:s + block]
        vis = visible(r, N, lts, lte, uts, ute, causal)
        S = np.where(vis, scale * (q[r] @ k.T), -np.inf)
        m = S.max(axis=1)
        has = np.isfinite(m)
        m0 = np.where(has, m, 0.0)
        E = np.where(vis, np.exp(S - m0[:, None]), 0.0)
        l = E.sum(axis=1)
        P = E / np.where(has, l, 1.0)[:, None]
        O[s:s + block] = P @ v
        LSE[s:s + block] = np.where(has, m0 + np.log(np.where(has, l, 1.0)), -np.inf)
    return O, LSE


def backward_head(q, k, v, do, lts, lte, uts, ute, causal: bool, scale: float, rows=None,
                  block: int = ROW_BLOCK):
    """dQ [R, d] for the selected rows and dK, dV [N, d] summed over those rows, fp64.

    With ``rows=None`` every row is used and dK, dV are complete. With a subset,
    dK_j and dV_j are complete for every key j whose visible rows all lie in
    the subset (rows that cannot see j contribute exactly zero)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    N = k.shape[0]
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    dQ = np.zeros((len(rows), q.shape[1]))
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for s in range(0, len(rows), block):
        r = rows[s:s + block]
        vis = visible(r, N, lts, lte, uts, ute, causal)
        S = np.where(vis, scale * (q[r] @ k.T), -np.inf)
        m = S.max(axis=1)
        has = np.isfinite(m)
        m0 = np.where(has, m, 0.0)
        E = np.where(vis, np.exp(S - m0[:, None]), 0.0)
        l = E.sum(axis=1)
        P = E / np.where(has, l, 1.0)[:, None]
        O = P @ v
        dO = do[r]
        D = (dO * O).sum(axis=1)
        dP = dO @ v.T
        dS = P * (dP - D[:, None])
        dQ[s:s + block] = scale * (dS @ k)
        dK += scale * (dS.T @ q[r])
        dV += P.T @ dO
    return dQ, dK, dV


def _head_bounds(mask, b: int, h: int, H: int):
    """This head's boundary vectors: head h reads mask head h // (H // Hm)."""
    Hm = mask.lts.shape[1]
    hm = h // (H // Hm)
    pick = lambda a: None if a is None else a[b, hm]
    return pick(mask.lts), pick(mask.lte), pick(mask.uts), pick(mask.ute)


def forward(q, k, v, mask, scale: float, heads=None):
    """O [B,H,N,d], LSE [B,H,N] (fp64) for every (b, h) in ``heads`` (default all);
    entries of heads not computed are NaN."""
    B, H, N, d = q.shape
    O = np.full((B, H, N, d), np.nan)
    LSE = np.full((B, H, N), np.nan)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        lts, lte, uts, ute = _head_bounds(mask, b, h, H)
        O[b, h], LSE[b, h] = forward_head(q[b, h], k[b, h], v[b, h], lts, lte, uts, ute,
                                          mask.causal, scale)
    return O, LSE


def backward(q, k, v, do, mask, scale: float, heads=None):
    """dQ, dK, dV [B,H,N,d] (fp64) for every (b, h) in ``heads`` (default all)."""
    B, H, N, d = q.shape
    out = [np.full((B, H, N, d), np.nan) for _ in range(3)]
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        lts, lte, uts, ute = _head_bounds(mask, b, h, H)
        dq, dk, dv = backward_head(q[b, h], k[b, h], v[b, h], do[b, h], lts, lte, uts, ute,
                                   mask.causal, scale)
        out[0][b, h], out[1][b, h], out[2][b, h] = dq, dk, dv
    return tuple(out)


def visible_count(N: int, lts, lte, uts, ute, causal: bool, block: int = 1024) -> int:
    """Number of visible (i, j) pairs of one mask head, counted on the dense mask."""
    total = 0
    for s in range(0, N, block):
        total += int(visible(np.arange(s, min(s + block, N)), N, lts, lte, uts, ute, causal).sum())
    return total
