"""Pins the fp64 oracle (forward and backward) to things other than itself:
torch's fp64 scaled_dot_product_attention and autograd, scipy's logsumexp and
softmax, central finite differences, and closed forms."""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

from mask_aware_exact_gb300 import workloads as W
from oracle import attention as A


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def random_case(N=96, d=16, seed=0, causal=True, upper=True):
    """Adversarial random bounds (some rows end up fully masked) and fp64 data."""
    spec = W.random_bounds(1, 1, N, causal, seed, upper)
    g = lambda a: None if a is None else a[0, 0]
    b = (g(spec.lts), g(spec.lte), g(spec.uts), g(spec.ute))
    vis = A.visible(np.arange(N), N, *b, causal)
    q, k, v, do = (rand((N, d), seed + i) for i in range(1, 5))
    return b, vis, q, k, v, do


def torch_sdpa(q, k, v, vis, scale):
    t = lambda x: torch.tensor(x, dtype=torch.float64, requires_grad=True)
    tq, tk, tv = t(q), t(k), t(v)
    o = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], attn_mask=torch.tensor(vis)[None, None],
        scale=scale)[0, 0]
    return o, (tq, tk, tv)


@pytest.mark.parametrize("seed,causal,upper", [(0, True, True), (1, False, True), (2, True, False),
                                               (3, False, False)])
def test_forward_vs_torch_sdpa_and_logsumexp(seed, causal, upper):
    N, d = 96, 16
    b, vis, q, k, v, do = random_case(N, d, seed, causal, upper)
    scale = 1 / np.sqrt(d)
    O, LSE = A.forward_head(q, k, v, *b, causal, scale, block=32)
    has = vis.any(axis=1)
    assert has.sum() > N // 4  # the case exercises visible rows
    o_ref, _ = torch_sdpa(q, k, v, vis, scale)
    np.testing.assert_allclose(O[has], o_ref.detach().numpy()[has], rtol=0, atol=1e-12)
    S = np.where(vis, scale * q @ k.T, -np.inf)
    np.testing.assert_allclose(LSE[has], logsumexp(S[has], axis=1), rtol=0, atol=1e-12)
    # fully masked rows: O = 0 and LSE = -inf
    assert np.all(O[~has] == 0) and np.all(np.isneginf(LSE[~has]))


def test_forward_unmasked_is_textbook_softmax_attention():
    N, d = 64, 8
    q, k, v = rand((N, d), 1), rand((N, d), 2), rand((N, d), 3)
    empty = np.full(N, N)
    scale = 0.37
    O, LSE = A.forward_head(q, k, v, empty, empty, None, None, False, scale)
    P = softmax(scale * q @ k.T, axis=1)
    np.testing.assert_allclose(O, P @ v, atol=1e-12)
    np.testing.assert_allclose(LSE, logsumexp(scale * q @ k.T, axis=1), atol=1e-12)


def test_forward_causal_is_textbook_causal():
    N, d = 64, 8
    q, k, v = rand((N, d), 4), rand((N, d), 5), rand((N, d), 6)
    empty = np.full(N, N)
    O, _ = A.forward_head(q, k, v, empty, empty, None, None, True, 0.5)
    S = 0.5 * q @ k.T + np.triu(np.full((N, N), -np.inf), 1)
    np.testing.assert_allclose(O, softmax(S, axis=1) @ v, atol=1e-12)


def test_single_visible_key_closed_form():
    # column j masked for every row except row j itself: each row sees exactly key i
    N, d = 40, 8
    q, k, v = rand((N, d), 7), rand((N, d), 8), rand((N, d), 9)
    j = np.arange(N)
    uts, ute = np.zeros(N, int), j          # rows [0, j) masked
    lts, lte = j + 1, np.full(N, N)         # rows [j+1, N) masked
    O, LSE = A.forward_head(q, k, v, lts, lte, uts, ute, False, 0.25)
    np.testing.assert_allclose(O, v, atol=1e-14)
    np.testing.assert_allclose(LSE, 0.25 * (q * k).sum(1), atol=1e-14)


def test_zero_query_gives_mean_of_visible_values():
    N, d = 48, 8
    spec = W.document_bounds(1, 1, [20, 28])
    lts, lte = spec.lts[0, 0], spec.lte[0, 0]
    k, v = rand((N, d), 10), rand((N, d), 11)
    O, LSE = A.forward_head(np.zeros((N, d)), k, v, lts, lte, None, None, True, 1.0)
    vis = A.visible(np.arange(N), N, lts, lte, None, None, True)
    expect = (vis @ v) / vis.sum(1, keepdims=True)
    np.testing.assert_allclose(O, expect, atol=1e-13)
    np.testing.assert_allclose(LSE, np.log(vis.sum(1)), atol=1e-13)


def test_probability_rows_sum_to_one():
    N, d = 80, 8
    b, vis, q, k, _, _ = random_case(N, d, 12)
    O, _ = A.forward_head(q, k, np.ones((N, 1)), *b, True, 0.3)
    has = vis.any(1)
    np.testing.assert_allclose(O[has, 0], 1.0, atol=1e-12)
    assert np.all(O[~has] == 0)


@pytest.mark.parametrize("seed,causal", [(20, True), (21, False)])
def test_backward_vs_torch_autograd(seed, causal):
    N, d = 96, 16
    b, vis, q, k, v, do = random_case(N, d, seed, causal)
    has = vis.any(1)
    scale = 1 / np.sqrt(d)
    dq, dk, dv = A.backward_head(q, k, v, do, *b, causal, scale, block=40)
    o, (tq, tk, tv) = torch_sdpa(q, k, v, vis, scale)
    # rows with no visible key produce NaN in torch; they carry no gradient here
    loss = (o[torch.tensor(has)] * torch.tensor(do)[torch.tensor(has)]).sum()
    loss.backward()
    np.testing.assert_allclose(dq[has], tq.grad.numpy()[has], atol=1e-11)
    np.testing.assert_allclose(dq[~has], 0.0, atol=0)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


def test_backward_finite_differences():
    N, d = 14, 4
    b, vis, q, k, v, do = random_case(N, d, 30, True)
    scale = 0.7
    dq, dk, dv = A.backward_head(q, k, v, do, *b, True, scale)

    def loss(q_, k_, v_):
        O, _ = A.forward_head(q_, k_, v_, *b, True, scale)
        return float((O * do).sum())

    h = 1e-6
    for name, X, G in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = Xp
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = Xm
            lm = loss(args["q"], args["k"], args["v"])
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(num - G) / max(np.linalg.norm(G), 1e-30)
        assert err < 1e-6, (name, err)


def test_backward_row_subset_gives_complete_key_gradients():
    # dK_j, dV_j from only the rows that see j equal the full result
    N, d = 64, 8
    spec = W.document_bounds(1, 1, [30, 34])
    lts, lte = spec.lts[0, 0], spec.lte[0, 0]
    q, k, v, do = (rand((N, d), 40 + i) for i in range(4))
    full = A.backward_head(q, k, v, do, lts, lte, None, None, True, 0.4)
    rows = np.arange(30, 64)  # rows of the second document
    sub = A.backward_head(q, k, v, do, lts, lte, None, None, True, 0.4, rows=rows)
    np.testing.assert_allclose(sub[1][30:], full[1][30:], atol=1e-13)
    np.testing.assert_allclose(sub[2][30:], full[2][30:], atol=1e-13)
    np.testing.assert_allclose(sub[0], full[0][30:], atol=1e-13)


def test_mask_heads_broadcast():
    # Hm = 2 mask heads over H = 4 heads: heads 0,1 use mask head 0; heads 2,3 mask head 1
    B, H, N, d = 1, 4, 32, 8
    q, k, v, do = (torch.tensor(rand((B, H, N, d), 50 + i)) for i in range(4))
    m0 = W.document_bounds(1, 1, [10, 22])
    m1 = W.causal_bounds(1, 1, N)
    spec = W.MaskSpec("mix", True, np.concatenate([m0.lts, m1.lts], 1),
                      np.concatenate([m0.lte, m1.lte], 1), None, None)
    O, _ = A.forward(q, k, v, spec, 0.3)
    for h in range(H):
        src = m0 if h < 2 else m1
        o, _ = A.forward_head(q[0, h], k[0, h], v[0, h], src.lts[0, 0], src.lte[0, 0], None, None,
                              True, 0.3)
        np.testing.assert_allclose(O[0, h], o, atol=0)


def test_batched_wrappers_vs_torch_autograd_per_head_masks():
    # The [B, H] wrappers against torch fp64 SDPA + autograd on the whole
    # batch at once, with a different dense mask for each (batch, mask head)
    # written straight from the family definitions (not from boundary
    # vectors). B = 2, H = 4, Hm = 2: heads 0, 1 read mask head 0 and heads
    # 2, 3 read mask head 1, so a wrong head -> mask-head mapping, a swapped
    # batch, or a permuted (dQ, dK, dV) return order fails here.
    from oracle import masks_independent as MI
    B, H, N, d = 2, 4, 40, 8
    docs = [[12, 28], [25, 15]]
    families = {  # (b, hm) -> (bounds spec [1, 1, N], dense visibility)
        (0, 0): (W.document_bounds(1, 1, docs[0]), MI.causal_document(docs[0])),
        (0, 1): (W.causal_bounds(1, 1, N), MI.causal(N)),
        (1, 0): (W.share_question_bounds(1, 1, 10, [18, 12]), MI.share_question(10, [18, 12])),
        (1, 1): (W.document_bounds(1, 1, docs[1]), MI.causal_document(docs[1])),
    }
    cat = lambda name: np.concatenate(
        [np.concatenate([getattr(families[(b, hm)][0], name) for hm in range(2)], 1)
         for b in range(B)], 0)
    spec = W.MaskSpec("per_batch_head", True, cat("lts"), cat("lte"), None, None)
    dense = np.zeros((B, H, N, N), bool)
    for b in range(B):
        for h in range(H):
            dense[b, h] = families[(b, 0 if h < 2 else 1)][1]
    q, k, v, do = (rand((B, H, N, d), 70 + i) for i in range(4))
    scale = 0.3
    O, LSE = A.forward(q, k, v, spec, scale)
    dq, dk, dv = A.backward(q, k, v, do, spec, scale)
    t = lambda x: torch.tensor(x, dtype=torch.float64, requires_grad=True)
    tq, tk, tv = t(q), t(k), t(v)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv,
                                                         attn_mask=torch.tensor(dense),
                                                         scale=scale)
    (o * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(O, o.detach().numpy(), atol=1e-12)
    S = np.where(dense, scale * np.einsum("bhid,bhjd->bhij", q, k), -np.inf)
    np.testing.assert_allclose(LSE, logsumexp(S, axis=-1), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


def test_batched_wrapper_heads_subset_leaves_others_unset():
    # only the requested heads are computed; the rest stay NaN
    B, H, N, d = 1, 3, 16, 4
    spec = W.causal_bounds(B, 1, N)
    q, k, v, do = (rand((B, H, N, d), 80 + i) for i in range(4))
    dq, dk, dv = A.backward(q, k, v, do, spec, 0.5, heads=[(0, 1)])
    for g in (dq, dk, dv):
        assert np.isnan(g[0, 0]).all() and np.isnan(g[0, 2]).all() and np.isfinite(g[0, 1]).all()
