"""CUDA forward and backward vs the fp64 oracle, element by element.

Small cases are compared in full (several tiles, PARTIAL and NONE tiles, fully
masked rows, mask heads, d = 64 and 128). The large workloads run in the same
launch configuration the benchmark times and are compared on sampled outputs
that the oracle computes one by one: query rows for O, LSE and dQ; key blocks
for dK and dV, using exactly the query rows that can see those keys (rows that
cannot see key j contribute nothing to dK_j or dV_j)."""
import math

import numpy as np
import pytest
import torch

from mask_aware_exact_gb300 import workloads as W
from oracle import attention as A

from gpu_common import (check_forward, check_grad, head_bounds, need_gpu, run_path, to_np)

pytestmark = pytest.mark.gpu


def full_compare(fm, q, k, v, do, spec, scale=None, what=""):
    B, H, N, d = q.shape
    scale_v = 1 / math.sqrt(d) if scale is None else scale
    out = run_path(fm, q, k, v, do, spec, scale=scale)
    o_ref, lse_ref = A.forward(q, k, v, spec, scale_v)
    dq_ref, dk_ref, dv_ref = A.backward(q, k, v, do, spec, scale_v)
    check_forward(to_np(out["o"]), to_np(out["lse"]), o_ref, lse_ref, what)
    check_grad("Q", to_np(out["dq"]), dq_ref, what)
    check_grad("K", to_np(out["dk"]), dk_ref, what)
    check_grad("V", to_np(out["dv"]), dv_ref, what)
    return out


def test_document_small_workload_full():
    fm = need_gpu()
    w = W.workload(0)
    q, k, v, do = W.make_qkv(w.B, w.H, w.N, w.d, w.seed)
    full_compare(fm, q, k, v, do, w.mask, what=w.name)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kind", ["causal", "document", "window_prefix", "share_question",
                                  "unmasked"])
def test_families_small(kind, d):
    fm = need_gpu()
    B, H, N = 2, 2, 640  # 5 x 5 tiles
    if kind == "causal":
        spec = W.causal_bounds(B, 1, N)
    elif kind == "document":
        spec = W.document_bounds(B, 1, [200, 37, 300, 103])
    elif kind == "window_prefix":
        spec = W.window_prefix_bounds(B, 1, N, 160, 96)
    elif kind == "share_question":
        spec = W.share_question_bounds(B, 1, 192, [150, 170, 128])
    else:
        e = np.full((B, 1, N), N, np.int32)
        spec = W.MaskSpec("none", False, e, e.copy(), None, None)
    q, k, v, do = W.make_qkv(B, H, N, d, seed=7)
    full_compare(fm, q, k, v, do, spec, what=f"{kind} d={d}")


@pytest.mark.parametrize("seed", range(4))
def test_random_bounds_with_fully_masked_rows(seed):
    fm = need_gpu()
    B, H, N, d = 1, 4, 384, 128
    Hm = [1, 2, 4, 1][seed]
    spec = W.random_bounds(B, Hm, N, causal=seed % 2 == 0, seed=300 + seed, upper=True)
    q, k, v, do = W.make_qkv(B, H, N, d, seed=seed)
    full_compare(fm, q, k, v, do, spec, what=f"random seed {seed}")


def test_fully_masked_rows_inside_partial_tiles():
    # rows 64..99 and 300..301 see no key at all; their tiles also hold
    # visible rows, so the convention is exercised inside PARTIAL tiles
    fm = need_gpu()
    B, H, N, d = 1, 2, 384, 128
    lts = np.full((1, 1, N), 64, np.int32)
    lte = np.full((1, 1, N), 100, np.int32)
    uts = np.full((1, 1, N), 300, np.int32)
    ute = np.full((1, 1, N), 302, np.int32)
    spec = W.MaskSpec("holes", True, lts, lte, uts, ute)
    q, k, v, do = W.make_qkv(B, H, N, d, seed=21)
    out = full_compare(fm, q, k, v, do, spec, what="masked rows")
    lse = to_np(out["lse"])
    assert np.all(np.isneginf(lse[:, :, 64:100])) and np.all(np.isneginf(lse[:, :, 300:302]))
    assert np.isfinite(lse[:, :, :64]).all() and np.isfinite(lse[:, :, 100:300]).all()


def test_all_masked_and_all_visible_blocks():
    # query block 1 entirely masked (every tile FULL), block 0 entirely visible
    fm = need_gpu()
    B, H, N, d = 1, 2, 256, 64
    lts = np.full((1, 1, N), 128, np.int32)
    lte = np.full((1, 1, N), 256, np.int32)
    spec = W.MaskSpec("block", False, lts, lte, None, None)
    q, k, v, do = W.make_qkv(B, H, N, d, seed=11)
    out = full_compare(fm, q, k, v, do, spec, what="masked block")
    assert np.all(np.isneginf(to_np(out["lse"])[:, :, 128:]))
    assert np.all(to_np(out["dq"])[:, :, 128:] == 0)


def test_custom_scale():
    fm = need_gpu()
    w = W.workload(0)
    q, k, v, do = W.make_qkv(w.B, w.H, w.N, w.d, 3)
    full_compare(fm, q, k, v, do, w.mask, scale=0.05, what="scale 0.05")


def test_repeatable():
    # forward and dK / dV are deterministic; dQ is summed by reductions whose
    # order may vary, so it is only required within tolerance
    fm = need_gpu()
    B, H, N, d = 1, 4, 1024, 128
    spec = W.document_bounds(B, 1, [300, 500, 224])
    q, k, v, do = W.make_qkv(B, H, N, d, seed=5)
    a = run_path(fm, q, k, v, do, spec)
    b = run_path(fm, q, k, v, do, spec)
    for key in ("o", "lse", "dk", "dv"):
        assert torch.equal(a[key], b[key]), key
    assert (a["dq"].float() - b["dq"].float()).abs().max().item() < 1e-2


# ---------------------------------------------------------------- full-size workloads
def sampled_compare(w, out, q, k, v, do, heads, row_blocks, key_blocks):
    d = w.d
    scale = 1 / math.sqrt(d)
    N = w.N
    for (b, h) in heads:
        lts, lte, uts, ute = head_bounds(w.mask, b, h, w.H)
        causal = w.mask.causal
        rows = np.concatenate([np.arange(r * 128, r * 128 + 128) for r in row_blocks])
        o_ref, lse_ref = A.forward_head(q[b, h], k[b, h], v[b, h], lts, lte, uts, ute, causal,
                                        scale, rows=rows)
        check_forward(to_np(out["o"][b, h])[rows], to_np(out["lse"][b, h])[rows], o_ref, lse_ref,
                      f"{w.name} head {(b, h)}")
        dq_ref, _, _ = A.backward_head(q[b, h], k[b, h], v[b, h], do[b, h], lts, lte, uts, ute,
                                       causal, scale, rows=rows)
        check_grad("Q", to_np(out["dq"][b, h])[rows], dq_ref, f"{w.name} head {(b, h)}")
        keys = np.concatenate([np.arange(c * 128, c * 128 + 128) for c in key_blocks])
        # every query row that sees at least one sampled key
        seen = np.zeros(N, bool)
        for s in range(0, N, 2048):
            vis = A.visible(np.arange(s, min(s + 2048, N)), N, lts, lte, uts, ute, causal)
            seen[s:s + vis.shape[0]] = vis[:, keys].any(axis=1)
        sub = np.nonzero(seen)[0]
        _, dk_ref, dv_ref = A.backward_head(q[b, h], k[b, h], v[b, h], do[b, h], lts, lte, uts,
                                            ute, causal, scale, rows=sub)
        check_grad("K", to_np(out["dk"][b, h])[keys], dk_ref[keys], f"{w.name} head {(b, h)}")
        check_grad("V", to_np(out["dv"][b, h])[keys], dv_ref[keys], f"{w.name} head {(b, h)}")


def _every(step, n, extra=()):
    return sorted(set(range(0, n, step)) | set(extra))


SAMPLES = {
    # workload index: (heads, query blocks, key blocks). Heads: the first and
    # the last of the head-major work order (the persistent forward and the
    # backward visit heads in order, longest blocks first within a head, so
    # these are the first and last heads the CTAs take); query blocks: every
    # 8th plus the blocks at document, question, window and prefix edges; key
    # blocks spread over the sequence.
    1: ([(0, 0), (1, 7), (3, 15)], _every(8, 64, [31, 63]), [0, 9, 20, 31, 40, 52, 63]),
    2: ([(0, 0), (0, 31)], _every(8, 256, [55, 56, 97, 255]),
        [3, 33, 60, 100, 140, 180, 220, 255]),
    3: ([(0, 0), (1, 31)], _every(8, 128, [31, 32, 81, 93, 114, 127]),
        [5, 33, 48, 64, 81, 100, 120, 127]),
    # at 128K every sampled row costs the oracle a 131072-key softmax: the
    # prefix edge (blocks 15 | 16), the first full window (31, 32) and the end
    4: ([(0, 0), (0, 7)], [0, 15, 16, 17, 31, 32, 500, 1022, 1023], [16, 17, 400, 1023]),
}


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_full_size_workload_sampled(idx):
    fm = need_gpu()
    w = W.workload(idx)
    q, k, v, do = W.make_qkv(w.B, w.H, w.N, w.d, w.seed)
    out = run_path(fm, q, k, v, do, w.mask)
    heads, rb, kb = SAMPLES[idx]
    sampled_compare(w, out, q, k, v, do, heads, rb, kb)
    # properties that hold at any size: finite outputs, every row sees a key
    for key in ("o", "dq", "dk", "dv"):
        assert torch.isfinite(out[key].float()).all(), key
    assert torch.isfinite(out["lse"]).all()


def test_window_prefix_reduced_full():
    # the prefix columns of the 128K window workload are seen by every row, so
    # their dK / dV are checked in full on the same family at N = 8192
    fm = need_gpu()
    B, H, N, d = 1, 2, 8192, 128
    spec = W.window_prefix_bounds(B, 1, N, 4096, 2048)
    q, k, v, do = W.make_qkv(B, H, N, d, seed=0)
    full_compare(fm, q, k, v, do, spec, what="window_prefix N=8192")


@pytest.mark.parametrize("N,d", [(16384, 128), (16347, 64), (32768, 64)])
def test_split_key_blocks_full(N, d, monkeypatch):
    # a 512-token global prefix: its four key blocks are seen by every query
    # block (128 of them at 16K, 256 at 32K), so the backward (splitting from
    # 0 key blocks on here, 512 by default) splits each over two (16K) or four
    # (32K) CTAs and adds the parts' dK, dV; compared in full with the oracle
    monkeypatch.setenv("FM_BWD_SPLIT_MIN_BLOCKS", "0")
    fm = need_gpu()
    B, H = 1, 1
    spec = W.window_prefix_bounds(B, 1, N, 1024, 512)
    q, k, v, do = W.make_qkv(B, H, N, d, seed=21)
    full_compare(fm, q, k, v, do, spec, what=f"split key blocks N={N} d={d}")


@pytest.mark.parametrize("N,d,kind", [(129, 64, "causal"), (200, 128, "document"),
                                      (333, 64, "random"), (600, 128, "window_prefix"),
                                      (1000, 128, "share_question"), (77, 128, "random")])
def test_ragged_sequence_lengths(N, d, kind):
    # N not a multiple of 128: short last query and key blocks, compared in full
    fm = need_gpu()
    B, H = 2, 2
    if kind == "causal":
        spec = W.causal_bounds(B, 1, N)
    elif kind == "document":
        spec = W.document_bounds(B, 1, [61, 100, 39])
    elif kind == "window_prefix":
        spec = W.window_prefix_bounds(B, 1, N, 150, 70)
    elif kind == "share_question":
        spec = W.share_question_bounds(B, 1, 300, [250, 290, 160])
    else:
        spec = W.random_bounds(B, 2, N, causal=N % 2 == 1, seed=N, upper=True)
    q, k, v, do = W.make_qkv(B, H, N, d, seed=N)
    full_compare(fm, q, k, v, do, spec, what=f"ragged N={N} {kind} d={d}")


@pytest.mark.parametrize("kind,N,d", [("bidirectional_document", 640, 128),
                                      ("bidirectional_document", 300, 64),
                                      ("block_causal", 640, 64), ("block_causal", 500, 128),
                                      ("per_head", 384, 128), ("block_sparse", 1024, 128),
                                      ("block_sparse", 700, 64), ("block_sparse", 896, 128)])
def test_more_mask_families(kind, N, d):
    fm = need_gpu()
    B = 2
    if kind == "block_sparse":
        # seeded runs of query blocks per key block plus a global first block;
        # block 64 (N = 700) and 96 (N = 896) make tiles with mixed columns
        block = {1024: 128, 700: 64, 896: 96}[N]
        spec, H = W.block_sparse_bounds(B, 1, N, block, seed=N), 2
    elif kind == "bidirectional_document":
        lengths = [N // 3, N // 4, N - N // 3 - N // 4]
        spec, H = W.bidirectional_document_bounds(B, 1, lengths), 2
    elif kind == "block_causal":
        spec, H = W.block_causal_bounds(B, 1, N, 96), 2
    else:
        # one mask per head (Hm = H = 4), four families with one causal flag
        parts = [W.document_bounds(B, 1, [100, 200, 84]), W.causal_bounds(B, 1, N),
                 W.share_question_bounds(B, 1, 128, [128, 128]),
                 W.random_bounds(B, 1, N, causal=True, seed=9, upper=True)]
        spec, H = W.stack_heads(parts), 4
    q, k, v, do = W.make_qkv(B, H, N, d, seed=N + d)
    full_compare(fm, q, k, v, do, spec, what=f"{kind} N={N} d={d}")


def test_classification_reused_across_layers():
    # one classification of the mask serves several forward calls (layers of a
    # model that share the mask), each with its own Q, K, V
    fm = need_gpu()
    B, H, N, d = 1, 4, 512, 128
    spec = W.document_bounds(B, 2, [200, 312])  # Hm = 2: two heads per mask head
    mask = fm.DeviceMask.from_spec(spec)
    ws = fm.alloc_workspace(B, H, mask.Hm, N, d, for_bwd=False)
    fm.flashmask_classify(mask, B, N, ws)
    for layer in range(3):
        q, k, v, _ = W.make_qkv(B, H, N, d, seed=40 + layer)
        o, lse = fm.flashmask_fwd(q.cuda(), k.cuda(), v.cuda(), mask, ws, ws_classified=True)
        o_ref, lse_ref = A.forward(q, k, v, spec, 1 / math.sqrt(d))
        check_forward(to_np(o), to_np(lse), o_ref, lse_ref, f"layer {layer}")
    st, site = fm.flashmask_check_status(ws)
    assert st == fm.FM_OK, (st, site)


def test_forwards_on_two_streams_with_their_own_workspaces():
    # the persistent forward takes its work items from a counter in the
    # workspace: two forwards in flight at once on two streams, each with its
    # own workspace, must not take each other's items. Each item's arithmetic
    # does not depend on which CTA runs it, so the results must be bit-equal
    # to the same two forwards run one after the other; V is halved so that
    # |O| stays below 4, where bf16 output rounding (half an ulp <= 2^-7)
    # keeps within the absolute O tolerance against the oracle.
    fm = need_gpu()
    B, H, N, d = 1, 8, 2048, 128
    specs = [W.document_bounds(B, 1, [700, 900, 448]), W.causal_bounds(B, 1, N)]
    inputs = []
    for i in range(2):
        q, k, v, _ = W.make_qkv(B, H, N, d, seed=60 + i)
        inputs.append((q, k, (v.float() * 0.5).to(torch.bfloat16)))
    masks = [fm.DeviceMask.from_spec(s) for s in specs]
    dev_in = [[x.cuda() for x in qkv] for qkv in inputs]
    # one after the other on the current stream
    seq = []
    for i in range(2):
        ws = fm.alloc_workspace(B, H, 1, N, d, for_bwd=False)
        o, lse = fm.flashmask_fwd(*dev_in[i], masks[i], ws)
        seq.append((o.clone(), lse.clone()))
    # in flight together on two streams
    wss = [fm.alloc_workspace(B, H, 1, N, d, for_bwd=False) for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):  # several rounds, so the two grids overlap on the device
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                outs.append((i, fm.flashmask_fwd(*dev_in[i], masks[i], wss[i],
                                                 stream=streams[i])))
    torch.cuda.synchronize()
    for i in range(2):
        st, site = fm.flashmask_check_status(wss[i])
        assert st == fm.FM_OK, (i, st, site)
    for i, (o, lse) in outs:
        assert torch.equal(o, seq[i][0]), f"stream {i}: O differs from the sequential run"
        assert torch.equal(lse, seq[i][1]), f"stream {i}: LSE differs from the sequential run"
    for i in range(2):
        o_ref, lse_ref = A.forward(*inputs[i], specs[i], 1 / math.sqrt(d))
        check_forward(to_np(seq[i][0]), to_np(seq[i][1]), o_ref, lse_ref, f"forward {i}")


@pytest.mark.parametrize("N,d", [(200, 128), (77, 64)])
def test_ragged_tail_ignores_neighbouring_head(N, d):
    # The short last block of a head is padded by the TMA loads: rows past the
    # head's end read zeros, never the next head's rows. So a neighbouring head
    # full of Inf / NaN must leave this head's outputs and gradients exact
    # (P = 0 on missing keys would still give 0 * Inf = NaN otherwise).
    fm = need_gpu()
    B, H = 1, 3
    spec = W.document_bounds(B, 1, [N // 2, N - N // 2])
    q, k, v, do = W.make_qkv(B, H, N, d, seed=N + 5)
    bad = [x.clone() for x in (q, k, v, do)]
    for x in bad:
        x[0, 1] = float("inf")
        x[0, 1, ::3] = float("nan")
    out = run_path(fm, *bad, spec)
    scale = 1 / math.sqrt(d)
    lts, lte, uts, ute = head_bounds(spec, 0, 0, H)
    for h in (0, 2):  # the finite heads on either side of the poisoned one
        o_ref, lse_ref = A.forward_head(q[0, h], k[0, h], v[0, h], lts, lte, uts, ute, True, scale)
        check_forward(to_np(out["o"][0, h]), to_np(out["lse"][0, h]), o_ref, lse_ref, f"head {h}")
        g_ref = A.backward_head(q[0, h], k[0, h], v[0, h], do[0, h], lts, lte, uts, ute, True, scale)
        for name, g, r in zip("QKV", (out["dq"], out["dk"], out["dv"]), g_ref):
            assert np.isfinite(to_np(g[0, h])).all(), f"d{name} of head {h} not finite"
            check_grad(name, to_np(g[0, h]), r, f"head {h}")
