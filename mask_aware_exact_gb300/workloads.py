"""Seeded synthetic inputs: Q/K/V/dO tensors and column-wise mask bounds.

This module only draws random numbers and writes the four boundary vectors of
each mask family; it holds none of the attention arithmetic. Both the CUDA path
(through the binding and ``bench.py``) and the CPU oracle (through the tests)
take their inputs from here.

Mask encoding ("FlashMask: Efficient and Rich Mask Extension of FlashAttention",
abstract: a column-wise sparse representation with O(N) memory; "FlashMask-3",
abstract: four query-axis boundary vectors indexed by key position). For key
column j the rows i with

    (causal and j > i)  or  LTS[j] <= i < LTE[j]  or  UTS[j] <= i < UTE[j]

are masked; every interval is half-open and an interval with start >= end masks
nothing. Vectors are int32 arrays shaped [B, Hm, N].

Tensor recipe: one ``torch.Generator`` seeded with ``seed`` draws fp32
``randn`` tensors shaped [B, H, N, d] in the order q, k, v, dO; each is then
rounded to bf16. Mask cuts use ``numpy.random.default_rng(seed)``.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class MaskSpec:
    """Boundary vectors of one mask plus the family parameters that made them."""

    family: str
    causal: bool
    lts: np.ndarray  # int32 [B, Hm, N]
    lte: np.ndarray
    uts: np.ndarray | None  # None: no upper interval
    ute: np.ndarray | None
    params: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.lts.shape[0]

    @property
    def Hm(self) -> int:
        return self.lts.shape[1]

    @property
    def N(self) -> int:
        return self.lts.shape[2]


@dataclass
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    seed: int
    mask: MaskSpec
    description: str


def make_qkv(B: int, H: int, N: int, d: int, seed: int = 0):
    """q, k, v, dO as bf16 CPU tensors [B, H, N, d], drawn in that order."""
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(4):
        out.append(torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(torch.bfloat16))
    return tuple(out)


# ----------------------------------------------------------------- cut recipes
def cuts_min_length(total: int, parts: int, min_len: int, rng: np.random.Generator) -> list[int]:
    """Split ``total`` into ``parts`` lengths by drawing parts-1 distinct cut
    points from 1..total-1, sorted, redrawn until every length is >= min_len."""
    while True:
        cuts = np.sort(rng.choice(np.arange(1, total), parts - 1, replace=False))
        edges = np.concatenate([[0], cuts, [total]])
        lens = np.diff(edges)
        if lens.min() >= min_len:
            return [int(x) for x in lens]


def lengths_uniform(total: int, lo: int, hi: int, rng: np.random.Generator) -> list[int]:
    """Draw lengths uniformly from [lo, hi] until their sum reaches ``total``;
    the last one is truncated so the lengths sum to exactly ``total``."""
    lens: list[int] = []
    s = 0
    while s < total:
        x = int(rng.integers(lo, hi + 1))
        x = min(x, total - s)
        lens.append(x)
        s += x
    return lens


# ----------------------------------------------------------------- encoders
def _empty(B: int, Hm: int, N: int) -> tuple[np.ndarray, np.ndarray]:
    return (np.full((B, Hm, N), N, dtype=np.int32), np.full((B, Hm, N), N, dtype=np.int32))


def causal_bounds(B: int, Hm: int, N: int) -> MaskSpec:
    """Plain causal: the causal flag alone; both intervals empty."""
    lts, lte = _empty(B, Hm, N)
    return MaskSpec("causal", True, lts, lte, None, None, {})


def document_bounds(B: int, Hm: int, lengths: list[int]) -> MaskSpec:
    """Causal attention within packed documents: a key in the document that
    ends at e is masked for every row i >= e."""
    N = int(sum(lengths))
    lts = np.empty(N, dtype=np.int32)
    s = 0
    for L in lengths:
        lts[s:s + L] = s + L
        s += L
    lts = np.broadcast_to(lts, (B, Hm, N)).copy()
    lte = np.full((B, Hm, N), N, dtype=np.int32)
    return MaskSpec("document", True, lts, lte, None, None, {"lengths": list(lengths)})


def share_question_bounds(B: int, Hm: int, q_len: int, answers: list[int]) -> MaskSpec:
    """Question of q_len tokens followed by answers; each answer attends the
    question and itself (causally), never another answer."""
    N = q_len + int(sum(answers))
    lts = np.full(N, N, dtype=np.int32)
    s = q_len
    for L in answers:
        lts[s:s + L] = s + L
        s += L
    lts = np.broadcast_to(lts, (B, Hm, N)).copy()
    lte = np.full((B, Hm, N), N, dtype=np.int32)
    return MaskSpec("share_question", True, lts, lte, None, None,
                    {"question": q_len, "answers": list(answers)})


def window_prefix_bounds(B: int, Hm: int, N: int, window: int, prefix: int) -> MaskSpec:
    """Causal sliding window of ``window`` keys (diagonal included) plus a
    global bidirectional prefix of ``prefix`` tokens, with causal=False:
    prefix keys are seen by every row; a key j >= prefix is masked for rows
    i < j (upper interval [0, j)) and rows i >= j + window (lower interval)."""
    j = np.arange(N, dtype=np.int64)
    in_prefix = j < prefix
    lts = np.where(in_prefix, N, np.minimum(j + window, N)).astype(np.int32)
    lte = np.full(N, N, dtype=np.int32)
    uts = np.zeros(N, dtype=np.int32)
    ute = np.where(in_prefix, 0, j).astype(np.int32)
    bc = lambda a: np.broadcast_to(a, (B, Hm, N)).copy()
    return MaskSpec("window_prefix", False, bc(lts), bc(lte), bc(uts), bc(ute),
                    {"window": window, "prefix": prefix})


def bidirectional_document_bounds(B: int, Hm: int, lengths: list[int]) -> MaskSpec:
    """Full (non-causal) attention within packed documents, causal=False: a key
    in the document [s, e) is masked for rows before the document (upper
    interval [0, s)) and rows after it (lower interval [e, N))."""
    N = int(sum(lengths))
    lts = np.empty(N, dtype=np.int32)
    ute = np.empty(N, dtype=np.int32)
    s = 0
    for L in lengths:
        lts[s:s + L] = s + L
        ute[s:s + L] = s
        s += L
    bc = lambda a: np.broadcast_to(a, (B, Hm, N)).copy()
    lte = np.full(N, N, dtype=np.int32)
    uts = np.zeros(N, dtype=np.int32)
    return MaskSpec("bidirectional_document", False, bc(lts), bc(lte), bc(uts), bc(ute),
                    {"lengths": list(lengths)})


def block_causal_bounds(B: int, Hm: int, N: int, block: int) -> MaskSpec:
    """Causal at block granularity (a block-sparse pattern), causal=False: a key
    in block c = j // block is masked for the rows of earlier blocks (upper
    interval [0, c * block)) and seen by every row from its block on."""
    j = np.arange(N, dtype=np.int64)
    ute = ((j // block) * block).astype(np.int32)
    bc = lambda a: np.broadcast_to(a, (B, Hm, N)).copy()
    lts = np.full(N, N, dtype=np.int32)
    return MaskSpec("block_causal", False, bc(lts), bc(lts.copy()), bc(np.zeros(N, np.int32)),
                    bc(ute), {"block": block})


def block_sparse_runs(N: int, block: int, seed: int, global_blocks: int = 1):
    """Seeded block-sparse pattern: for every key block c (``block`` keys) a run
    [a_c, b_c] of query blocks that see it, drawn from
    ``numpy.random.default_rng(seed)`` with a_c uniform in [0, c] and b_c
    uniform in [c, nb - 1] (so the diagonal block stays visible); the first
    ``global_blocks`` key blocks are seen by every query block (a = 0,
    b = nb - 1). Returns int lists (a, b) of length nb = ceil(N / block)."""
    rng = np.random.default_rng(seed)
    nb = (N + block - 1) // block
    a, b = [], []
    for c in range(nb):
        if c < global_blocks:
            a.append(0)
            b.append(nb - 1)
        else:
            a.append(int(rng.integers(0, c + 1)))
            b.append(int(rng.integers(c, nb)))
    return a, b


def block_sparse_bounds(B: int, Hm: int, N: int, block: int, seed: int,
                        global_blocks: int = 1) -> MaskSpec:
    """Block-sparse mask in which every key block is seen by one contiguous run
    of query blocks (``block_sparse_runs``), causal=False: a key in block c
    masks the rows before its run (upper interval [0, a_c * block)) and the
    rows after it (lower interval [(b_c + 1) * block, N)). Patterns in which a
    key block is seen by two separate runs need more than two intervals per
    column and are not representable in this encoding."""
    a, b = block_sparse_runs(N, block, seed, global_blocks)
    c = np.arange(N) // block
    ute = (np.asarray(a, np.int64)[c] * block).astype(np.int32)
    lts = np.minimum((np.asarray(b, np.int64)[c] + 1) * block, N).astype(np.int32)
    bc = lambda x: np.broadcast_to(x, (B, Hm, N)).copy()
    return MaskSpec("block_sparse", False, bc(lts), bc(np.full(N, N, np.int32)),
                    bc(np.zeros(N, np.int32)), bc(ute),
                    {"block": block, "seed": seed, "global_blocks": global_blocks,
                     "runs": (a, b)})


def stack_heads(specs: list[MaskSpec]) -> MaskSpec:
    """One mask per head (Hm = len(specs)): the specs' [B, 1, N] vectors side by
    side. All must share B, N and the causal flag; a spec without an upper
    interval contributes an empty one."""
    causal = specs[0].causal
    assert all(s.causal == causal for s in specs)
    def up(s, which):
        v = getattr(s, which)
        if v is not None:
            return v
        return np.zeros_like(s.lts)
    any_upper = any(s.uts is not None for s in specs)
    cat = lambda name: np.concatenate([getattr(s, name) for s in specs], axis=1)
    uts = np.concatenate([up(s, "uts") for s in specs], axis=1) if any_upper else None
    ute = np.concatenate([up(s, "ute") for s in specs], axis=1) if any_upper else None
    return MaskSpec("per_head", causal, cat("lts"), cat("lte"), uts, ute,
                    {"families": [s.family for s in specs]})


def random_bounds(B: int, Hm: int, N: int, causal: bool, seed: int, upper: bool = True) -> MaskSpec:
    """Adversarial bounds for fuzzing: values anywhere in [-8, N+8], empty and
    reversed intervals, intervals touching 0 and N, overlapping LT/UT."""
    rng = np.random.default_rng(seed)
    def vec():
        kind = rng.integers(0, 4, size=(B, Hm, N))
        a = rng.integers(-8, N + 9, size=(B, Hm, N))
        b = rng.integers(-8, N + 9, size=(B, Hm, N))
        a = np.where(kind == 1, 0, a)          # touches 0
        b = np.where(kind == 2, N, b)          # touches N
        s = np.minimum(a, b)
        e = np.maximum(a, b)
        swap = kind == 3                       # reversed (empty) interval
        return np.where(swap, e, s).astype(np.int32), np.where(swap, s, e).astype(np.int32)
    lts, lte = vec()
    uts, ute = vec() if upper else (None, None)
    return MaskSpec("random", causal, lts, lte, uts, ute, {"seed": seed})


# ----------------------------------------------------------------- the five workloads
def workload(idx: int) -> Workload:
    """The five synthetic workloads (index 0..4), each with seed 0."""
    seed = 0
    if idx == 0:
        rng = np.random.default_rng(seed)
        lens = cuts_min_length(256, 3, 32, rng)
        return Workload("document3_b1h2n256d64", 1, 2, 256, 64, seed,
                        document_bounds(1, 1, lens),
                        "B=1 H=2 N=256 d=64, causal document mask, 3 packed docs (min 32)")
    if idx == 1:
        return Workload("causal_b4h16n8192d128", 4, 16, 8192, 128, seed,
                        causal_bounds(4, 1, 8192),
                        "B=4 H=16 N=8192 d=128, plain causal mask")
    if idx == 2:
        rng = np.random.default_rng(seed)
        lens = lengths_uniform(32768, 512, 8192, rng)
        return Workload("document_b1h32n32768d128", 1, 32, 32768, 128, seed,
                        document_bounds(1, 1, lens),
                        "B=1 H=32 N=32768 d=128, causal document mask, doc lengths U[512,8192]")
    if idx == 3:
        rng = np.random.default_rng(seed)
        answers = cuts_min_length(12288, 4, 512, rng)
        return Workload("share_question_b2h32n16384d128", 2, 32, 16384, 128, seed,
                        share_question_bounds(2, 1, 4096, answers),
                        "B=2 H=32 N=16384 d=128, share-question mask, question 4096 + 4 answers")
    if idx == 4:
        return Workload("window_prefix_b1h8n131072d128", 1, 8, 131072, 128, seed,
                        window_prefix_bounds(1, 1, 131072, 4096, 2048),
                        "B=1 H=8 N=131072 d=128, causal sliding window 4096 + global prefix 2048")
    raise IndexError(idx)


WORKLOAD_NAMES = [
    "document3_b1h2n256d64",
    "causal_b4h16n8192d128",
    "document_b1h32n32768d128",
    "share_question_b2h32n16384d128",
    "window_prefix_b1h8n131072d128",
]
