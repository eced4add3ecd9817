"""Pins the e4m3 rounding and the block quantisation of oracle.fp8 against what
the format's definition and an independent library conversion fix: torch's
float8_e4m3fn cast (round to nearest even, no saturation) on in-range values, a
brute-force nearest-value search over the 254 finite codes, the format's
landmark values, and the error bounds of round-to-nearest with 3 mantissa
bits."""
import numpy as np
import pytest
import torch

from oracle import fp8 as F


def finite_table():
    t = F.e4m3_table()
    return t[np.isfinite(t)]


def test_table_landmarks():
    t = F.e4m3_table()
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isfinite(t).sum() == 254
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0  # largest finite
    assert t[0x01] == 2.0 ** -9                   # smallest subnormal
    assert t[0x08] == 2.0 ** -6                   # smallest normal
    assert t[0x38] == 1.0 and t[0x39] == 1.125
    assert np.all(np.diff(t[:0x7F]) > 0)          # codes 0..0x7E increase
    assert np.array_equal(t[0x80:0xFF], -t[0x00:0x7F])


def test_table_matches_torch_float8():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    t = F.e4m3_table()
    fin = np.isfinite(t)
    assert np.array_equal(np.isnan(lib), ~fin)
    assert np.array_equal(lib[fin], t[fin])


def test_round_matches_torch_cast_in_range():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, s, 20000) for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x[np.abs(x) <= 448.0]
    # every midpoint between neighbouring finite values (the ties)
    pos = np.sort(finite_table()[finite_table() >= 0])
    mids = (pos[1:] + pos[:-1]) / 2
    x = np.concatenate([x, mids, -mids]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(F.e4m3_round(x.astype(np.float64)), lib)


def brute_round(x):
    """Nearest finite value; on a tie the one whose code has an even mantissa."""
    t = F.e4m3_table()
    out = np.empty(len(x))
    for n, xv in enumerate(x):
        if abs(xv) >= 448.0:
            out[n] = np.copysign(448.0, xv)
            continue
        dist = np.abs(t - xv)
        dist[~np.isfinite(t)] = np.inf
        best = np.flatnonzero(dist == np.nanmin(dist))
        even = [c for c in best if (c & 1) == 0]
        out[n] = t[even[0] if even else best[0]]
    return out


def test_round_brute_force():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-480, 480, 3000), rng.normal(0, 0.02, 3000),
                        rng.uniform(-2.0 ** -5, 2.0 ** -5, 2000)])
    pos = np.sort(finite_table()[finite_table() >= 0])
    mids = (pos[1:] + pos[:-1]) / 2
    x = np.concatenate([x, mids, -mids, pos, -pos])
    assert np.array_equal(F.e4m3_round(x), brute_round(x))


@pytest.mark.parametrize("x,want", [
    (1.0625, 1.0),        # tie between 1.0 (mantissa 000) and 1.125 (001): even
    (1.1875, 1.25),       # tie between 1.125 (001) and 1.25 (010): even
    (2.0 ** -10, 0.0),    # tie between 0 and the smallest subnormal: even (0)
    (3 * 2.0 ** -10, 2.0 ** -8),  # tie between 2^-9 (m=1) and 2^-8 (m=2)
    (448.0, 448.0), (460.0, 448.0), (500.0, 448.0), (1e9, 448.0),  # saturating
    (-1.0625, -1.0), (-500.0, -448.0), (0.0, 0.0),
])
def test_round_special_values(x, want):
    assert F.e4m3_round(np.array([x]))[0] == want


def test_round_error_bounds():
    # round to nearest with 3 mantissa bits: relative error <= 2^-4 on normals,
    # absolute error <= 2^-10 in the subnormal range
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.uniform(2.0 ** -6, 448, 50000), rng.uniform(0, 2.0 ** -6, 5000)])
    r = F.e4m3_round(x)
    norm = x >= 2.0 ** -6
    assert np.all(np.abs(r[norm] - x[norm]) <= 2.0 ** -4 * x[norm])
    assert np.all(np.abs(r[~norm] - x[~norm]) <= 2.0 ** -10)


def test_quantize_rows_blocks_and_scales():
    rng = np.random.default_rng(3)
    N, d = 300, 128  # blocks of 128, 128 and a short one of 44 rows
    x = rng.normal(0, 1, (N, d)).astype(np.float32)
    x[128:256] = 0.0  # an all-zero block
    codes, scales, deq = F.quantize_rows(x)
    assert scales.dtype == np.float32 and scales.shape == (3,)
    for t, blk in enumerate((slice(0, 128), slice(128, 256), slice(256, 300))):
        am = np.abs(x[blk]).max()
        if am == 0:
            assert scales[t] == 1.0 and np.all(codes[blk] == 0)
            continue
        assert scales[t] == np.float32(np.float32(am) / np.float32(448.0))
        assert np.abs(codes[blk]).max() == 448.0  # the largest element maps to 448
        assert set(np.unique(codes[blk])) <= set(finite_table())
        # dequantised values within the rounding bound of the originals
        s = np.float64(scales[t])
        err = np.abs(deq[blk] - x[blk])
        bound = np.maximum(2.0 ** -4 * np.abs(x[blk]), 2.0 ** -10 * s) * (1 + 1e-6)
        assert np.all(err <= bound)


def test_quantize_head_single_scale():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 3, (200, 128)).astype(np.float32)
    codes, s, deq = F.quantize_head(x)
    assert s == np.float32(np.float32(np.abs(x).max()) / np.float32(448.0))
    assert np.abs(codes).max() == 448.0
    assert np.all(np.abs(deq - x) <= np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s) * (1 + 1e-6))
