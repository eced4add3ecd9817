"""e4m3 block quantisation of attention operands (test infrastructure only).

Follows "FlashAttention-3" (abstract: block quantization for FP8 attention):
each block of an operand is divided by its own scale and rounded to FP8, and
the products run on the quantised values. The FP8 format is E4M3 as the OCP
8-bit floating point specification defines it: sign, 4 exponent bits with
bias 7, 3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9; the
one NaN pattern per sign is S.1111.111, so the largest finite value is
1.75 * 2^8 = 448 and there is no infinity.

Readings taken where the page is silent (the CUDA path makes the same ones):
  - blocks: 128 consecutive rows of one head for Q and K (the rows of one
    attention tile), the whole head for V;
  - scale = absmax / 448 (1 for an all-zero block) so that the largest element
    maps to the largest finite e4m3 value;
  - a value becomes e4m3(x * (1 / scale)), rounded to nearest with ties to the
    even mantissa and saturated at +-448. The scale, its reciprocal and the
    product are rounded to fp32 exactly as the kernel rounds them, because
    these fp32 values decide the integer codes (the e4m3 rounding itself is
    exact arithmetic here, in fp64).
Nothing else of the FP8 forward is restated: its score and output products on
the dequantised operands are the fp64 attention of oracle.attention, and the
further rounding of P to e4m3 is bounded in the parity test, not modelled.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_table() -> np.ndarray:
    """Every finite e4m3 value indexed by its byte code (NaN at 0x7F and 0xFF)."""
    vals = np.empty(256)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e, m = (code >> 3) & 0xF, code & 0x7
        if e == 15 and m == 7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * m * 2.0 ** -9
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value of each element (ties to the even mantissa), saturated
    at +-448; the result is returned as fp64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # binade exponent: a = f * 2^E with f in [0.5, 1), so a lies in [2^(E-1), 2^E);
    # below 2^-6 the subnormal spacing 2^-9 applies
    _, E = np.frexp(np.maximum(a, 2.0 ** -6))
    step = np.ldexp(1.0, E - 1 - 3)  # 3 mantissa bits
    r = np.round(a / step) * step  # numpy rounds half to even: the even mantissa
    r = np.minimum(r, E4M3_MAX)
    return np.where(np.signbit(x), -r, r)


def scale_of(absmax) -> np.float32:
    """fp32 scale of a block whose largest magnitude is `absmax` (1 if zero)."""
    m = np.float32(absmax)
    return np.float32(m / np.float32(E4M3_MAX)) if m > 0 else np.float32(1.0)


def quantize_block(x, s: np.float32) -> np.ndarray:
    """e4m3 values of x * (1 / s) with the reciprocal and the product in fp32."""
    inv = np.float32(np.float32(1.0) / s)
    y = np.asarray(x, dtype=np.float32) * inv  # fp32 product, round to nearest
    return e4m3_round(y.astype(np.float64))


def quantize_rows(x, block: int = BLOCK):
    """Per-block quantisation of one head's [N, d] rows (blocks of `block` rows;
    the last may be short). Returns (codes as e4m3 values [N, d], fp32 scales
    [ceil(N / block)], dequantised fp64 values codes * scale)."""
    x = np.asarray(x, dtype=np.float32)
    N = x.shape[0]
    nb = (N + block - 1) // block
    codes = np.empty(x.shape)
    scales = np.empty(nb, dtype=np.float32)
    for t in range(nb):
        blk = x[t * block:(t + 1) * block]
        s = scale_of(np.abs(blk).max() if blk.size else 0.0)
        scales[t] = s
        codes[t * block:(t + 1) * block] = quantize_block(blk, s)
    deq = codes * np.repeat(scales.astype(np.float64), block)[:N, None]
    return codes, scales, deq


def quantize_head(x):
    """One scale for the whole head: (codes [N, d], fp32 scale, dequantised)."""
    x = np.asarray(x, dtype=np.float32)
    s = scale_of(np.abs(x).max() if x.size else 0.0)
    codes = quantize_block(x, s)
    return codes, s, codes * np.float64(s)
