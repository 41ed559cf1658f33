"""Oracle: the 8-bit E4M3 float format of an FP8 paged KV cache (test infrastructure only).

"EAGLE-3 paper explainer" (0h-n0), operations section, model-optimisation list: quantisation
and the tuning of the PagedAttention KV cache are listed as ways to cut GPU memory. The page
names no format. Reading: the cache holds E4M3 codes as the OCP 8-bit floating-point format
defines them:
- a sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
- exponent field 0 holds the subnormals m/8 * 2^-6;
- S.1111.111 is NaN, and there are no infinities, so the largest magnitude is 1.75 * 2^8 = 448.

Each KV head g carries an fp32 scale for K and one for V: a stored code c stands for
decode(c) * scale[g].

Quantisation (the commit of new rows) takes y = x / scale in fp32 (one IEEE division). It then
rounds y to the nearest E4M3 value, ties to the even code, and saturates finite values beyond
448 to +-448. A negative value that rounds to zero keeps its sign (code 0x80).
"""

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """uint8 codes -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    out = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


# the 127 non-negative finite magnitudes, code 0 .. 126, in increasing order
_GRID = e4m3_decode(np.arange(127, dtype=np.uint8))


def e4m3_encode(x):
    """float32 values -> uint8 codes: round to nearest, ties to the even code, finite values
    beyond 448 saturate, NaN -> 0x7F."""
    x = np.asarray(x, np.float32)
    a = np.abs(x.astype(np.float64))
    hi = np.clip(np.searchsorted(_GRID, a, side="left"), 0, 126)   # first grid value >= a
    lo = np.maximum(hi - 1, 0)
    d_hi = _GRID[hi] - a
    d_lo = a - _GRID[lo]
    take_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(take_lo, lo, hi)
    code = np.where(a >= E4M3_MAX, 126, code)                      # saturation (finite and inf)
    code = code.astype(np.int64) | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def kv_quantize(x, scale):
    """Codes of x / scale, the division in fp32. x: float values (bf16-representable, as the
    tree K/V are); scale: broadcastable fp32 scale."""
    y = np.asarray(x, np.float32) / np.asarray(scale, np.float32)
    return e4m3_encode(y.astype(np.float32))


def kv_dequantize(codes, scale):
    """float64 values of codes * scale (scale broadcast against the codes)."""
    return e4m3_decode(codes) * np.asarray(scale, np.float64)
