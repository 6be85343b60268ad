"""OCP 8-bit floating point, E4M3 variant, written from the format's definition.

Test infrastructure only (see the package docstring).

The pages ask for an 8-bit KV cache ("Why a Second Kind of Engine: Batching, Paged Attention
and Throughput", section "The memory that concurrency actually costs": quantising the cache to
eight bits roughly halves it; "08 serving many users", section "Static or continuous": FP8 KV
adds KV capacity).  They do not fix the encoding; the plainest reading is the OCP OFP8 E4M3
format, which this module restates:

* bit 7 is the sign, bits 6..3 the exponent field e (bias 7), bits 2..0 the mantissa m;
* e = 0: subnormal, value m * 2**-9 (so 0x00 is +0 and 0x80 is -0);
* e = 1..15: normal, value 2**(e-7) * (1 + m/8), except e = 15, m = 7 (S.1111.111) is NaN;
* there are no infinities; the largest finite magnitude is 2**8 * 1.75 = 448.

Encoding (``encode_f32``) rounds an fp32 value to the nearest finite E4M3 value, ties to the
code with an even mantissa, and saturates magnitudes above 448 (including infinities) to 448;
NaN encodes as 0x7F.
"""

from __future__ import annotations

import numpy as np


def decode(codes) -> np.ndarray:
    """E4M3 byte(s) -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m, -9)
    val = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)


_POS = decode(np.arange(127, dtype=np.uint8))  # codes 0x00..0x7E, increasing, all finite
assert np.all(np.diff(_POS) > 0)


def encode_f32(x) -> np.ndarray:
    """fp32 value(s) -> E4M3 codes: round to nearest even, saturate to +-448, NaN -> 0x7F."""
    xf = np.asarray(x, dtype=np.float32)
    a = np.abs(xf).astype(np.float64)  # exact widening
    neg = np.signbit(xf)
    nan = np.isnan(xf)
    a = np.where(nan, 0.0, a)
    hi = np.searchsorted(_POS, a, side="left")          # _POS[hi-1] < a <= _POS[hi]
    sat = hi >= _POS.shape[0]                            # a > 448
    hi_c = np.minimum(hi, _POS.shape[0] - 1)
    lo_c = np.maximum(hi_c - 1, 0)
    hi_v = _POS[hi_c]
    lo_v = _POS[lo_c]
    mid = (lo_v + hi_v) * 0.5                            # exact in fp64
    pick_hi = (a > mid) | ((a == mid) & ((hi_c & 1) == 0))
    code = np.where(pick_hi, hi_c, lo_c)
    code = np.where(a == hi_v, hi_c, code)
    code = np.where(sat, _POS.shape[0] - 1, code)
    code = np.where(hi == 0, 0, code)                    # a == 0
    out = (code | np.where(neg, 0x80, 0)).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), out).astype(np.uint8)
