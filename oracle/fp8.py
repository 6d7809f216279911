"""FP8 E4M3 codes to values, from the format's definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The FP8 path the pages attribute to FA3 and name for later versions
(ainexis "Tri Dao FlashAttention-4", section 背景; wittx "FlashAttention-4",
closing section) is not specified there. Reading: the OCP 8-bit E4M3 format
("fn": finite only), the format of FA3's FP8 inputs:
* bit 7 sign, bits 6..3 exponent e (bias 7), bits 2..0 mantissa m;
* e = 0: subnormal, value 2^(1 - 7) * m / 8;
* 1 <= e <= 15: normal, value 2^(e - 7) * (1 + m / 8), except e = 15, m = 7,
  which is NaN (there are no infinities); the largest finite value is 448.
Attention with E4M3 inputs is attention on these values times each tensor's
descale factor, so the forward's oracle is :func:`attention_fwd` on them.
"""

from __future__ import annotations

import numpy as np


def e4m3_decode(codes) -> np.ndarray:
    """Values (fp64) of E4M3 codes given as integers 0..255 (any array shape)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag
