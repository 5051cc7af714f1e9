"""OCP FP8 E4M3 codec (the "fn" variant: no infinities, one NaN per sign).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages fix an FP8 latent cache of one byte per element ("G5 MLA KV
访存建模设计规格" 用例说明, use case 1) but not the format.  The format used is
the OCP 8-bit floating point E4M3 encoding: 1 sign bit, 4 exponent bits with
bias 7, 3 mantissa bits; exponent field 0 is subnormal (value m/8 * 2^-6);
S.1111.111 is NaN; the largest finite magnitude is S.1111.110 = 448.
"""
from __future__ import annotations

import numpy as np


def decode(codes) -> np.ndarray:
    """Exact float64 value of each e4m3 code (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    val = sign * val
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def codebook() -> np.ndarray:
    """Values of the 256 codes, index = code."""
    return decode(np.arange(256, dtype=np.uint8))


def encode(x) -> np.ndarray:
    """Encode float values as e4m3, round to nearest with ties to the even code, saturating.

    Finite inputs whose magnitude exceeds 448 encode as +-448 (0x7E / 0xFE);
    NaN encodes as 0x7F.  The rounding is done on the exact value of the input:
    the candidates are the two neighbouring representable magnitudes and the
    nearer one wins, the one with an even mantissa on a tie.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    mags = decode(np.arange(0x7F, dtype=np.uint8))         # codes 0x00..0x7E, increasing
    idx_hi = np.searchsorted(mags, np.minimum(a, 448.0), side="left")
    idx_hi = np.clip(idx_hi, 0, 0x7E)
    idx_lo = np.clip(idx_hi - 1, 0, 0x7E)
    d_lo = np.abs(a - mags[idx_lo])
    d_hi = np.abs(mags[idx_hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((idx_hi & 1) == 0))
    code = np.where(pick_hi, idx_hi, idx_lo).astype(np.int64)
    code = np.where(a >= 448.0, 0x7E, code)
    code = np.where(sign, code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)
