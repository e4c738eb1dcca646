"""FP8 (E4M3) KV storage: the code of a value and the value of a code.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages ask for fewer bytes moved: the memory-systems notes ("Core
Ideas" 1) count quantization among the optimizations judged by bytes moved,
and "PagedAttention Kernel：大模型推理优化的显存管理革新" section 6 computes
in FP16 and accumulates in FP32.  The reading taken here: keys and values are
stored as 8-bit floats of the E4M3 format, one scale per cache (k_scale,
v_scale).

E4M3 (as the OCP 8-bit floating point specification defines it): bit 7 is
the sign, bits 6..3 the exponent e (bias 7), bits 2..0 the mantissa m.
  e = 0:        value (-1)^s · m · 2^-9                 (zero and subnormals)
  e = 1..15:    value (-1)^s · (1 + m/8) · 2^(e-7)      (normals)
  e = 15, m = 7: NaN (there is no infinity); the largest finite is 448.

Storing x with scale c: code = RNE-to-E4M3(x / c) with the division in
fp32 (IEEE, round to nearest) and saturation, i.e. a finite quotient beyond
±448 (or an infinity) stores ±448; NaN stores a NaN code.  Reading a code
gives decode(code) · c, exact in fp64.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _decode_table() -> np.ndarray:
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            out[code] = np.nan
        elif e == 0:
            out[code] = sign * m * 2.0 ** -9
        else:
            out[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


DECODE = _decode_table()  # value of every code, fp64


def decode(codes: np.ndarray) -> np.ndarray:
    """fp64 value of E4M3 codes (uint8)."""
    return DECODE[np.asarray(codes, dtype=np.uint8)]


def encode(x: np.ndarray) -> np.ndarray:
    """E4M3 codes of fp32 values, round to nearest, ties to the even code
    (the one with an even mantissa), saturating to ±448; NaN gives 0x7F
    (0xFF when the sign bit is set)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    sign = np.signbit(x).astype(np.uint8) << np.uint8(7)
    mag = np.zeros(a.shape, dtype=np.uint8)
    # The non-negative codes 0x00..0x7E are in increasing order of value.
    pos = DECODE[:0x7F]
    # index of the largest representable value <= a (a < 448 here)
    fin = np.isfinite(a) & (a < E4M3_MAX)
    lo = np.searchsorted(pos, a[fin], side="right") - 1
    lo_val = pos[lo]
    hi_val = pos[lo + 1]
    d_lo = a[fin] - lo_val
    d_hi = hi_val - a[fin]
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((lo & 1) == 1))  # tie: the even mantissa
    mag[fin] = np.where(take_hi, lo + 1, lo).astype(np.uint8)
    mag[~fin] = 0x7E  # >= 448 or infinite: saturate
    mag[np.isnan(a)] = 0x7F
    return mag | sign


def quantize(x: np.ndarray, scale: float) -> np.ndarray:
    """Codes storing fp32 values ``x`` with ``scale``: encode(x / scale),
    the quotient rounded to fp32."""
    q = np.asarray(x, dtype=np.float32) / np.float32(scale)
    return encode(q)
