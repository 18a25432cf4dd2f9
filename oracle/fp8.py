"""FP8 (E4M3) storage of the KV cache — oracle side (test infrastructure only).

The pages describe a bf16 cache only; an 8-bit cache is this library's
extension.  The format is the OCP 8-bit floating point E4M3 ("FN") encoding:
1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, subnormals at
exponent 0, no infinities, and S.1111.111 as NaN, so the largest finite
magnitude is 1.75 * 2^8 = 448.

Quantisation of a value x with a per-tensor scale s: y = fp32(fp32(x) * fp32(1 / s))
(both products rounded to float32, the reciprocal rounded once), then the
E4M3 code nearest to y, ties to the even code, magnitudes above 448 clamped
to 448 ("saturate to finite"), NaN to the NaN code.  Dequantisation:
value(code) * s.  Everything here is written from that definition: the code
table is enumerated from the bit fields and rounding is a nearest search
over it.
"""

from __future__ import annotations

import numpy as np

NAN_CODE = 0x7F
MAX_FINITE = 448.0


def e4m3_values() -> np.ndarray:
    """float64 value of each of the 256 codes (NaN for the two NaN codes)."""
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            out[code] = np.nan
        elif e == 0:
            out[code] = sign * (m / 8.0) * 2.0 ** -6
        else:
            out[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_VALUES = e4m3_values()
_POS_CODES = np.arange(0, 0x7F)            # 0x00 .. 0x7e: +0 .. +448, increasing
_POS_VALUES = _VALUES[_POS_CODES]


def e4m3_encode(y) -> np.ndarray:
    """Nearest E4M3 code of each value (ties to the even code, saturating)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), MAX_FINITE)
    nan = np.isnan(y)
    a = np.where(nan, 0.0, a)
    j = np.searchsorted(_POS_VALUES, a)                 # first value >= a
    j_c = np.minimum(j, len(_POS_VALUES) - 1)
    exact = _POS_VALUES[j_c] == a
    lo = np.maximum(j - 1, 0)
    hi = j_c
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    c = np.where(exact, j_c, pick)
    sign = np.where(np.signbit(y), 0x80, 0)
    codes = (sign | _POS_CODES[c]).astype(np.uint8)
    return np.where(nan, NAN_CODE, codes).astype(np.uint8)


def quantize(x, scale: float) -> np.ndarray:
    """E4M3 codes of fp32(x) * fp32(1 / scale) (see the module docstring)."""
    inv = np.float32(1.0) / np.float32(scale)
    y = np.asarray(x, dtype=np.float32) * inv
    return e4m3_encode(y.astype(np.float64))


def dequantize(codes, scale: float) -> np.ndarray:
    """float64 values of codes times the scale."""
    return _VALUES[np.asarray(codes, dtype=np.int64)] * float(scale)


def write_kv(k_codes, v_codes, k, v, slot_mapping, block_size: int, k_scale: float,
             v_scale: float):
    """The scatter of an 8-bit cache: each new token's row is quantised, then stored.

    "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §2.3补充 第一步
    places token t's K/V at slot_mapping[t]; here the stored row is its E4M3
    codes.  A negative slot is skipped.  Returns new code arrays.
    """
    kc = np.array(k_codes, copy=True)
    vc = np.array(v_codes, copy=True)
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        b, off = divmod(int(slot), block_size)
        kc[b, off] = quantize(k[t], k_scale)
        vc[b, off] = quantize(v[t], v_scale)
    return kc, vc
