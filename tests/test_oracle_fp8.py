"""Pins of the 8-bit (E4M3) cache oracle against the format's definition:
bit-field values, round trips, ties to the even code, saturation, NaN, and a
brute-force nearest search written independently of the oracle's."""

import numpy as np
import pytest

from oracle import fp8

V = fp8.e4m3_values()


def test_table_from_the_bit_fields():
    assert V[0x00] == 0.0 and np.signbit(V[0x80])
    assert V[0x01] == 2.0 ** -9 and V[0x07] == 7 * 2.0 ** -9      # subnormals
    assert V[0x08] == 2.0 ** -6                                   # smallest normal
    assert V[0x30] == 0.5 and V[0x38] == 1.0 and V[0xC0] == -2.0
    assert V[0x7E] == 448.0 and V[0xFE] == -448.0                 # largest finite
    assert np.isnan(V[0x7F]) and np.isnan(V[0xFF])
    assert np.isnan(V).sum() == 2
    pos = V[:0x7F]
    assert np.all(np.diff(pos) > 0)                               # codes sort by value


def test_every_finite_value_round_trips():
    codes = np.array([c for c in range(256) if not np.isnan(V[c])])
    assert np.array_equal(fp8.e4m3_encode(V[codes]), codes.astype(np.uint8))


@pytest.mark.parametrize("x,code", [
    (1.0625, 0x38),          # halfway 1.0 / 1.125: even code 0x38
    (1.1875, 0x3A),          # halfway 1.125 / 1.25: even code 0x3a
    (2.0 ** -10, 0x00),      # halfway 0 / smallest subnormal: 0
    (3 * 2.0 ** -10, 0x02),  # halfway 2^-9 / 2^-8: 0x02
    (-1.0625, 0xB8),
    (449.0, 0x7E), (464.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE),     # saturate to finite
    (1.05, 0x38), (1.07, 0x39), (1.1, 0x39),
])
def test_rounding_and_saturation(x, code):
    assert int(fp8.e4m3_encode(np.array([x]))[0]) == code


def test_nan_and_signed_zero():
    c = fp8.e4m3_encode(np.array([np.nan, -0.0, 0.0, -1e-30]))
    assert c.tolist() == [0x7F, 0x80, 0x00, 0x80]


def _brute(y):
    # nearest finite code by exhaustive distance, ties to the even code;
    # magnitudes past 448 clamp to 448
    finite = [c for c in range(256) if not np.isnan(V[c])]
    out = []
    for v in y:
        v = max(-448.0, min(448.0, v))
        d = [abs(V[c] - v) for c in finite]
        best = min(d)
        cands = [c for c, dc in zip(finite, d) if dc == best]
        if v == 0:
            cands = [0x80 if np.signbit(v) else 0x00]
        cands = [c for c in cands if (c & 0x80) == (0x80 if v < 0 else 0)] or cands
        even = [c for c in cands if c % 2 == 0]
        out.append((even or cands)[0])
    return np.array(out, dtype=np.uint8)


def test_matches_brute_force_nearest():
    rng = np.random.default_rng(8)
    y = np.concatenate([rng.standard_normal(400) * 3, rng.standard_normal(200) * 300,
                        rng.standard_normal(100) * 0.01, (V[1:0x7E] + V[2:0x7F]) / 2])
    assert np.array_equal(fp8.e4m3_encode(y), _brute(y.tolist()))


def test_quantize_multiplies_by_the_rounded_reciprocal():
    assert int(fp8.quantize(np.array([3.0]), 0.5)[0]) == 0x4C     # 6.0 = 1.5 * 2^2
    # the reciprocal and the product are float32 roundings
    x = np.array([1.0000001], dtype=np.float32)
    s = 3.0
    y = np.float32(x[0]) * (np.float32(1.0) / np.float32(s))
    assert int(fp8.quantize(x, s)[0]) == int(fp8.e4m3_encode(np.array([float(y)]))[0])


def test_dequantized_relative_error_bound():
    # normal range: |error| <= half a unit in the last place = 2^-4 relative
    rng = np.random.default_rng(9)
    x = rng.uniform(2.0 ** -6, 448.0, 2000) * rng.choice([-1, 1], 2000)
    back = fp8.dequantize(fp8.quantize(x, 1.0), 1.0)
    assert np.all(np.abs(back - x) <= np.abs(x) * 2.0 ** -4)
    s = 0.037
    back = fp8.dequantize(fp8.quantize(x * s, s), s)
    assert np.all(np.abs(back - x * s) <= np.abs(x * s) * 2.0 ** -4 * 1.0001)


def test_write_kv_quantises_rows_and_skips_negative_slots():
    kc = np.zeros((2, 2, 1, 4), np.uint8)
    k = np.array([[[1.0, 2.0, 448.0, -0.5]], [[9.0, 9.0, 9.0, 9.0]], [[0.0, 1.0625, 3.0, 1e9]]])
    out_k, out_v = fp8.write_kv(kc, kc, k, -k, [1, -1, 2], 2, 1.0, 2.0)
    assert out_k.reshape(4, 4).tolist()[0] == [0, 0, 0, 0]
    assert out_k.reshape(4, 4).tolist()[1] == [0x38, 0x40, 0x7E, 0xB0]
    assert out_k.reshape(4, 4).tolist()[2] == [0x00, 0x38, 0x44, 0x7E]
    assert out_v.reshape(4, 4).tolist()[1] == [0xB0, 0xB8, 0xF6, 0x28]
