"""Pins of the oracle's INT8 codec (CPU only).

The brute force below recomputes every step with exact rational arithmetic
(``fractions.Fraction``) and its own IEEE round-to-nearest-even to float32, so
it does not share numpy's float32 arithmetic with the oracle.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import int8_codec

F32_MAX = Fraction(np.finfo(np.float32).max.item())


def f32_rne(fr: Fraction) -> Fraction:
    """Round an exact rational to the nearest float32 (ties to even), as a Fraction.

    Returns +-inf as ``None`` sentinels are awkward; here overflow returns the
    Python float inf.
    """
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    # fix rounding of the log estimate
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q_exp = max(e - 23, -149)                    # quantum exponent (subnormals: 2^-149)
    q = Fraction(2) ** q_exp
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * q
    if r > F32_MAX:
        return math.inf * sign
    return sign * r


def rint_half_even(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def brute_row(row):
    xs = [Fraction(float(v)) for v in np.asarray(row, np.float32)]
    m = max(abs(v) for v in xs)
    if m == 0:
        return [0] * len(xs), Fraction(0)
    scale = f32_rne(m / 127)
    inv = f32_rne(Fraction(127) / m)
    codes = []
    for v in xs:
        if inv == math.inf:
            c = 0 if v == 0 else (127 if v > 0 else -127)
        else:
            p = f32_rne(v * inv)
            c = 0 if p == 0 else (127 if p == math.inf else (-127 if p == -math.inf else rint_half_even(p)))
            c = max(-127, min(127, c))
        codes.append(c)
    return codes, scale


def _check_against_brute(x):
    codes, scales = int8_codec.quantize_rows(x)
    for r in range(x.shape[0]):
        bc, bs = brute_row(x[r])
        assert list(codes[r].astype(int)) == bc, f"row {r}"
        assert Fraction(float(scales[r])) == bs, f"row {r}"


def test_brute_force_random_rows():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((24, 128)).astype(np.float32)
    x[3] *= 1e-3
    x[5] *= 1e5
    x[7, 11] = 8.0                         # an outlier row
    _check_against_brute(x)


def test_brute_force_small_and_subnormal_rows():
    rng = np.random.default_rng(1)
    rows = []
    for mag in (1e-30, 1e-36, 2e-37, 1e-39, 3e-45):
        r = (rng.standard_normal(128) * mag).astype(np.float32)
        r[rng.integers(0, 128, 8)] = 0.0
        rows.append(r)
    _check_against_brute(np.stack(rows))


def test_ties_round_half_even():
    # absmax 127 -> inv = 1 and scale = 1 exactly, so x * inv == x.
    row = np.zeros(128, np.float32)
    row[:8] = [127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 126.5, -1.5]
    codes, scale = int8_codec.quantize_rows(row[None])
    assert scale[0] == 1.0
    assert list(codes[0, :8]) == [127, 2, 4, -2, 0, 0, 126, -2]


def test_zero_row():
    codes, scale = int8_codec.quantize_rows(np.zeros((2, 128), np.float32))
    assert np.all(codes == 0) and np.all(scale == 0)


def test_absmax_maps_to_127_and_range():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((200, 128)).astype(np.float32)
    codes, _ = int8_codec.quantize_rows(x)
    j = np.argmax(np.abs(x), axis=1)
    top = codes[np.arange(200), j].astype(int)
    np.testing.assert_array_equal(top, np.where(x[np.arange(200), j] > 0, 127, -127))
    assert codes.min() >= -127 and codes.max() <= 127


def test_integer_rows_round_trip_exactly():
    rng = np.random.default_rng(3)
    x = rng.integers(-127, 128, (10, 128)).astype(np.float32)
    x[:, 0] = 127.0
    codes, scale = int8_codec.quantize_rows(x)
    np.testing.assert_array_equal(codes.astype(np.float32), x)
    np.testing.assert_array_equal(scale, np.ones(10, np.float32))


@pytest.mark.parametrize("seed", [4, 5])
def test_round_trip_error_within_half_scale(seed):
    # Invariant 5: |x - q * scale| <= scale / 2, up to the float32 roundings of
    # inv (|x * inv - 127 x / m| <= 127 * 2^-23 codes) and of scale
    # (|q| * |scale - m / 127| <= m * 2^-24), together below scale * 2^-15.
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((500, 128)).astype(np.float32)
    hit = rng.random((500, 128)) < 0.01
    x = np.where(hit, np.sign(rng.standard_normal((500, 128))) * 8.0, x).astype(np.float32)
    codes, scale = int8_codec.quantize_rows(x)
    err = np.abs(x.astype(np.float64) - int8_codec.dequantize_rows(codes, scale))
    bound = scale.astype(np.float64)[:, None] / 2 * (1 + 2.0 ** -14)
    assert np.all(err <= bound)
