"""Per-(token, head) absmax FP8 (E4M3) codec for K/V rows (oracle; test infrastructure only).

The comparison cache format next to the INT8 one: the pages store the KV
cache in INT8 (Hy-Nomas auf einer RTX 4090, section "Das Single-GPU-Preset",
``kv_cache_quantization: int8``) and name no FP8 cache; this variant keeps the
INT8 layout (one byte per value, one float32 scale per row of ``head_dim``
values) with the byte read as an OCP E4M3 float (1 sign, 4 exponent bits with
bias 7, 3 mantissa bits; no infinities; largest finite 448; the all-ones
magnitude 0x7F is NaN).  Written out in IEEE float32 so every bit is defined:

    m     = max_i |x_i|                      (exact)
    scale = fl32(m / 448)                    (IEEE division, round to nearest)
    inv   = fl32(448 / m)                    (IEEE division, round to nearest)
    y_i   = fl32(x_i * inv)                  (IEEE product)
    q_i   = E4M3(y_i)   round to nearest, ties to the even code, magnitudes
                        above 448 saturate to 448, the sign of y_i kept (a
                        negative value that rounds to zero is 0x80)

with the conventions of the INT8 codec for a row whose ``inv`` overflows
(absmax below ``448 / FLT_MAX``): a NaN product (0 * inf) gives the code 0
and +-inf gives +-448.  An all-zero row has ``scale = 0`` and codes 0 (its
products are all NaN).  Dequantisation is ``x_hat = value(q) * scale``.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
MAX_E4M3 = 448.0


def e4m3_values() -> np.ndarray:
    """Value of every magnitude code 0x00 .. 0x7E (float64); 0x7F is NaN."""
    vals = np.zeros(0x7F, dtype=np.float64)
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals[c] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_VALS = e4m3_values()


def decode(codes: np.ndarray) -> np.ndarray:
    """Float64 value of E4M3 codes (uint8 or int8 bit patterns); 0x7F / 0xFF decode to NaN."""
    c = np.asarray(codes).astype(np.uint8)
    mag = c & 0x7F
    out = np.where(mag == 0x7F, np.nan, _VALS[np.minimum(mag, 0x7E)])
    return np.where(c & 0x80, -out, out)


def round_e4m3(y: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8) of float32 values: nearest, ties to even code, saturating; NaN -> 0."""
    y = np.asarray(y, dtype=F32).astype(np.float64)
    a = np.abs(y)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, MAX_E4M3))
    hi = np.clip(np.searchsorted(_VALS, a, side="left"), 0, 0x7E)   # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_hi = _VALS[hi] - a
    d_lo = a - _VALS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo).astype(np.uint8)
    sign = np.signbit(y) & ~nan
    return np.where(sign, mag | 0x80, mag).astype(np.uint8)


def quantize_rows(x: np.ndarray):
    """Quantise the last axis of ``x`` row by row.

    Returns ``(codes uint8 [..., D], scales float32 [...])``.
    """
    x = np.asarray(x, dtype=F32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        m = np.max(np.abs(x), axis=-1)
        scale = (m / F32(MAX_E4M3)).astype(F32)
        inv = (F32(MAX_E4M3) / m).astype(F32)
        prod = (x * inv[..., None]).astype(F32)
    codes = round_e4m3(prod)
    zero = m == 0
    if np.any(zero):
        scale = np.where(zero, F32(0.0), scale).astype(F32)
    return codes, scale.astype(F32)


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """``x_hat = value(q) * scale`` in float64 (exact: a 4-bit mantissa times a float32)."""
    return decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]
