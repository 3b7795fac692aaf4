"""Per-(token, head) absmax INT8 codec for K/V rows (oracle; test infrastructure only).

The low-memory preset stores the KV cache in INT8 and computes in BF16
(Hy-Nomas auf einer RTX 4090, section "Das Single-GPU-Preset":
``kv_cache_quantization: int8``; the blog.authon.dev install guide repeats the
key in its low-memory config excerpt).  The pages give no formula; the reading
used here is symmetric absmax quantisation with one float32 scale per row of
``head_dim`` values (one token of one head of one block), written out in IEEE
float32 so that every bit of the result is defined:

    m     = max_i |x_i|                      (exact)
    scale = fl32(m / 127)                    (IEEE division, round to nearest)
    inv   = fl32(127 / m)                    (IEEE division, round to nearest)
    q_i   = clamp(rint(fl32(x_i * inv)), -127, 127)   (rint: half to even)

with the conversion conventions of a round-to-nearest float->int instruction:
a NaN product (only ``0 * inf``, when ``inv`` overflows for a row whose absmax
is below ``127 / FLT_MAX``) gives 0 and +-inf gives +-127.  An all-zero row has
``scale = 0`` and codes 0.  Dequantisation is ``x_hat = q * scale``.  The code
-128 is never produced.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def quantize_rows(x: np.ndarray):
    """Quantise the last axis of ``x`` row by row.

    ``x``: float32-representable values, any leading shape, last axis = one row.
    Returns ``(codes int8 [..., D], scales float32 [...])``.
    """
    x = np.asarray(x, dtype=F32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        m = np.max(np.abs(x), axis=-1)                       # exact in float32
        scale = (m / F32(127.0)).astype(F32)                 # IEEE float32 division
        inv = (F32(127.0) / m).astype(F32)                   # inf when m == 0 or tiny
        prod = (x * inv[..., None]).astype(F32)              # IEEE float32 product
        r = np.rint(prod)                                    # half to even
    r = np.where(np.isnan(r), F32(0.0), r)
    r = np.clip(r, -127.0, 127.0)
    codes = r.astype(np.int8)
    zero = m == 0
    if np.any(zero):
        codes[zero] = 0
        scale = np.where(zero, F32(0.0), scale).astype(F32)
    return codes, scale.astype(F32)


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """``x_hat = q * scale`` in float64 (exact: an 8-bit integer times a float32)."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]
