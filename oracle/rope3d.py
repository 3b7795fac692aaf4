"""3D rotary position embedding (oracle, float64; test infrastructure only).

The model card lists "3D RoPE" for the 54-block MMDiT (Hy-Nomas auf einer RTX
4090, section "Modell und Dateien"; the orcarouter.ai explainer, section "Die
Schleife", names 3D rotary position embeddings).  The pages give no formula, so
this module writes out the plainest reading, which the tests pin:

* the head dimension is split into three contiguous chunks of ``d_t, d_h, d_w``
  dims (32/48/48 for 128) at offsets ``0, d_t, d_t + d_h``, one per axis
  (latent frame t, grid row h, grid column w);
* within the chunk of axis ``a`` the pair ``(x[o + 2i], x[o + 2i + 1])`` for
  ``i in [0, d_a / 2)`` is rotated by the angle ``pos_a * f_{a,i}`` with
  ``f_{a,i} = theta ** (-2 i / d_a)``:
  ``(x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos)``;
* a video token at latent frame ``frame`` of the segment, row ``h`` and column
  ``w`` has positions ``(t0 + frame, h, w)``, where ``t0`` is the absolute index
  of the segment's first latent frame (positions continue from the cached
  frames);
* text tokens are not rotated.

Parity unpinned: the interleaved pairing and the per-axis frequency exponent are
conventions the pages do not fix; both alternatives satisfy every invariant the
tests check (norm preservation, shift invariance, identity at position 0), so
they are pinned only by this definition.
"""
from __future__ import annotations

import numpy as np


def axis_frequencies(d_a: int, theta: float) -> np.ndarray:
    """``f_i = theta ** (-2 i / d_a)`` for ``i in [0, d_a / 2)``, float64."""
    if d_a % 2:
        raise ValueError("axis sub-dimension must be even")
    i = np.arange(d_a // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / np.float64(d_a))


def video_positions(frames: int, grid_h: int, grid_w: int, t0: int):
    """Integer (t, h, w) positions of the video tokens, in (frame, h, w) row-major order."""
    f, h, w = np.meshgrid(np.arange(frames), np.arange(grid_h), np.arange(grid_w), indexing="ij")
    return (f.reshape(-1).astype(np.int64) + int(t0), h.reshape(-1).astype(np.int64),
            w.reshape(-1).astype(np.int64))


def rotate(x: np.ndarray, pos_t, pos_h, pos_w, theta: float = 10000.0,
           split=(32, 48, 48)) -> np.ndarray:
    """Rotate rows of ``x`` (``[n][heads][D]`` or ``[n][D]``) by explicit positions.

    ``pos_*`` are length-``n`` arrays (any real values).  Returns a new float64
    array; dims beyond ``sum(split)`` are copied unchanged.
    """
    x = np.asarray(x, dtype=np.float64)
    squeeze = x.ndim == 2
    if squeeze:
        x = x[:, None, :]
    n, _, d = x.shape
    if sum(split) > d:
        raise ValueError("rotary split exceeds head dim")
    out = x.copy()
    offset = 0
    for pos, d_a in zip((pos_t, pos_h, pos_w), split):
        pos = np.asarray(pos, dtype=np.float64).reshape(n, 1)
        ang = pos * axis_frequencies(d_a, theta)[None, :]           # [n][d_a/2]
        c = np.cos(ang)[:, None, :]
        s = np.sin(ang)[:, None, :]
        x0 = x[:, :, offset + 0:offset + d_a:2]
        x1 = x[:, :, offset + 1:offset + d_a:2]
        out[:, :, offset + 0:offset + d_a:2] = x0 * c - x1 * s
        out[:, :, offset + 1:offset + d_a:2] = x0 * s + x1 * c
        offset += d_a
    return out[:, 0, :] if squeeze else out


def rope3d_segment(x: np.ndarray, frames: int, grid_h: int, grid_w: int, t0: int,
                   theta: float = 10000.0, split=(32, 48, 48)) -> np.ndarray:
    """Apply the segment's 3D RoPE to ``x`` (``[n_q][heads][D]``).

    The first ``frames * grid_h * grid_w`` rows are video tokens and are rotated
    at positions ``(t0 + frame, h, w)``; the remaining (text) rows are returned
    unchanged.  Returns float64.
    """
    x = np.asarray(x, dtype=np.float64)
    n_video = frames * grid_h * grid_w
    if n_video > x.shape[0]:
        raise ValueError("more video tokens than rows")
    out = x.copy()
    pt, ph, pw = video_positions(frames, grid_h, grid_w, t0)
    out[:n_video] = rotate(x[:n_video], pt, ph, pw, theta, split)
    return out
