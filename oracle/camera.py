"""Camera cross-attention of the video tokens (oracle, float64; test infrastructure only).

Camera control enters as 4x4 extrinsic matrices grouped over four frames and
fed through cross-attention in every block (the blog.authon.dev guide to
running Hy-Nomas on an RTX 4090, section "What Hy-Nomas is", model-card specs;
the orcarouter.ai explainer, section "Zwei Lenkräder, und nur eines davon ist
ein Prompt").  One latent frame covers four video frames (4x temporal
compression, the same spec list).  Reading: the camera encoder (trained
weights, upstream) gives latent frame ``f`` of the segment ``n_cam`` key and
value tokens per head, and every video token of that latent frame attends to
exactly those tokens with exact softmax; text tokens take no part.

Parity unpinned as to the reading itself (which tokens a frame's group
yields, and that video tokens see only their own frame's group); the tests
pin this definition: a single camera token returns its value, equal keys
average the values, a brute-force softmax per row, and tokens of one frame
ignore every other frame's camera tokens.
"""
from __future__ import annotations

import numpy as np

from .attention import attention


def camera_cross_attention(q_video, k_cam, v_cam, frames: int, tpf: int, scale: float) -> np.ndarray:
    """``O [frames*tpf][H][D]``: row ``f*tpf + t`` attends to ``k_cam[f]``, ``v_cam[f]`` (``[n_cam][H][D]``)."""
    q = np.asarray(q_video, np.float64)[:frames * tpf]
    kc = np.asarray(k_cam, np.float64)
    vc = np.asarray(v_cam, np.float64)
    out = np.zeros_like(q)
    for f in range(frames):
        rows = slice(f * tpf, (f + 1) * tpf)
        out[rows], _ = attention(q[rows], kc[f], vc[f], scale)
    return out
