"""Segment attention over the resident KV cache plus the current segment (oracle, float64).

What the pages fix: Hy-Nomas is a segment-autoregressive diffusion transformer
whose next segment is conditioned on a lifelong KV cache of the earlier
latents' keys and values (Hy-Nomas: Was Tencent ... tatsaechlich macht, section
"Die Schleife"); its dual-stream blocks use "segment-wise causal joint
attention" (the madebyagents.com model page, component list), with 16 heads of
128 dims (Hy-Nomas auf einer RTX 4090, section "Modell und Dateien").

Reading used here: exact softmax attention per head,

    S = s * Q K^T,   P = rowsoftmax(S),   O = P V,   LSE = log sum_j exp(S_j)

with ``s = 1 / sqrt(head_dim)``, queries = the current segment's video and text
tokens, keys/values = [resident cache (dequantised if INT8) ; current
segment's own K/V].  Every current query sees every key in that set: the mask
is causal across segments only (bidirectional inside a segment, as in MMDiT
joint attention), and frames evicted by the window are simply absent.
The key order does not matter mathematically.

:func:`full_sequence_attention` states the same thing a second way, as one
masked attention over a whole session's tokens with the segment-causal,
windowed mask written in absolute frame numbers.  It never touches a ring
buffer, so its agreement with the per-call form pins the cache's slot
arithmetic and eviction.
"""
from __future__ import annotations

import math

import numpy as np

from . import int8_codec
from .ring_cache import _bf16_round


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def attention(q, k, v, scale: float, mask=None, chunk: int = 512):
    """Exact softmax attention per head in float64.

    ``q``: ``[Nq][H][D]``; ``k``, ``v``: ``[Nk][H][D]``; ``mask``: optional bool
    ``[Nq][Nk]`` (True = visible).  Returns ``(O [Nq][H][D], LSE [H][Nq])`` with
    the natural-log LSE.  Queries are processed in row chunks to bound memory.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, h, d = q.shape
    o = np.empty((nq, h, v.shape[2]), np.float64)
    lse = np.empty((h, nq), np.float64)
    for hh in range(h):
        kh = k[:, hh, :]
        vh = v[:, hh, :]
        for r0 in range(0, nq, chunk):
            r1 = min(nq, r0 + chunk)
            s = scale * (q[r0:r1, hh, :] @ kh.T)
            if mask is not None:
                s = np.where(mask[r0:r1], s, -np.inf)
            m = np.max(s, axis=1, keepdims=True)
            p = np.exp(s - m)
            l = np.sum(p, axis=1, keepdims=True)
            o[r0:r1, hh, :] = (p @ vh) / l
            lse[hh, r0:r1] = (m + np.log(l))[:, 0]
    return o, lse


def segment_attention(q, k_cur, v_cur, k_cache, v_cache, scale: float, rows=None):
    """Attention of the current segment's queries over [cache ; current] keys.

    ``k_cache``/``v_cache``: ``[Nc][H][D]`` (already dequantised), may have
    ``Nc = 0``.  ``rows``: optional subset of query rows (for sampled checks).
    """
    k = np.concatenate([np.asarray(k_cache, np.float64), np.asarray(k_cur, np.float64)], axis=0)
    v = np.concatenate([np.asarray(v_cache, np.float64), np.asarray(v_cur, np.float64)], axis=0)
    qq = np.asarray(q, np.float64)
    if rows is not None:
        qq = qq[np.asarray(rows)]
    return attention(qq, k, v, scale)


def full_sequence_attention(segments, tpf: int, past_frames: int, cache_dtype: str,
                            scale: float):
    """Whole-session masked attention (the segment-causal mask in absolute frames).

    ``segments``: list of dicts, in session order, each with ``frames`` (latent
    frames of video), ``q``, ``k_cur``, ``v_cur`` (``[Nq_s][H][D]``, video rows
    first) and ``k_app``, ``v_app`` (``[frames * tpf][H][D]``: what the
    KV-write pass appends after the segment).

    Keys of the session are laid out as [appended video rows of every segment ;
    current rows of every segment].  Query ``i`` of segment ``s`` (first
    absolute frame ``T_s``) sees
      * current row ``j`` of segment ``s'`` iff ``s' == s``;
      * appended video row ``j`` of segment ``s'`` at absolute frame ``f_j`` iff
        ``s' < s`` and (no window or ``f_j >= T_s - past_frames``).
    Appended rows enter in their cached form (INT8 codec round trip, or bf16).
    Returns a list of ``(O_s, LSE_s)``.
    """
    app_k, app_v, app_seg, app_frame = [], [], [], []
    cur_k, cur_v, cur_seg = [], [], []
    t = 0
    firsts = []
    for s, seg in enumerate(segments):
        firsts.append(t)
        ka = np.asarray(seg["k_app"], np.float32)
        va = np.asarray(seg["v_app"], np.float32)
        if cache_dtype == "int8":
            kc, ks = int8_codec.quantize_rows(ka)
            vc, vs = int8_codec.quantize_rows(va)
            app_k.append(int8_codec.dequantize_rows(kc, ks))
            app_v.append(int8_codec.dequantize_rows(vc, vs))
        else:
            app_k.append(_bf16_round(ka))
            app_v.append(_bf16_round(va))
        n_app = ka.shape[0]
        app_seg.append(np.full(n_app, s))
        app_frame.append(t + np.arange(n_app) // tpf)
        cur_k.append(np.asarray(seg["k_cur"], np.float64))
        cur_v.append(np.asarray(seg["v_cur"], np.float64))
        cur_seg.append(np.full(seg["k_cur"].shape[0], s))
        t += seg["frames"]
    keys = np.concatenate(app_k + cur_k, axis=0)
    vals = np.concatenate(app_v + cur_v, axis=0)
    a_seg = np.concatenate(app_seg)
    a_frame = np.concatenate(app_frame)
    c_seg = np.concatenate(cur_seg)
    out = []
    for s, seg in enumerate(segments):
        vis_app = a_seg < s
        if past_frames > 0:
            vis_app &= a_frame >= firsts[s] - past_frames
        vis_cur = c_seg == s
        row_mask = np.concatenate([vis_app, vis_cur])
        q = np.asarray(seg["q"], np.float64)
        mask = np.broadcast_to(row_mask[None, :], (q.shape[0], row_mask.shape[0]))
        out.append(attention(q, keys, vals, scale, mask=mask))
    return out
