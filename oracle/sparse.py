"""Block-sparse segment attention (oracle, float64; test infrastructure only).

The single-GPU preset's backend list mentions a sparse attention mode that
keeps the first two denoising steps dense and afterwards attends to a
quarter of the candidate video key blocks (Hy-Nomas auf einer RTX 4090,
section "Das Single-GPU-Preset"; the blog.authon.dev guide's low-memory
config excerpt).  The pages give neither the block size nor the selection
rule, so this module writes out the plainest reading:

* candidates are the resident cache's key tiles of 128 tokens (tile t holds
  cache slots [128 t, 128 t + 128) that are resident); the current segment's
  own keys (video and text) are always attended;
* queries are grouped in blocks of 512 rows; for head h and query group g
  the score of tile t is the dot product of the group's mean query and the
  tile's mean key, qbar[h, g] . kbar[h, t] (the softmax scale does not change
  the order);
* the ceil(keep * T) highest-scoring tiles are kept (ties: lower tile index
  first), listed in increasing tile order;
* every query of group g attends to the kept tiles' keys plus all current
  keys, with exact softmax.

Parity unpinned: the selection rule itself (pooled-mean scores, tile and
group sizes) is a reading, pinned only by this definition; the tests pin its
implementation (brute-force ranking, a planted dominant tile), the mask (keep
= 1 is dense attention, each group equals dense attention over its gathered
keys) and the ordering conventions.
"""
from __future__ import annotations

import math

import numpy as np

from .attention import attention

KEY_TILE = 128
QUERY_GROUP = 512


def tile_means(k_cache: np.ndarray, tile: int = KEY_TILE) -> np.ndarray:
    """Mean key of every tile: ``[H][T][D]`` from ``[Nc][H][D]`` (the last tile may be partial)."""
    k = np.asarray(k_cache, np.float64)
    n, h, d = k.shape
    t = -(-n // tile)
    out = np.zeros((h, t, d), np.float64)
    for i in range(t):
        out[:, i, :] = k[i * tile:min(n, (i + 1) * tile)].mean(axis=0)
    return out


def group_means(q: np.ndarray, group: int = QUERY_GROUP) -> np.ndarray:
    """Mean query of every group of ``group`` rows: ``[H][G][D]`` from ``[Nq][H][D]``."""
    q = np.asarray(q, np.float64)
    n, h, d = q.shape
    g = -(-n // group)
    out = np.zeros((h, g, d), np.float64)
    for i in range(g):
        out[:, i, :] = q[i * group:min(n, (i + 1) * group)].mean(axis=0)
    return out


def keep_count(n_tiles: int, keep: float) -> int:
    """Tiles kept out of ``n_tiles`` for a keep fraction in (0, 1]."""
    return min(n_tiles, int(math.ceil(keep * n_tiles - 1e-9)))


def select_tiles(qbar: np.ndarray, kbar: np.ndarray, keep: float):
    """Kept tile indices per (head, group): a list of lists of increasing ints, and the scores."""
    h, g, _ = qbar.shape
    t = kbar.shape[1]
    k = keep_count(t, keep)
    scores = np.einsum("hgd,htd->hgt", qbar, kbar)
    kept = []
    for hh in range(h):
        row = []
        for gg in range(g):
            order = sorted(range(t), key=lambda i: (-scores[hh, gg, i], i))
            row.append(sorted(order[:k]))
        kept.append(row)
    return kept, scores


def sparse_segment_attention(q, k_cur, v_cur, k_cache, v_cache, scale: float, kept, rows=None):
    """Attention of each query group over its kept cache tiles plus all current keys.

    ``kept[h][g]``: increasing tile indices.  Returns ``(O [Nq][H][D], LSE [H][Nq])``
    (only ``rows`` when given, in that order).
    """
    q = np.asarray(q, np.float64)
    kc = np.asarray(k_cache, np.float64)
    vc = np.asarray(v_cache, np.float64)
    kn = np.asarray(k_cur, np.float64)
    vn = np.asarray(v_cur, np.float64)
    nq, h, d = q.shape
    sel_rows = np.arange(nq) if rows is None else np.asarray(rows)
    o = np.zeros((len(sel_rows), h, d), np.float64)
    lse = np.zeros((h, len(sel_rows)), np.float64)
    for hh in range(h):
        for gi in np.unique(sel_rows // QUERY_GROUP):
            idx = np.nonzero(sel_rows // QUERY_GROUP == gi)[0]
            tiles = kept[hh][int(gi)]
            cache_rows = np.concatenate([np.arange(t * KEY_TILE, min(kc.shape[0], (t + 1) * KEY_TILE))
                                         for t in tiles]) if len(tiles) else np.zeros(0, np.int64)
            keys = np.concatenate([kc[cache_rows, hh:hh + 1], kn[:, hh:hh + 1]], axis=0)
            vals = np.concatenate([vc[cache_rows, hh:hh + 1], vn[:, hh:hh + 1]], axis=0)
            oo, ll = attention(q[sel_rows[idx], hh:hh + 1], keys, vals, scale)
            o[idx, hh] = oo[:, 0]
            lse[hh, idx] = ll[0]
    return o, lse
