"""Pins of the block-sparse oracle (CPU)."""
import itertools

import numpy as np

from oracle import attention as o_attn
from oracle import sparse


def _data(nq=1100, nc=700, h=2, d=128, seed=7):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s)
    return f(nq, h, d), f(nq, h, d), f(nq, h, d), f(nc, h, d), f(nc, h, d)


def test_keep_all_is_dense_attention():
    q, kn, vn, kc, vc = _data()
    qbar, kbar = sparse.group_means(q), sparse.tile_means(kc)
    kept, _ = sparse.select_tiles(qbar, kbar, 1.0)
    assert all(kept[h][g] == list(range(kbar.shape[1])) for h in range(2) for g in range(qbar.shape[1]))
    o, lse = sparse.sparse_segment_attention(q, kn, vn, kc, vc, 0.088, kept)
    ref_o, ref_lse = o_attn.segment_attention(q, kn, vn, kc, vc, 0.088)
    np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_each_group_equals_dense_attention_over_its_gathered_keys():
    q, kn, vn, kc, vc = _data(seed=8)
    kept = [[[0, 3, 5], [1], [], [2, 4]], [[5], [0, 1, 2, 3, 4, 5], [3], [0]]]
    o, lse = sparse.sparse_segment_attention(q, kn, vn, kc, vc, 0.1, kept)
    for h, g in itertools.product(range(2), range(3)):
        rows = np.arange(512 * g, min(len(q), 512 * (g + 1)))
        gathered = [np.arange(128 * t, min(len(kc), 128 * (t + 1))) for t in kept[h][g]]
        idx = np.concatenate(gathered) if gathered else np.zeros(0, int)
        keys = np.concatenate([kc[idx], kn])[:, h:h + 1]
        vals = np.concatenate([vc[idx], vn])[:, h:h + 1]
        # brute force: softmax written out per row
        for r in rows[::97]:
            s = 0.1 * keys[:, 0] @ q[r, h]
            p = np.exp(s - s.max())
            np.testing.assert_allclose(o[r, h], p @ vals[:, 0] / p.sum(), rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse[h, r], s.max() + np.log(p.sum()), rtol=1e-12)


def test_selection_matches_brute_force_ranking_and_keep_count():
    rng = np.random.default_rng(9)
    qbar, kbar = rng.standard_normal((3, 4, 16)), rng.standard_normal((3, 11, 16))
    for keep, want in ((0.25, 3), (0.5, 6), (1 / 11, 1), (0.99, 11)):
        kept, scores = sparse.select_tiles(qbar, kbar, keep)
        for h, g in itertools.product(range(3), range(4)):
            s = [float(qbar[h, g] @ kbar[h, t]) for t in range(11)]
            top = sorted(range(11), key=lambda t: (-s[t], t))[:want]
            assert kept[h][g] == sorted(top)
            assert len(kept[h][g]) == want == sparse.keep_count(11, keep)


def test_ties_prefer_the_lower_tile_and_planted_tile_is_kept():
    qbar = np.ones((1, 1, 4))
    kbar = np.zeros((1, 6, 4))
    kept, _ = sparse.select_tiles(qbar, kbar, 0.5)     # all scores tie at 0
    assert kept[0][0] == [0, 1, 2]
    kbar[0, 4] = 5.0                                    # one clearly aligned tile
    kept, _ = sparse.select_tiles(qbar, kbar, 1 / 6)
    assert kept[0][0] == [4]


def test_means_over_partial_tiles_and_groups():
    q, _, _, kc, _ = _data(nq=600, nc=200)
    kbar, qbar = sparse.tile_means(kc), sparse.group_means(q)
    np.testing.assert_allclose(kbar[:, 1], kc[128:200].mean(axis=0), rtol=1e-12)
    np.testing.assert_allclose(qbar[:, 1], q[512:600].mean(axis=0), rtol=1e-12)
