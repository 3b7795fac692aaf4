"""Pins of the oracle's 3D RoPE (CPU only).

Each check comes from mathematics the rotary embedding must satisfy, computed a
different way from the oracle (complex exponentials, geometric identities,
shift invariance), so that a dropped term, a wrong sign, a wrong pair index or
a wrong axis chunk fails at least one of them.
"""
import numpy as np
import pytest

from oracle import rope3d

SPLIT = (32, 48, 48)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_identity_at_position_zero():
    x = _rand((7, 3, 128), 0)
    z = np.zeros(7)
    np.testing.assert_array_equal(rope3d.rotate(x, z, z, z), x)


def test_norm_preserved_per_pair():
    x = _rand((50, 2, 128), 1)
    rng = np.random.default_rng(2)
    pt, ph, pw = (rng.integers(0, 200, 50) for _ in range(3))
    y = rope3d.rotate(x, pt, ph, pw)
    nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-12, atol=1e-12)


def test_frequency_geometry():
    # f_i * f_{d/2 - i} == 1 / theta for a geometric ladder from 1 down to 1/theta
    # over d/2 steps (the pair index runs over d/2 entries with exponent -2i/d).
    for d in (32, 48, 8):
        f = rope3d.axis_frequencies(d, 10000.0)
        assert f.shape == (d // 2,)
        assert f[0] == 1.0
        ext = np.append(f, 1.0 / 10000.0)          # the would-be entry i = d/2
        np.testing.assert_allclose(ext * ext[::-1], np.full(d // 2 + 1, 1e-4), rtol=1e-13)
        ratios = f[1:] / f[:-1]
        np.testing.assert_allclose(ratios, np.full(d // 2 - 1, 10000.0 ** (-2.0 / d)), rtol=1e-13)


def test_matches_complex_rotation_per_axis():
    # Textbook 1-D RoPE: pair (x0, x1) is the complex number x0 + i x1 multiplied
    # by exp(i * pos * f).  Compute it with complex exponentials, axis by axis.
    x = _rand((9, 2, 128), 3)
    pos = {"t": np.arange(9) + 5, "h": (np.arange(9) * 3) % 7, "w": (np.arange(9) * 5) % 11}
    y = rope3d.rotate(x, pos["t"], pos["h"], pos["w"], theta=10000.0, split=SPLIT)
    off = 0
    for axis, d in zip("thw", SPLIT):
        i = np.arange(d // 2)
        freq = np.exp(-np.log(10000.0) * (2.0 * i / d))
        z = x[:, :, off:off + d:2] + 1j * x[:, :, off + 1:off + d:2]
        rot = z * np.exp(1j * pos[axis][:, None, None] * freq[None, None, :])
        np.testing.assert_allclose(y[:, :, off:off + d:2], rot.real, atol=1e-12)
        np.testing.assert_allclose(y[:, :, off + 1:off + d:2], rot.imag, atol=1e-12)
        off += d


def test_each_axis_touches_only_its_chunk():
    x = _rand((1, 1, 128), 4)
    base = rope3d.rotate(x, [3], [4], [5])
    for axis, (lo, hi) in zip(range(3), ((0, 32), (32, 80), (80, 128))):
        p = [3, 4, 5]
        p[axis] += 1
        y = rope3d.rotate(x, [p[0]], [p[1]], [p[2]])
        changed = np.nonzero(np.abs(y - base)[0, 0] > 1e-15)[0]
        assert changed.min() >= lo and changed.max() < hi


@pytest.mark.parametrize("shift", [(1, 0, 0), (0, 3, 0), (0, 0, 7), (40, 11, 13)])
def test_shift_invariance_of_scores(shift):
    # Invariant 3: q.k after rotation depends only on the position difference.
    rng = np.random.default_rng(5)
    q = rng.standard_normal((30, 2, 128))
    k = rng.standard_normal((30, 2, 128))
    pq = [rng.integers(0, 60, 30) for _ in range(3)]
    pk = [rng.integers(0, 60, 30) for _ in range(3)]
    s0 = np.einsum("nhd,nhd->nh", rope3d.rotate(q, *pq), rope3d.rotate(k, *pk))
    pq2 = [p + c for p, c in zip(pq, shift)]
    pk2 = [p + c for p, c in zip(pk, shift)]
    s1 = np.einsum("nhd,nhd->nh", rope3d.rotate(q, *pq2), rope3d.rotate(k, *pk2))
    np.testing.assert_allclose(s1, s0, atol=1e-10)


def test_relative_rotation():
    # R(p)q . R(p')k == q . R(p' - p)k
    rng = np.random.default_rng(6)
    q = rng.standard_normal((10, 128))
    k = rng.standard_normal((10, 128))
    pq = [rng.integers(0, 50, 10) for _ in range(3)]
    pk = [rng.integers(0, 50, 10) for _ in range(3)]
    lhs = np.sum(rope3d.rotate(q, *pq) * rope3d.rotate(k, *pk), axis=1)
    rel = [b - a for a, b in zip(pq, pk)]
    rhs = np.sum(q * rope3d.rotate(k, *rel), axis=1)
    np.testing.assert_allclose(lhs, rhs, atol=1e-10)


def test_video_positions_order_and_text_untouched():
    frames, gh, gw, t0 = 2, 3, 4, 9
    pt, ph, pw = rope3d.video_positions(frames, gh, gw, t0)
    n = np.arange(frames * gh * gw)
    np.testing.assert_array_equal(pt, t0 + n // (gh * gw))
    np.testing.assert_array_equal(ph, (n % (gh * gw)) // gw)
    np.testing.assert_array_equal(pw, n % gw)
    x = _rand((frames * gh * gw + 5, 2, 128), 7)
    y = rope3d.rope3d_segment(x, frames, gh, gw, t0)
    np.testing.assert_array_equal(y[frames * gh * gw:], x[frames * gh * gw:])
    # the first video token sits at (t0, 0, 0): only the t chunk moves
    np.testing.assert_array_equal(y[0, :, 32:], x[0, :, 32:])
    assert np.any(y[0, :, :32] != x[0, :, :32])
