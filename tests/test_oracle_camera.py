"""Pins of the oracle's camera cross-attention (CPU)."""
import math

import numpy as np

from oracle.camera import camera_cross_attention


def _data(frames=3, tpf=5, n_cam=4, h=2, d=128, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((frames * tpf, h, d)), rng.standard_normal((frames, n_cam, h, d)),
            rng.standard_normal((frames, n_cam, h, d)))


def test_single_camera_token_returns_its_value():
    q, k, v = _data(n_cam=1)
    o = camera_cross_attention(q, k, v, 3, 5, 0.09)
    for f in range(3):
        np.testing.assert_array_equal(o[f * 5:(f + 1) * 5], np.broadcast_to(v[f, 0], (5, 2, 128)))


def test_equal_keys_average_the_values():
    q, k, v = _data()
    k[:] = k[:, :1]
    o = camera_cross_attention(q, k, v, 3, 5, 0.09)
    for f in range(3):
        np.testing.assert_allclose(o[f * 5:(f + 1) * 5], np.broadcast_to(v[f].mean(axis=0), (5, 2, 128)),
                                   rtol=1e-12, atol=1e-12)


def test_brute_force_rows():
    q, k, v = _data(seed=1)
    s = 0.0883883
    o = camera_cross_attention(q, k, v, 3, 5, s)
    for r in range(15):
        f = r // 5
        for h in range(2):
            sc = [s * sum(q[r, h, i] * k[f, j, h, i] for i in range(128)) for j in range(4)]
            mx = max(sc)
            w = [math.exp(x - mx) for x in sc]
            want = sum(w[j] * v[f, j, h] for j in range(4)) / sum(w)
            np.testing.assert_allclose(o[r, h], want, rtol=1e-12, atol=1e-12)


def test_tokens_see_only_their_own_frame():
    q, k, v = _data(seed=2)
    o = camera_cross_attention(q, k, v, 3, 5, 0.09)
    k2, v2 = k.copy(), v.copy()
    k2[1] += 5.0
    v2[1] *= -3.0
    o2 = camera_cross_attention(q, k2, v2, 3, 5, 0.09)
    np.testing.assert_array_equal(o[:5], o2[:5])
    np.testing.assert_array_equal(o[10:], o2[10:])
    assert not np.allclose(o[5:10], o2[5:10])
