"""Pins of the oracle's ring cache (CPU only).

The ring's slot arithmetic is checked against an independent deque model of
"the last W frames", against the window numbers the pages print, and against a
per-frame dictionary of what was appended.
"""
import collections
import json
import os

import numpy as np
import pytest

from oracle import int8_codec, ring_cache

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_window_numbers_from_the_pages():
    g = _load("window_sysram.json")
    shape = _load("model_shape.json")
    assert g["video_frames_per_segment"] // shape["latent_temporal_compression"] == g["segment_latent_frames"]
    c = ring_cache.RingCache(1, 1, 8, 1, 1, capacity_frames=g["past_frames"],
                             past_frames=g["past_frames"], dtype="int8", store=False)
    for n, total in zip(g["after_segments"], g["total_frames"]):
        c.append(n_frames=g["segment_latent_frames"])
        assert c.total_frames == total
        assert c.valid_frames == g["gpu_frames"]
        assert c.resident_frames() == list(range(total - g["gpu_frames"], total))
        # a segment longer than the window writes only its last W frames
        assert sorted(c.frame_of_slot.tolist()) == list(range(total - 18, total))


def test_archive_size_consistent_with_int8_rows_and_fp32_scales():
    # A full copy of every appended frame (INT8 K and V codes plus one float32
    # scale per (block, head, token)) over 30 latent frames of a 23x40 grid and
    # 54 blocks of 16 x 128 comes to within 0.5% of the archive growth the page
    # logs per segment.
    g = _load("window_sysram.json")
    s = _load("model_shape.json")
    gh = -(-s["output_height"] // s["latent_spatial_compression"])
    gw = s["output_width"] // s["latent_spatial_compression"]
    assert (gh, gw) == (23, 40)
    c = ring_cache.RingCache(s["double_stream_blocks"], s["heads"], s["head_dim"], gh, gw,
                             capacity_frames=g["segment_latent_frames"], past_frames=0,
                             dtype="int8", store=False)
    gib = c.bytes() / 2 ** 30
    per_segment = np.diff([0.0] + g["cpu_archive_gib"])
    assert np.all(np.abs(per_segment / gib - 1.0) < 0.005)


def _deque_check(c, dq):
    assert c.resident_frames() == list(dq)
    assert c.valid_frames == len(dq)
    held = {int(f) for f in c.frame_of_slot if f >= 0}
    assert set(dq) <= held
    for f in dq:
        assert c.frame_of_slot[f % c.capacity_frames] == f


@pytest.mark.parametrize("window", [1, 5, 18])
def test_random_appends_match_deque_model(window):
    rng = np.random.default_rng(window)
    c = ring_cache.RingCache(1, 1, 8, 2, 3, capacity_frames=window, past_frames=window,
                             dtype="int8", store=False)
    dq = collections.deque(maxlen=window)
    total = 0
    for _ in range(60):
        n = int(rng.integers(0, 3 * window + 2))
        plan = c.append(n_frames=n)
        written = [fa for _, fa, _ in plan]
        new = list(range(total, total + n))
        dq.extend(new)
        total += n
        assert written == [f for f in new if f in dq]
        for fs, fa, sf in plan:
            assert fa == total - n + fs and sf == fa % window
        _deque_check(c, dq)
        if rng.random() < 0.05:
            c.reset()
            dq.clear()
            total = 0
            assert c.valid_frames == 0 and c.total_frames == 0


def test_no_window_capacity_error_and_slots():
    c = ring_cache.RingCache(1, 1, 8, 1, 2, capacity_frames=5, past_frames=0, dtype="bf16",
                             store=False)
    c.append(n_frames=3)
    assert c.frame_of_slot.tolist()[:3] == [0, 1, 2]
    with pytest.raises(ring_cache.CapacityError):
        c.append(n_frames=3)
    c.append(n_frames=2)
    assert c.valid_frames == 5 and c.resident_frames() == [0, 1, 2, 3, 4]


def test_window_requires_capacity_equal_past_frames():
    with pytest.raises(ValueError):
        ring_cache.RingCache(1, 1, 8, 1, 1, capacity_frames=20, past_frames=18, dtype="int8")


@pytest.mark.parametrize("dtype", ["int8", "bf16"])
def test_stored_rows_follow_their_frames(dtype):
    blocks, heads, d, gh, gw, W = 2, 3, 16, 2, 2, 5
    tpf = gh * gw
    c = ring_cache.RingCache(blocks, heads, d, gh, gw, capacity_frames=W, past_frames=W, dtype=dtype)
    rng = np.random.default_rng(9)
    by_frame = {}
    total = 0
    for n in (2, 3, 4, 7, 1):
        k = rng.standard_normal((blocks, n * tpf, heads, d)).astype(np.float32)
        v = rng.standard_normal((blocks, n * tpf, heads, d)).astype(np.float32)
        c.append(k, v)
        for fs in range(n):
            by_frame[total + fs] = (k[:, fs * tpf:(fs + 1) * tpf], v[:, fs * tpf:(fs + 1) * tpf])
        total += n
        for f in c.resident_frames():
            sf = f % W
            kk, vv = by_frame[f]
            for b in range(blocks):
                for h in range(heads):
                    sl = slice(sf * tpf, (sf + 1) * tpf)
                    if dtype == "int8":
                        codes, sc = int8_codec.quantize_rows(kk[b, :, h])
                        np.testing.assert_array_equal(c.k_codes[b, h, sl], codes)
                        np.testing.assert_array_equal(c.k_scales[b, h, sl], sc)
                        codes, sc = int8_codec.quantize_rows(vv[b, :, h])
                        np.testing.assert_array_equal(c.v_codes[b, h, sl], codes)
                        np.testing.assert_array_equal(c.v_scales[b, h, sl], sc)
                    else:
                        # bf16 storage: within half a bf16 ulp of the input
                        rel = np.abs(c.k_vals[b, h, sl] - kk[b, :, h]) / np.maximum(np.abs(kk[b, :, h]), 1e-30)
                        assert np.all(rel <= 2.0 ** -8)
        # resident K as returned for attention: slot order, frames of the window only
        kc, _ = c.cache_kv(1)
        assert kc.shape == (c.valid_frames * tpf, heads, d)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9, -(1.0 + 2.0 ** -8)], np.float32)
    y = ring_cache._bf16_round(x)
    np.testing.assert_array_equal(y, [1.0, 1.0 + 2.0 ** -6, 1.0, -1.0])
