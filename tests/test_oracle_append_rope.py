"""Pins of the oracle's KV write with position encoding (CPU)."""
import numpy as np

from oracle import ring_cache
from oracle.rope3d import rope3d_segment


def _seg(frames, gh=3, gw=4, heads=2, seed=0):
    rng = np.random.default_rng(seed)
    n = frames * gh * gw
    return (rng.standard_normal((n, heads, 128)).astype(np.float32),
            rng.standard_normal((n, heads, 128)).astype(np.float32))


def _cache(dtype, cap=8, past=0):
    return ring_cache.RingCache(1, 2, 128, 3, 4, cap, past, dtype)


def test_no_rotary_dims_is_plain_append():
    k, v = _seg(3)
    a, b = _cache("int8"), _cache("int8")
    a.append(k, v)
    b.append_rope(k, v, split=(0, 0, 0))
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name))


def test_positions_continue_across_segments():
    # two segments written one after the other hold the keys of one
    # five-frame segment rotated from frame 0
    k1, v1 = _seg(2, seed=1)
    k2, v2 = _seg(3, seed=2)
    c = _cache("bf16")
    c.append_rope(k1, v1)
    c.append_rope(k2, v2)
    whole = rope3d_segment(np.concatenate([k1, k2]), 5, 3, 4, 0)
    kc, vc = c.cache_kv(0)
    want = ring_cache._bf16_round(whole.astype(np.float32))
    np.testing.assert_array_equal(kc, want)
    np.testing.assert_array_equal(vc, ring_cache._bf16_round(np.concatenate([v1, v2])))
    # the first token of the first frame sits at the origin: not rotated
    np.testing.assert_array_equal(kc[0], ring_cache._bf16_round(k1[0]))


def test_frames_dropped_by_the_window_keep_absolute_positions():
    k, v = _seg(5, seed=3)
    c = _cache("bf16", cap=3, past=3)
    c.append(*_seg(1, seed=4))                  # one frame already cached: t0 = 1
    c.append_rope(k, v)                        # frames 1..5; 3..5 stay resident
    whole = rope3d_segment(k, 5, 3, 4, 1)
    tpf = 12
    for fa in (3, 4, 5):
        slot = fa % 3
        got = c.k_vals[0, :, slot * tpf:(slot + 1) * tpf].transpose(1, 0, 2)
        fs = fa - 1
        np.testing.assert_array_equal(got, ring_cache._bf16_round(whole[fs * tpf:(fs + 1) * tpf].astype(np.float32)))
