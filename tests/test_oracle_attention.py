"""Pins of the oracle's segment attention (CPU only).

Invariants 1, 2, 4 and 6, the textbook reduction to PyTorch's scaled dot
product attention, closed-form LSE values, key-order invariance and RoPE shift
invariance of whole attention outputs.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, int8_codec, ring_cache, rope3d
from synth import CONFIGS, current_qkv, history_segments


def _rng(seed):
    return np.random.default_rng(seed)


def test_rows_sum_to_one_via_constant_values():
    # Invariant 1: with V = 1 everywhere, O = sum_j P_ij = 1 for every row.
    r = _rng(0)
    q, k = r.standard_normal((37, 3, 128)) * 3, r.standard_normal((91, 3, 128)) * 3
    o, _ = attention.attention(q, k, np.ones((91, 3, 128)), 1 / math.sqrt(128))
    np.testing.assert_allclose(o, 1.0, atol=1e-12)


def test_single_visible_key_returns_its_value():
    # Invariant 2: one current video token, empty cache, no text.
    r = _rng(1)
    q, k, v = (r.standard_normal((1, 2, 128)) for _ in range(3))
    o, lse = attention.segment_attention(q, k, v, np.zeros((0, 2, 128)), np.zeros((0, 2, 128)),
                                         1 / math.sqrt(128))
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse[:, 0], np.einsum("hd,hd->h", q[0], k[0]) / math.sqrt(128), atol=1e-12)


def test_single_visible_key_through_the_mask():
    # Invariant 2 through the full-sequence form: segment 1's only current token
    # sees segment 0's single appended key only if the window keeps it.
    r = _rng(2)
    seg0 = dict(frames=1, q=r.standard_normal((1, 1, 128)), k_cur=r.standard_normal((1, 1, 128)),
                v_cur=r.standard_normal((1, 1, 128)), k_app=r.standard_normal((1, 1, 128)).astype(np.float32),
                v_app=r.standard_normal((1, 1, 128)).astype(np.float32))
    seg1 = dict(frames=1, q=r.standard_normal((1, 1, 128)) * 0, k_cur=r.standard_normal((1, 1, 128)),
                v_cur=r.standard_normal((1, 1, 128)), k_app=seg0["k_app"], v_app=seg0["v_app"])
    # q = 0: both visible keys score 0 -> O is the mean of the two visible values
    (o0, _), (o1, lse1) = attention.full_sequence_attention([seg0, seg1], 1, 1, "bf16", 0.1)
    np.testing.assert_allclose(o0, seg0["v_cur"], atol=1e-15)
    vapp = ring_cache._bf16_round(seg0["v_app"])
    np.testing.assert_allclose(o1[0], 0.5 * (vapp[0] + seg1["v_cur"][0]), atol=1e-15)
    np.testing.assert_allclose(lse1, math.log(2.0), atol=1e-15)


def test_lse_closed_form_uniform_scores():
    r = _rng(3)
    nk = 57
    o, lse = attention.attention(np.zeros((5, 2, 128)), r.standard_normal((nk, 2, 128)),
                                 r.standard_normal((nk, 2, 128)), 0.3)
    np.testing.assert_allclose(lse, math.log(nk), atol=1e-14)


def _bruteforce(q, k, v, scale):
    """Scalar triple loops in pure Python (independent of numpy's matmul/softmax)."""
    nq, h, d = q.shape
    nk = k.shape[0]
    o = [[[0.0] * d for _ in range(h)] for _ in range(nq)]
    lse = [[0.0] * nq for _ in range(h)]
    ql, kl, vl = q.tolist(), k.tolist(), v.tolist()
    for hh in range(h):
        for i in range(nq):
            s = []
            for j in range(nk):
                acc = 0.0
                qi, kj = ql[i][hh], kl[j][hh]
                for t in range(d):
                    acc += qi[t] * kj[t]
                s.append(acc * scale)
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = math.fsum(e)
            for t in range(d):
                o[i][hh][t] = math.fsum(e[j] * vl[j][hh][t] for j in range(nk)) / z
            lse[hh][i] = m + math.log(z)
    return np.array(o), np.array(lse)


def test_bruteforce_on_tiny_config():
    # Invariant 6 on config 1 (2 heads, 4x6 grid, 2 cached frames, 1 + 16 text
    # current tokens; INT8 cache through the codec; RoPE applied to current Q/K).
    wl = CONFIGS["c1_tiny"]
    c = ring_cache.RingCache(1, wl.heads, wl.head_dim, wl.grid_h, wl.grid_w,
                             wl.capacity_frames, wl.past_frames, wl.cache_dtype)
    for k, v in history_segments(wl):
        c.append(k[None], v[None])
    q, k, v = current_qkv(wl)
    q = rope3d.rope3d_segment(q, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0)
    k = rope3d.rope3d_segment(k, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0)
    kc, vc = c.cache_kv(0)
    assert kc.shape[0] == 48 and q.shape[0] == 40
    scale = attention.default_scale(wl.head_dim)
    o, lse = attention.segment_attention(q, k, v, kc, vc, scale)
    ob, lb = _bruteforce(q, np.concatenate([kc, k]), np.concatenate([vc, v]), scale)
    np.testing.assert_allclose(o, ob, atol=1e-12)
    np.testing.assert_allclose(lse, lb, atol=1e-12)


def test_matches_torch_sdpa_float64():
    r = _rng(4)
    q, k, v = r.standard_normal((33, 4, 128)), r.standard_normal((70, 4, 128)), r.standard_normal((70, 4, 128))
    kc, vc = r.standard_normal((45, 4, 128)), r.standard_normal((45, 4, 128))
    o, _ = attention.segment_attention(q, k, v, kc, vc, attention.default_scale(128))
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(np.concatenate([kc, k])).permute(1, 0, 2)
    tv = torch.from_numpy(np.concatenate([vc, v])).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(o, ref, atol=1e-12)


def test_key_order_is_irrelevant():
    r = _rng(5)
    q, k, v = r.standard_normal((20, 2, 128)), r.standard_normal((30, 2, 128)), r.standard_normal((30, 2, 128))
    kc, vc = r.standard_normal((50, 2, 128)), r.standard_normal((50, 2, 128))
    perm = r.permutation(50)
    a = attention.segment_attention(q, k, v, kc, vc, 0.09)
    b = attention.segment_attention(q, k, v, kc[perm], vc[perm], 0.09)
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


def test_rope_shift_leaves_attention_unchanged():
    # Invariant 3 at the attention level: rotating every cached and current
    # video key and query at positions shifted by a constant changes nothing.
    r = _rng(6)
    gh, gw, fc, fh = 3, 4, 2, 3
    tpf = gh * gw
    qv, kv, vv = (r.standard_normal((fc * tpf, 2, 128)) for _ in range(3))
    kh, vh = r.standard_normal((fh * tpf, 2, 128)), r.standard_normal((fh * tpf, 2, 128))
    outs = []
    for shift in (0, 37):
        q = rope3d.rope3d_segment(qv, fc, gh, gw, fh + shift)
        k = rope3d.rope3d_segment(kv, fc, gh, gw, fh + shift)
        kc = rope3d.rope3d_segment(kh, fh, gh, gw, shift)
        outs.append(attention.segment_attention(q, k, vv, kc, vh, 0.088))
    np.testing.assert_allclose(outs[0][0], outs[1][0], atol=1e-10)


@pytest.mark.parametrize("dtype,window", [("int8", 5), ("bf16", 0), ("int8", 0), ("bf16", 3)])
def test_full_sequence_mask_equals_ring_cache_calls(dtype, window):
    # Invariant 4: queries of segment s see exactly segments < s (window-limited)
    # plus their own segment, whether stated as a whole-session mask in absolute
    # frames or as per-call attention over the ring cache.
    r = _rng(7)
    gh, gw, heads, d, n_text = 2, 3, 2, 128, 3
    tpf = gh * gw
    frames = [2, 3, 4, 1, 3]
    cap = window if window else sum(frames)
    c = ring_cache.RingCache(1, heads, d, gh, gw, cap, window, dtype)
    segs = []
    for f in frames:
        nq = f * tpf + n_text
        segs.append(dict(frames=f,
                         q=r.standard_normal((nq, heads, d)),
                         k_cur=r.standard_normal((nq, heads, d)),
                         v_cur=r.standard_normal((nq, heads, d)),
                         k_app=r.standard_normal((f * tpf, heads, d)).astype(np.float32),
                         v_app=r.standard_normal((f * tpf, heads, d)).astype(np.float32)))
    scale = attention.default_scale(d)
    full = attention.full_sequence_attention(segs, tpf, window, dtype, scale)
    for s, seg in enumerate(segs):
        kc, vc = c.cache_kv(0)
        o, lse = attention.segment_attention(seg["q"], seg["k_cur"], seg["v_cur"], kc, vc, scale)
        np.testing.assert_allclose(o, full[s][0], atol=1e-12)
        np.testing.assert_allclose(lse, full[s][1], atol=1e-12)
        c.append(seg["k_app"][None], seg["v_app"][None])


def test_full_sequence_detects_a_leaked_evicted_frame():
    # A plausible ring bug (one stale frame left visible) must change the result.
    r = _rng(8)
    tpf, heads, d = 2, 1, 128
    segs = [dict(frames=2, q=r.standard_normal((4, heads, d)), k_cur=r.standard_normal((4, heads, d)),
                 v_cur=r.standard_normal((4, heads, d)),
                 k_app=r.standard_normal((4, heads, d)).astype(np.float32),
                 v_app=r.standard_normal((4, heads, d)).astype(np.float32)) for _ in range(3)]
    full = attention.full_sequence_attention(segs, tpf, 2, "int8", 0.1)
    # segment 2 sees only frames 2,3 of the cache; adding frame 1 changes its output
    kc = np.concatenate([segs[0]["k_app"][2:], segs[1]["k_app"]])
    vc = np.concatenate([segs[0]["v_app"][2:], segs[1]["v_app"]])
    kq, ks = int8_codec.quantize_rows(kc)
    vq, vs = int8_codec.quantize_rows(vc)
    o, _ = attention.segment_attention(segs[2]["q"], segs[2]["k_cur"], segs[2]["v_cur"],
                                       int8_codec.dequantize_rows(kq, ks),
                                       int8_codec.dequantize_rows(vq, vs), 0.1)
    assert np.max(np.abs(o - full[2][0])) > 1e-3
