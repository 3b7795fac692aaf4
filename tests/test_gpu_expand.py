"""GPU parity of the BF16 expansion of a one-byte cache (nomas_kvcache_expand),
through the C ABI, against the CPU oracle.

The expansion writes x_hat = bf16(fl32(code * scale)) for every resident slot,
the value the attention kernel's dequantising warps use; the tests rebuild
those values from the oracle codec's codes and scales (a float32 product, then
round to nearest even to bf16) and compare bit for bit.  Attention over the
expanded copy meets the attention tolerances against the oracle's INT8 cache.
"""
import numpy as np
import pytest
import torch

from synth import CONFIGS, segment_kv, small_variant, current_qkv

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import segment_causal_kv_int8_b300 as nomas
    from _gpu_common import assert_attn_close, build_caches, f64, gpu_segment, oracle_segment, to_dev
    from oracle import fp8_codec, ring_cache
    from oracle.ring_cache import _bf16_round


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()
    assert nomas.device_error(clear=True) == 0


def _codec_values(codes, scales, cache_dtype):
    """bf16(fl32(value(code) * scale)) per element, as float64."""
    if cache_dtype == "int8":
        vals = np.asarray(codes).astype(np.float32)
    else:
        vals = fp8_codec.decode(codes).astype(np.float32)
    prod = vals * np.asarray(scales, dtype=np.float32)[..., None]  # one float32 rounding
    return _bf16_round(prod)


def _shadow_like(gc, wl, blocks=1):
    s = nomas.KVCache(blocks, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, "bf16")
    s.k.fill_(7.0)
    s.v.fill_(7.0)
    return s


def _check_expanded(shadow, gc, oc, cache_dtype):
    assert shadow.total_frames == gc.total_frames and shadow.valid_frames == gc.valid_frames
    n = gc.valid_frames * gc.tpf
    for got_t, codes, scales in ((shadow.k, oc.k_codes, oc.k_scales), (shadow.v, oc.v_codes, oc.v_scales)):
        want = _codec_values(codes[:, :, :n], scales[:, :, :n], cache_dtype)
        np.testing.assert_array_equal(f64(got_t)[:, :, :n], want)
        # slots outside the resident window are not written
        assert bool((got_t[:, :, n:] == 7.0).all())


CASES = [
    # windowed ring that has wrapped (10 frames through a 4-frame window)
    dict(heads=2, grid_h=5, grid_w=7, cache_frames_hist=(3, 3, 4), cur_frames=2, n_text=5, past_frames=4,
         capacity_frames=4),
    # no window, the ring partly filled
    dict(heads=3, grid_h=9, grid_w=15, cache_frames_hist=(2, 1), cur_frames=3, n_text=40, past_frames=0,
         capacity_frames=6),
]


@pytest.mark.parametrize("cache_dtype", ["int8", "fp8"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_expanded_window_equals_the_codec_values(cache_dtype, case):
    wl = small_variant(CONFIGS["c2_bf16_hist8"], **CASES[case], cache_dtype=cache_dtype, seed=800 + case)
    gc, oc = build_caches(wl)
    shadow = _shadow_like(gc, wl)
    gc.expand_into(shadow)
    torch.cuda.synchronize()
    _check_expanded(shadow, gc, oc, cache_dtype)


def test_expansion_covers_every_block_and_head():
    # Three blocks of the c3 grid, one 8-frame segment each: every (block, head)
    # plane and both tensors.
    wl = small_variant(CONFIGS["c3_int8_window18"], heads=4, seed=810)
    blocks = 3
    gc = nomas.KVCache(blocks, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, "int8")
    oc = ring_cache.RingCache(blocks, wl.heads, 128, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, "int8")
    kv = [segment_kv(wl, 0, 8, b) for b in range(blocks)]
    k = np.stack([x[0] for x in kv])
    v = np.stack([x[1] for x in kv])
    gc.append(to_dev(k, "bf16"), to_dev(v, "bf16"))
    oc.append(k, v)
    shadow = _shadow_like(gc, wl, blocks)
    gc.expand_into(shadow)
    torch.cuda.synchronize()
    _check_expanded(shadow, gc, oc, "int8")


@pytest.mark.parametrize("name", ["c3_int8_window18"])
def test_attention_over_the_expanded_window(name):
    # The c3 shape: the BF16 copy of the INT8 window, attended by the BF16
    # kernel, against the oracle's INT8 cache (every 7th query row) and
    # against the INT8 kernel on the same inputs.
    wl = CONFIGS[name]
    gc, oc = build_caches(wl)
    shadow = _shadow_like(gc, wl)
    gc.expand_into(shadow)
    q, k, v = current_qkv(wl)
    out_s, lse_s = gpu_segment(wl, shadow, q, k, v)
    out_i, _ = gpu_segment(wl, gc, q, k, v)
    torch.cuda.synchronize()
    rows = np.arange(0, wl.n_q, 7)
    ref_o, ref_lse = oracle_segment(wl, oc, q, k, v, rows=rows)
    assert_attn_close(out_s, ref_o, lse_s, ref_lse, rows=rows)
    # same dequantised values, different kernels (and work plans): equal up to
    # the order of float32 accumulation
    d = np.abs(f64(out_s) - f64(out_i))
    assert d.max() <= 8e-3 and d.mean() <= 2e-4, (d.max(), d.mean())
