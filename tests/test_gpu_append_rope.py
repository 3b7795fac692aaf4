"""GPU parity of the KV write with position encoding (3D RoPE of K fused into
the append), through the C ABI.

Against the oracle: the GPU rotates in float32 and the oracle in float64
(rounded to float32 before the codec), so a stored value may differ where the
two land on opposite sides of a rounding boundary: an INT8 code by one, a
bf16 value by one unit in the last place.  The tests bound how often that
happens and check everything else bit for bit.  Against the GPU's own
two-pass path (RoPE, then append) the float32 case is bit-exact.
"""
import numpy as np
import pytest
import torch

from synth import CONFIGS, segment_kv, small_variant

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import segment_causal_kv_int8_b300 as nomas
    from _gpu_common import f64, to_dev
    from oracle import ring_cache


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()
    assert nomas.device_error(clear=True) == 0


def _caches(wl, blocks=1):
    gc = nomas.KVCache(blocks, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, wl.cache_dtype)
    oc = ring_cache.RingCache(blocks, wl.heads, 128, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames,
                              wl.cache_dtype)
    return gc, oc


def _segments(wl, blocks):
    """Seeded segments: lists of (k, v) ``[blocks][F*tpf][heads][128]`` float32."""
    segs = []
    for s, frames in enumerate(wl.cache_frames_hist):
        ks, vs = zip(*(segment_kv(wl, s, frames, b) for b in range(blocks)))
        segs.append((np.stack(ks), np.stack(vs)))
    return segs


def _compare_to_oracle(gc, oc, max_frac=1e-4):
    assert gc.total_frames == oc.total_frames and gc.valid_frames == oc.valid_frames
    if oc.dtype == "int8":
        np.testing.assert_array_equal(gc.v.cpu().numpy(), oc.v_codes)
        np.testing.assert_array_equal(gc.v_scale.cpu().numpy().view(np.uint32), oc.v_scales.view(np.uint32))
        gs, os_ = gc.k_scale.cpu().numpy().astype(np.float64), oc.k_scales.astype(np.float64)
        assert np.all(np.abs(gs - os_) <= 1e-6 * np.abs(os_)), "K scale off by more than float32 rotation error"
        d = gc.k.cpu().numpy().astype(np.int32) - oc.k_codes.astype(np.int32)
        assert np.abs(d).max() <= 1
        assert np.count_nonzero(d) <= max(8, max_frac * d.size), f"{np.count_nonzero(d)} codes differ"
    else:
        np.testing.assert_array_equal(f64(gc.v), oc.v_vals)
        g, o = f64(gc.k), oc.k_vals
        diff = g != o
        # one bf16 ulp (2^-7 relative at most), plus the float32 rotation error
        # where x0 c - x1 s cancels to a value near zero (N(0,1) data)
        assert np.all(np.abs(g - o) <= 2.0 ** -7 * np.abs(o) + 1e-5), "K differs by more than one bf16 ulp"
        assert np.count_nonzero(diff) <= max(8, max_frac * diff.size), f"{np.count_nonzero(diff)} values differ"


CASES = [
    # heads, grid, segments (frames each), cache dtype, window / capacity, input dtype, blocks
    dict(heads=3, grid_h=5, grid_w=7, cache_frames_hist=(2, 3, 1), cache_dtype="int8", past_frames=0,
         capacity_frames=6, io_dtype="f32", blocks=2),
    dict(heads=17, grid_h=4, grid_w=6, cache_frames_hist=(3, 5, 2), cache_dtype="int8", past_frames=4,
         capacity_frames=4, io_dtype="bf16", blocks=1),
    dict(heads=2, grid_h=9, grid_w=15, cache_frames_hist=(2, 2), cache_dtype="bf16", past_frames=3,
         capacity_frames=3, io_dtype="bf16", blocks=2),
    dict(heads=16, grid_h=3, grid_w=5, cache_frames_hist=(7,), cache_dtype="bf16", past_frames=0,
         capacity_frames=7, io_dtype="f32", blocks=1),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_append_rope_matches_oracle(case):
    wl = small_variant(CONFIGS["c2_bf16_hist8"], **CASES[case], seed=500 + case)
    gc, oc = _caches(wl, wl.blocks)
    for k, v in _segments(wl, wl.blocks):
        gc.append_rope(to_dev(k, wl.io_dtype), to_dev(v, wl.io_dtype), wl.theta, wl.rope_split)
        oc.append_rope(k, v, wl.theta, wl.rope_split)
    _compare_to_oracle(gc, oc)


@pytest.mark.parametrize("cache_dtype", ["int8", "bf16"])
def test_float32_input_equals_rope_then_append(cache_dtype):
    wl = small_variant(CONFIGS["c2_bf16_hist8"], heads=5, grid_h=6, grid_w=7, cache_frames_hist=(3, 4, 2),
                       cache_dtype=cache_dtype, past_frames=5, capacity_frames=5, io_dtype="f32", seed=600)
    fused, _ = _caches(wl, 2)
    two_pass, _ = _caches(wl, 2)
    for k, v in _segments(wl, 2):
        kd, vd = to_dev(k, "f32"), to_dev(v, "f32")
        fused.append_rope(kd, vd, 10000.0, (32, 48, 48))
        frames = k.shape[1] // wl.tpf
        kr = kd.clone()
        for b in range(2):
            nomas.rope3d(kr[b], None, frames, wl.grid_h, wl.grid_w, two_pass.total_frames, 10000.0, (32, 48, 48))
        two_pass.append(kr, vd)
    for name in ("k", "v", "k_scale", "v_scale"):
        a, b = getattr(fused, name), getattr(two_pass, name)
        if a is not None:
            assert torch.equal(a, b), name


def test_full_size_int8_window():
    wl = CONFIGS["c3_int8_window18"]
    gc, oc = _caches(wl, 1)
    for k, v in _segments(wl, 1):
        gc.append_rope(to_dev(k, "bf16"), to_dev(v, "bf16"), wl.theta, wl.rope_split)
        oc.append_rope(k, v, wl.theta, wl.rope_split)
    _compare_to_oracle(gc, oc)


def test_bad_rope_arguments_are_rejected():
    wl = small_variant(CONFIGS["c1_tiny"], io_dtype="bf16")
    gc, _ = _caches(wl, 1)
    k, v = segment_kv(wl, 0, 1, 0)
    kd, vd = to_dev(k, "bf16"), to_dev(v, "bf16")
    for theta, split in ((0.0, (32, 48, 48)), (1e4, (31, 48, 48)), (1e4, (64, 48, 48))):
        with pytest.raises(nomas.NomasError):
            gc.append_rope(kd, vd, theta, split)
    assert gc.total_frames == 0
