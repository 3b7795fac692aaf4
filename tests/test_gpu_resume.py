"""Checkpoint / resume of a session: the cache is caller-owned tensors plus a
plain descriptor struct, so saving both and restoring them into fresh buffers
continues the session exactly (the service keeps the cache between calls:
Hy-Nomas auf einer RTX 4090, section "Setup", preserve_kv_cache)."""
import ctypes

import numpy as np
import pytest
import torch

from synth import CONFIGS, current_qkv, segment_kv, small_variant

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import segment_causal_kv_int8_b300 as nomas
    from _gpu_common import build_caches, gpu_segment, to_dev


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()
    assert nomas.device_error(clear=True) == 0


@pytest.mark.parametrize("cache_dtype", ["int8", "bf16", "fp8"])
def test_saved_cache_resumes_bit_exact(cache_dtype):
    wl = small_variant(CONFIGS["c2_bf16_hist8"], heads=3, grid_h=6, grid_w=9, cache_frames_hist=(2, 3, 2),
                       cur_frames=2, n_text=11, cache_dtype=cache_dtype, past_frames=5, capacity_frames=5,
                       seed=1200)
    live, _ = build_caches(wl)
    torch.cuda.synchronize()
    # checkpoint: the descriptor's bytes and host copies of the buffers
    saved_desc = bytes(live.desc)
    saved = {n: getattr(live, n).cpu().clone() for n in ("k", "v", "k_scale", "v_scale")
             if getattr(live, n) is not None}
    # resume into fresh device buffers
    resumed = nomas.KVCache(1, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, cache_dtype)
    for n, t in saved.items():
        getattr(resumed, n).copy_(t)
    d = nomas.nomas_kvcache.from_buffer_copy(saved_desc)
    resumed.desc.total_frames, resumed.desc.valid_frames = d.total_frames, d.valid_frames
    assert nomas.nomas_kvcache_validate(ctypes.byref(resumed.desc)) == nomas.NOMAS_OK
    q, k, v = current_qkv(wl)
    for cache in (live, resumed):
        cache._out = gpu_segment(wl, cache, q, k, v, num_splits=2)
    assert torch.equal(live._out[0], resumed._out[0]) and torch.equal(live._out[1], resumed._out[1])
    # the next segment goes to the same slots in both
    k2, v2 = segment_kv(wl, 7, 3, 0)
    for cache in (live, resumed):
        cache.append(to_dev(k2, wl.io_dtype), to_dev(v2, wl.io_dtype))
    for n in saved:
        assert torch.equal(getattr(live, n), getattr(resumed, n)), n
    assert (live.total_frames, live.valid_frames) == (resumed.total_frames, resumed.valid_frames)
