"""The allocation-free attention entry point agrees with the workspace one.

Callers that cannot allocate device memory on this path (an engine that has
already reserved nearly all of HBM for its own pools, or a latency-bound loop
that cannot accept an allocation's implicit synchronisation) call
nomas_segment_attn_noalloc, whose split-KV scratch is a fixed array inside the
library.  These checks call it through the C ABI and compare it with
nomas_segment_attn given a caller-provided workspace, on two calls in a row
(the second call finds the scratch as the first left it), and check that a
request larger than the fixed scratch is refused without a launch.

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from synth import CONFIGS, current_qkv, small_variant

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import segment_causal_kv_int8_b300 as nomas
    from _gpu_common import ATTN_MAX_ABS, ATTN_MEAN_ABS, LSE_ABS, build_caches, to_dev


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _run_both(wl, splits):
    gc, _ = build_caches(wl)
    q, k, v = (to_dev(x, "bf16") for x in current_qkv(wl))
    nomas.rope3d(q, k, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    scale = 1.0 / np.sqrt(wl.head_dim)

    ws = torch.empty(max(gc.workspace_bytes(wl.n_video, wl.n_text, splits), 256), dtype=torch.uint8,
                     device="cuda")
    ref_lse = torch.empty((wl.heads, wl.n_q), dtype=torch.float32, device="cuda")
    ref = nomas.segment_attn(gc, 0, q, k, v, wl.n_video, wl.n_text, softmax_scale=scale, lse=ref_lse,
                             workspace=ws, num_splits=splits)

    out = torch.full_like(q, float("nan"))
    lse = torch.full((wl.heads, wl.n_q), float("nan"), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = nomas.nomas_segment_attn_noalloc(ctypes.byref(gc.desc), 0, _ptr(q), _ptr(k), _ptr(v), wl.n_video,
                                          wl.n_text, scale, _ptr(out), _ptr(lse), splits, stream)
    assert st == nomas.NOMAS_OK, nomas.nomas_status_string(st)
    torch.cuda.synchronize()
    return out, lse, ref, ref_lse


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    shapes = [
        small_variant(CONFIGS["c2_bf16_hist8"], heads=4, seed=40),        # BF16 cache
        small_variant(CONFIGS["c3_int8_window18"], heads=2, seed=41),     # INT8 windowed cache
    ]
    for wl in shapes:
        out, lse, ref, ref_lse = _run_both(wl, splits=2)
        o, r = out.float().cpu().numpy(), ref.float().cpu().numpy()
        assert np.isfinite(o).all()
        err = np.abs(o - r)
        assert err.max() <= ATTN_MAX_ABS and err.mean() <= ATTN_MEAN_ABS
        lerr = np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy())
        assert lerr.max() <= LSE_ABS
    assert nomas.device_error(clear=True) == 0


def test_noalloc_refuses_requests_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    wl = CONFIGS["c3_int8_window18"]   # 16 heads x 7616 queries: 4 splits need ~250 MB of scratch
    gc, _ = build_caches(wl)
    need = gc.workspace_bytes(wl.n_video, wl.n_text, 4)
    assert need > 64 * 2 ** 20
    q = torch.zeros((wl.n_q, wl.heads, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = nomas.nomas_segment_attn_noalloc(ctypes.byref(gc.desc), 0, _ptr(q), _ptr(q), _ptr(q), wl.n_video,
                                          wl.n_text, 0.088, _ptr(out), _ptr(None), 4, stream)
    assert st == nomas.NOMAS_ERR_CAPACITY
