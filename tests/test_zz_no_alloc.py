"""The allocation-free attention entry point agrees with the workspace one.

Callers that cannot allocate device memory on this path (an engine that has
already reserved nearly all of HBM for its own pools, or a latency-bound loop
that cannot accept an allocation's implicit synchronisation) call
nomas_segment_attn_noalloc, whose split-KV scratch is a fixed array inside the
library.  These checks call it through the C ABI:

* on a plan that uses the scratch, it equals nomas_segment_attn given a
  caller-provided workspace bit for bit (same plan, same kernels), on two calls
  in a row with different inputs, so the second call starts from the scratch
  the first one left behind;
* it agrees with the float64 oracle on a ragged shape;
* with the automatic plan on the INT8-window shape (7616 queries, 18 resident
  frames) it runs, uses the scratch, and equals the workspace entry point;
* an explicit piece count whose scratch exceeds the array is refused without
  a launch.

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
    from _gpu_common import assert_attn_close, build_caches, oracle_segment, to_dev

SCRATCH_CAP = 64 * 2 ** 20


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()
    assert nomas.device_error(clear=True) == 0


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _inputs(wl, step):
    q, k, v = (to_dev(x, "bf16") for x in current_qkv(wl, step=step))
    nomas.rope3d(q, k, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    return q, k, v


def _noalloc(gc, wl, q, k, v, splits):
    out = torch.full_like(q, float("nan"))
    lse = torch.full((wl.heads, wl.n_q), float("nan"), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = nomas.nomas_segment_attn_noalloc(ctypes.byref(gc.desc), 0, _ptr(q), _ptr(k), _ptr(v), wl.n_video,
                                          wl.n_text, 1.0 / np.sqrt(wl.head_dim), _ptr(out), _ptr(lse), splits,
                                          stream)
    assert st == nomas.NOMAS_OK, nomas.nomas_status_string(st)
    return out, lse


def _with_workspace(gc, wl, q, k, v, splits):
    ws = torch.empty(max(gc.workspace_bytes(wl.n_video, wl.n_text, splits), 256), dtype=torch.uint8,
                     device="cuda")
    lse = torch.empty((wl.heads, wl.n_q), dtype=torch.float32, device="cuda")
    out = nomas.segment_attn(gc, 0, q, k, v, wl.n_video, wl.n_text, softmax_scale=1.0 / np.sqrt(wl.head_dim),
                             lse=lse, workspace=ws, num_splits=splits)
    return out, lse


def test_noalloc_equals_workspace_entry_point_on_two_calls_in_a_row():
    shapes = [
        small_variant(CONFIGS["c2_bf16_hist8"], heads=4, seed=40),        # BF16 cache
        small_variant(CONFIGS["c3_int8_window18"], heads=2, seed=41),     # INT8 windowed cache
    ]
    for wl in shapes:
        gc, _ = build_caches(wl)
        need = gc.workspace_bytes(wl.n_video, wl.n_text, 2)
        assert 0 < need <= SCRATCH_CAP   # two pieces per unit: the scratch is in use
        for step in (0, 1):              # different inputs; the second call finds the first call's scratch
            q, k, v = _inputs(wl, step)
            out, lse = _noalloc(gc, wl, q, k, v, 2)
            ref, ref_lse = _with_workspace(gc, wl, q, k, v, 2)
            torch.cuda.synchronize()
            assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


def test_noalloc_matches_oracle_on_a_ragged_shape():
    wl = small_variant(CONFIGS["c2_bf16_hist8"], heads=3, grid_h=5, grid_w=7, cache_frames_hist=(2, 1),
                       cur_frames=2, n_text=9, cache_dtype="int8", past_frames=0, capacity_frames=6, seed=42)
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    ref_o, ref_lse = oracle_segment(wl, oc, q, k, v)
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    nomas.rope3d(qd, kd, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    assert gc.workspace_bytes(wl.n_video, wl.n_text, 2) > 0
    out, lse = _noalloc(gc, wl, qd, kd, vd, 2)
    torch.cuda.synchronize()
    assert_attn_close(out, ref_o, lse, ref_lse)


def test_noalloc_automatic_plan_runs_on_the_int8_window():
    wl = CONFIGS["c3_int8_window18"]
    gc, _ = build_caches(wl)
    plan = gc.attn_plan(wl.n_video, wl.n_text, 0)
    assert plan["pieces_per_split_unit"] > 1 and 0 < plan["workspace_bytes"] <= SCRATCH_CAP
    q, k, v = _inputs(wl, 0)
    out, lse = _noalloc(gc, wl, q, k, v, 0)
    ref, ref_lse = _with_workspace(gc, wl, q, k, v, 0)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


def test_noalloc_refuses_explicit_pieces_beyond_its_scratch():
    wl = CONFIGS["c3_int8_window18"]   # 240 pair units x 4 pieces need ~250 MB of scratch
    gc, _ = build_caches(wl)
    assert gc.workspace_bytes(wl.n_video, wl.n_text, 4) > SCRATCH_CAP
    q = torch.zeros((wl.n_q, wl.heads, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = nomas.nomas_segment_attn_noalloc(ctypes.byref(gc.desc), 0, _ptr(q), _ptr(q), _ptr(q), wl.n_video,
                                          wl.n_text, 0.088, _ptr(out), _ptr(None), 4, stream)
    assert st == nomas.NOMAS_ERR_CAPACITY
