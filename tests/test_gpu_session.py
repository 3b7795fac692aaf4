"""The session workload as a chain on the GPU, checked against the oracle.

Turns of the 54-block session use full-size calls (16 heads x 128, 23x40 grid,
8 latent frames + 256 text queries, INT8 cache with an 18-frame window); the
chain here keeps 3 blocks and runs 5 turns, which is enough for the window to
fill and wrap (resident frames 0, 8, 16, 18, 18).  After every append the
INT8 codes, scales and metadata of every block must equal the oracle ring bit
for bit; the attention is checked on sampled calls (first and last denoising
step, first and last block) on a sample of query rows.  Inputs come from the
seeded device-side generators; the oracle receives copies of them.
"""
import dataclasses

import numpy as np
import pytest
import torch

from synth import CONFIGS, current_qkv_torch, segment_kv_torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import segment_causal_kv_int8_b300 as nomas
    from _gpu_common import assert_attn_close
    from oracle import attention as o_attn
    from oracle import ring_cache as o_cache
    from oracle import rope3d as o_rope


def _rows(n_q, n_video, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(n_q, size=40, replace=False).tolist()) | {0, n_video - 1, n_video, n_q - 1}
    return np.array(sorted(rows))


def test_session_chain_window_wrap_and_sampled_attention():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    wl = dataclasses.replace(CONFIGS["c5_session12"], blocks=3)
    turns, steps = 5, (0, wl.steps - 1)
    gc = nomas.KVCache(wl.blocks, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, "int8")
    oc = o_cache.RingCache(wl.blocks, wl.heads, wl.head_dim, wl.grid_h, wl.grid_w, wl.capacity_frames,
                           wl.past_frames, "int8")
    scale = o_attn.default_scale(wl.head_dim)
    for turn in range(turns):
        t0 = gc.total_frames
        assert t0 == oc.total_frames
        for step in steps:
            for block in (0, wl.blocks - 1):
                q, k, v = current_qkv_torch(wl, turn, step, block, "cuda")
                qh, kh, vh = (x.float().cpu().numpy() for x in (q, k, v))
                nomas.rope3d(q, k, wl.cur_frames, wl.grid_h, wl.grid_w, t0, wl.theta, wl.rope_split)
                lse = torch.empty((wl.heads, wl.n_q), dtype=torch.float32, device="cuda")
                ws = torch.empty(max(gc.workspace_bytes(wl.n_video, wl.n_text), 256), dtype=torch.uint8,
                                 device="cuda")
                out = nomas.segment_attn(gc, block, q, k, v, wl.n_video, wl.n_text, lse=lse, workspace=ws)
                rows = _rows(wl.n_q, wl.n_video, 1000 * turn + 10 * step + block)
                qr = o_rope.rope3d_segment(qh, wl.cur_frames, wl.grid_h, wl.grid_w, t0, wl.theta, wl.rope_split)
                kr = o_rope.rope3d_segment(kh, wl.cur_frames, wl.grid_h, wl.grid_w, t0, wl.theta, wl.rope_split)
                kc, vc = oc.cache_kv(block)
                assert kc.shape[0] == min(t0, wl.window) * wl.tpf
                ref_o, ref_lse = o_attn.segment_attention(qr, kr, vh, kc, vc, scale, rows=rows)
                assert_attn_close(out, ref_o, lse, ref_lse, rows=rows)
        kseg, vseg = segment_kv_torch(wl, turn, wl.cur_frames, wl.blocks, "cuda")
        gc.append(kseg, vseg)
        oc.append(kseg.float().cpu().numpy(), vseg.float().cpu().numpy())
        torch.cuda.synchronize()
        assert (gc.total_frames, gc.valid_frames) == (oc.total_frames, oc.valid_frames)
        np.testing.assert_array_equal(gc.k.cpu().numpy(), oc.k_codes)
        np.testing.assert_array_equal(gc.v.cpu().numpy(), oc.v_codes)
        np.testing.assert_array_equal(gc.k_scale.cpu().numpy().view(np.uint32), oc.k_scales.view(np.uint32))
        np.testing.assert_array_equal(gc.v_scale.cpu().numpy().view(np.uint32), oc.v_scales.view(np.uint32))
    assert gc.valid_frames == wl.window and gc.total_frames == turns * wl.cur_frames
    assert nomas.device_error(clear=True) == 0
