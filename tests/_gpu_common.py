"""Helpers shared by the GPU parity tests: seeded inputs -> torch tensors, tolerances."""
import numpy as np
import torch

import segment_causal_kv_int8_b300 as nomas
from oracle import attention as o_attn
from oracle import ring_cache as o_cache
from oracle import rope3d as o_rope
from synth import current_qkv, history_segments

# Tolerances stated for the hot path: attention outputs on N(0,1) inputs,
# max abs <= 2e-2 and mean abs <= 2e-3; float32 RoPE <= 1e-5 relative per
# (token, head) vector (inf-norm of the difference over the inf-norm of the
# reference vector).
ATTN_MAX_ABS = 2e-2
ATTN_MEAN_ABS = 2e-3
ROPE_REL = 1e-5
# LSE: the GPU rounds the rotated Q and K (and dequantised K) to bf16, 2^-9
# relative each, so a score s*q.k moves by ~ s*|q||k|*2^-9*sqrt(2/3) ~ 1.6e-3
# (one standard deviation) on N(0,1) data with s = 1/sqrt(128); the LSE
# inherits a weighted mean of those shifts.  1e-2 is about six of them.
LSE_ABS = 1e-2


def to_dev(x: np.ndarray, io_dtype: str, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return (t.to(torch.bfloat16) if io_dtype == "bf16" else t).to(device)


def f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def build_caches(wl, block=0, device="cuda"):
    """GPU cache and oracle cache for ``wl`` with its history appended (one block)."""
    gc = nomas.KVCache(1, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, wl.cache_dtype,
                       device=device)
    oc = o_cache.RingCache(1, wl.heads, wl.head_dim, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames,
                           wl.cache_dtype)
    for k, v in history_segments(wl, block):
        gc.append(to_dev(k, wl.io_dtype, device), to_dev(v, wl.io_dtype, device))
        oc.append(k[None], v[None])
    return gc, oc


def oracle_segment(wl, oc, q, k, v, rows=None, block=0):
    """Oracle attention of the current segment after its RoPE (float64)."""
    qr = o_rope.rope3d_segment(q, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    kr = o_rope.rope3d_segment(k, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    kc, vc = oc.cache_kv(block)
    return o_attn.segment_attention(qr, kr, v, kc, vc, o_attn.default_scale(wl.head_dim), rows=rows)


def gpu_segment(wl, gc, q, k, v, num_splits=0, with_lse=True, block=0):
    """GPU path: RoPE (bf16 in place) then segment attention; returns (out, lse) tensors."""
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    nomas.rope3d(qd, kd, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    lse = torch.empty((wl.heads, wl.n_q), dtype=torch.float32, device="cuda") if with_lse else None
    ws = None
    nbytes = gc.workspace_bytes(wl.n_video, wl.n_text, num_splits)
    if nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = nomas.segment_attn(gc, block, qd, kd, vd, wl.n_video, wl.n_text, lse=lse, workspace=ws,
                             num_splits=num_splits)
    return out, lse


def assert_attn_close(out, ref_o, lse=None, ref_lse=None, rows=None):
    o = f64(out)
    if rows is not None:
        o = o[np.asarray(rows)]
    err = np.abs(o - ref_o)
    assert np.isfinite(o).all(), "non-finite attention output"
    assert err.max() <= ATTN_MAX_ABS, f"max abs err {err.max():.3e}"
    assert err.mean() <= ATTN_MEAN_ABS, f"mean abs err {err.mean():.3e}"
    if lse is not None:
        l = lse.detach().cpu().numpy().astype(np.float64)
        if rows is not None:
            l = l[:, np.asarray(rows)]
        lerr = np.abs(l - ref_lse)
        assert lerr.max() <= LSE_ABS, f"lse max abs err {lerr.max():.3e}"
    return float(err.max()), float(err.mean())
