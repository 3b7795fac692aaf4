"""Host KV archive: every appended frame, once quantised, copied to host memory.

The low-memory recipe keeps the last past_frames latent frames on the GPU and
every earlier frame in host RAM.  The checks append a sequence of segments
(one longer than the window) to an INT8 windowed cache through
nomas_kvcache_append_archive and compare the host archive, frame by frame,
with the oracle codec applied to that frame's K and V (bit for bit), and the
ring with the oracle ring cache, then check the archive's bounds and the
capacity error.
"""
import ctypes

import numpy as np
import pytest
import torch

from synth import CONFIGS, segment_kv, small_variant

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import segment_causal_kv_int8_b300 as nomas
    from _gpu_common import to_dev
    from oracle import int8_codec, ring_cache


def _frame_records(archive, frame_bytes, blocks, heads, tpf, d):
    """Split an archive into per-frame (k_codes, v_codes, k_scales, v_scales)."""
    out = []
    for f in range(len(archive) // frame_bytes):
        rec = archive[f * frame_bytes:(f + 1) * frame_bytes]
        n = blocks * heads * tpf
        kc = rec[:n * d].view(np.int8).reshape(blocks, heads, tpf, d)
        vc = rec[n * d:2 * n * d].view(np.int8).reshape(blocks, heads, tpf, d)
        ks = rec[2 * n * d:2 * n * d + 4 * n].view(np.float32).reshape(blocks, heads, tpf)
        vs = rec[2 * n * d + 4 * n:].view(np.float32).reshape(blocks, heads, tpf)
        out.append((kc, vc, ks, vs))
    return out


@pytest.mark.parametrize("in_dtype", ["bf16", "f32"])
def test_archive_holds_every_frame_bit_exact(in_dtype):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    blocks, heads, gh, gw, W = 3, 2, 3, 5, 4
    wl = small_variant(CONFIGS["c1_tiny"], heads=heads, grid_h=gh, grid_w=gw, io_dtype=in_dtype, outlier_p=0.01)
    tpf = gh * gw
    gc = nomas.KVCache(blocks, heads, gh, gw, W, W, "int8")
    oc = ring_cache.RingCache(blocks, heads, 128, gh, gw, W, W, "int8")
    frame_bytes = gc.archive_frame_bytes()
    assert frame_bytes == 2 * blocks * heads * tpf * (128 + 4)
    seg_frames = (3, 2, 6, 1)          # the third segment is longer than the window
    guard = 4096
    archive = torch.full((sum(seg_frames) * frame_bytes + guard,), 0xA5, dtype=torch.uint8).pin_memory()
    used, expected = 0, []
    for s, f in enumerate(seg_frames):
        kv = [segment_kv(wl, 50 + s, f, b) for b in range(blocks)]
        k = np.stack([x[0] for x in kv])
        v = np.stack([x[1] for x in kv])
        if s == 1:
            k[0, 3, 1] = 0.0   # an all-zero row
        used = gc.append_archive(to_dev(k, in_dtype), to_dev(v, in_dtype), archive, used)
        oc.append(k, v)
        for fr in range(f):
            rows = slice(fr * tpf, (fr + 1) * tpf)
            kf = np.transpose(k[:, rows], (0, 2, 1, 3))      # [blocks][heads][tpf][128]
            vf = np.transpose(v[:, rows], (0, 2, 1, 3))
            expected.append(int8_codec.quantize_rows(kf) + int8_codec.quantize_rows(vf))
        torch.cuda.synchronize()
        assert used == len(expected) * frame_bytes
        assert (gc.total_frames, gc.valid_frames) == (oc.total_frames, oc.valid_frames)
        np.testing.assert_array_equal(gc.k.cpu().numpy(), oc.k_codes)
        np.testing.assert_array_equal(gc.v_scale.cpu().numpy().view(np.uint32), oc.v_scales.view(np.uint32))
    arch = archive.numpy()
    records = _frame_records(arch[:used], frame_bytes, blocks, heads, tpf, 128)
    assert len(records) == sum(seg_frames)
    for (kc, vc, ks, vs), (ekc, eks, evc, evs) in zip(records, expected):
        np.testing.assert_array_equal(kc, ekc)
        np.testing.assert_array_equal(vc, evc)
        np.testing.assert_array_equal(ks.view(np.uint32), eks.view(np.uint32))
        np.testing.assert_array_equal(vs.view(np.uint32), evs.view(np.uint32))
    assert (arch[used:] == 0xA5).all()  # nothing written past the frames


def test_archive_capacity_error_changes_nothing():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    gc = nomas.KVCache(1, 2, 3, 5, 4, 4, "int8")
    fb = gc.archive_frame_bytes()
    small = torch.zeros((2 * fb,), dtype=torch.uint8).pin_memory()
    k = torch.zeros((1, 3 * 15, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nomas.NomasError) as e:
        gc.append_archive(k, k, small, 0)
    assert e.value.status == nomas.NOMAS_ERR_CAPACITY
    assert gc.total_frames == 0
    g16 = nomas.KVCache(1, 2, 3, 5, 4, 4, "bf16")
    with pytest.raises(nomas.NomasError) as e:
        g16.append_archive(k, k, small, 0)
    assert e.value.status == nomas.NOMAS_ERR_UNSUPPORTED
