"""GPU parity of the FP8 (E4M3) cache variant and of the large-append path,
through the C ABI, against the CPU oracle.

FP8 is a comparison format beside the pages' INT8 cache: the same layout (one
byte per value, one float32 scale per row), E4M3 codes.  Codes and scales must
equal the oracle codec bit for bit; the attention over an FP8 cache meets the
attention tolerances against the oracle's dequantised cache.
"""
import numpy as np
import pytest
import torch

from synth import CONFIGS, current_qkv, segment_kv, small_variant

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import segment_causal_kv_int8_b300 as nomas
    from _gpu_common import assert_attn_close, build_caches, f64, gpu_segment, oracle_segment, to_dev
    from oracle import fp8_codec, ring_cache
    from oracle import sparse as o_sparse


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()
    assert nomas.device_error(clear=True) == 0


def _bits(gc, oc):
    np.testing.assert_array_equal(gc.k.cpu().numpy(), oc.k_codes)
    np.testing.assert_array_equal(gc.v.cpu().numpy(), oc.v_codes)
    np.testing.assert_array_equal(gc.k_scale.cpu().numpy().view(np.uint32), oc.k_scales.view(np.uint32))
    np.testing.assert_array_equal(gc.v_scale.cpu().numpy().view(np.uint32), oc.v_scales.view(np.uint32))
    assert gc.total_frames == oc.total_frames and gc.valid_frames == oc.valid_frames


@pytest.mark.parametrize("cache_dtype", ["int8", "fp8"])
def test_large_append_takes_the_staged_path_bit_exact(cache_dtype):
    # 5 blocks x 8 frames x 920 tokens x 16 heads of bf16 K and V: 301 MB of
    # input, above the size at which the append streams through shared memory
    wl = small_variant(CONFIGS["c3_int8_window18"], cache_dtype=cache_dtype, seed=700)
    blocks = 5
    gc = nomas.KVCache(blocks, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, cache_dtype)
    oc = ring_cache.RingCache(blocks, wl.heads, 128, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames,
                              cache_dtype)
    kv = [segment_kv(wl, 0, 8, b) for b in range(blocks)]
    k = np.stack([x[0] for x in kv])
    v = np.stack([x[1] for x in kv])
    assert 2 * k.size * 2 >= 256 << 20
    gc.append(to_dev(k, "bf16"), to_dev(v, "bf16"))
    oc.append(k, v)
    _bits(gc, oc)


FP8_RAGGED = [
    dict(heads=3, grid_h=5, grid_w=7, cache_frames_hist=(2, 1), cur_frames=2, n_text=9, past_frames=0,
         capacity_frames=6),
    dict(heads=2, grid_h=5, grid_w=7, cache_frames_hist=(3, 3, 3), cur_frames=3, n_text=5, past_frames=4,
         capacity_frames=4),
    dict(heads=2, grid_h=16, grid_w=16, cache_frames_hist=(1,), cur_frames=1, n_text=0, past_frames=0,
         capacity_frames=2),
]


@pytest.mark.parametrize("case", range(len(FP8_RAGGED)))
@pytest.mark.parametrize("splits", [1, 3])
def test_fp8_attention_ragged(case, splits):
    wl = small_variant(CONFIGS["c2_bf16_hist8"], **FP8_RAGGED[case], cache_dtype="fp8", seed=800 + case)
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    ref_o, ref_lse = oracle_segment(wl, oc, q, k, v)
    out, lse = gpu_segment(wl, gc, q, k, v, num_splits=splits)
    assert_attn_close(out, ref_o, lse, ref_lse)


def test_fp8_attention_full_size_window_sampled():
    wl = small_variant(CONFIGS["c3_int8_window18"], cache_dtype="fp8")
    gc, oc = build_caches(wl)
    _bits(gc, oc)
    q, k, v = current_qkv(wl)
    rng = np.random.default_rng(wl.seed)
    rows = np.array(sorted(set(rng.choice(wl.n_q, 64, replace=False).tolist())
                           | {0, 255, 256, wl.n_video - 1, wl.n_video, wl.n_q - 1}))
    ref_o, ref_lse = oracle_segment(wl, oc, q, k, v, rows=rows)
    out, lse = gpu_segment(wl, gc, q, k, v, num_splits=0)
    assert_attn_close(out, ref_o, lse, ref_lse, rows=rows)


def test_fp8_sparse_selection_and_attention():
    wl = small_variant(CONFIGS["c2_bf16_hist8"], heads=2, grid_h=16, grid_w=16, cache_frames_hist=(2, 3),
                       cur_frames=2, n_text=100, cache_dtype="fp8", past_frames=4, capacity_frames=4, seed=900)
    gc, oc = build_caches(wl)
    q, _, _ = current_qkv(wl)
    tiles, counts = nomas.sparse_select(gc, 0, to_dev(q, "bf16"), wl.n_video, wl.n_text, 0.5)
    kc, _ = oc.cache_kv(0)
    kept, scores = o_sparse.select_tiles(o_sparse.group_means(q), o_sparse.tile_means(kc), 0.5)
    k_keep = o_sparse.keep_count(kc.shape[0] // 128 + (kc.shape[0] % 128 > 0), 0.5)
    tl, cn = tiles.cpu().numpy(), counts.cpu().numpy()
    for h in range(wl.heads):
        for g in range(len(kept[0])):
            assert cn[h, g] == k_keep
            row = tl[h, g, :k_keep]
            if list(row) != kept[h][g]:
                cut = np.sort(scores[h, g])[::-1][k_keep - 1]
                assert np.all(scores[h, g][row] >= cut - 2e-5)


def test_fp8_fused_rope_append_and_archive():
    wl = small_variant(CONFIGS["c2_bf16_hist8"], heads=4, grid_h=6, grid_w=8, cache_dtype="fp8", past_frames=3,
                       capacity_frames=3, io_dtype="bf16", seed=950)
    gc = nomas.KVCache(1, wl.heads, wl.grid_h, wl.grid_w, 3, 3, "fp8")
    oc = ring_cache.RingCache(1, wl.heads, 128, wl.grid_h, wl.grid_w, 3, 3, "fp8")
    fb = gc.archive_frame_bytes()
    assert fb == 2 * wl.heads * wl.tpf * (128 + 4)
    archive = torch.zeros((5 * fb,), dtype=torch.uint8).pin_memory()
    used = 0
    for s, frames in enumerate((2, 3)):
        k, v = segment_kv(wl, s, frames, 0)
        gc.append_rope(to_dev(k, "bf16"), to_dev(v, "bf16"), wl.theta, wl.rope_split)
        oc.append_rope(k, v, wl.theta, wl.rope_split)
    # keys: float32 rotation on the GPU against float64 in the oracle may land
    # on opposite sides of an E4M3 rounding boundary: one step apart at most
    gk, ok_ = fp8_codec.decode(gc.k.cpu().numpy()), fp8_codec.decode(oc.k_codes)
    step = np.maximum(np.abs(ok_) * 2.0 ** -3, 2.0 ** -9)
    assert np.all(np.abs(gk - ok_) <= step)
    assert np.count_nonzero(gk != ok_) <= max(8, 1e-3 * gk.size)
    np.testing.assert_array_equal(gc.v.cpu().numpy(), oc.v_codes)
    # the archive copies what the ring holds, frame by frame
    k, v = segment_kv(wl, 2, 2, 0)
    used = gc.append_archive(to_dev(k, "bf16"), to_dev(v, "bf16"), archive, used)
    torch.cuda.synchronize()
    assert used == 2 * fb
    rec = archive.numpy()
    n = wl.heads * wl.tpf * 128
    for i, fa in enumerate((5, 6)):
        slot = fa % 3
        r = rec[i * fb:(i + 1) * fb]
        ring_k = gc.k[0, :, slot * wl.tpf:(slot + 1) * wl.tpf].cpu().numpy().reshape(-1)
        np.testing.assert_array_equal(r[:n], ring_k)
        ring_vs = gc.v_scale[0, :, slot * wl.tpf:(slot + 1) * wl.tpf].cpu().numpy().reshape(-1)
        np.testing.assert_array_equal(r[2 * n + wl.heads * wl.tpf * 4:].view(np.float32), ring_vs)
