"""GPU parity of block-sparse segment attention (tile selection and the sparse
attention kernel) against the CPU oracle, through the C ABI.

The selection is compared on identical inputs (the un-rotated bf16 queries
and the cache both sides hold bit for bit); the attention is given the
oracle's own kept lists.  Nothing the GPU produces is fed to the oracle.
"""
import numpy as np
import pytest
import torch

from synth import CONFIGS, current_qkv, small_variant

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import segment_causal_kv_int8_b300 as nomas
    from _gpu_common import assert_attn_close, build_caches, f64, to_dev
    from oracle import attention as o_attn
    from oracle import rope3d as o_rope
    from oracle import sparse as o_sparse


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()
    assert nomas.device_error(clear=True) == 0


# Scores are float32 dot products of float32 means on the GPU; near-equal
# scores may order differently from the float64 oracle.  A swap is accepted
# only between tiles whose oracle scores lie within SCORE_TOL of the cut.
SCORE_TOL = 2e-5

CASES = [
    # ragged tiles, INT8, two query groups with a short second one
    dict(heads=3, grid_h=5, grid_w=7, cache_frames_hist=(8, 8, 4), cur_frames=16, n_text=9, cache_dtype="int8",
         past_frames=0, capacity_frames=24),
    # BF16, window wrapped, several groups
    dict(heads=2, grid_h=9, grid_w=15, cache_frames_hist=(3, 3, 3), cur_frames=5, n_text=40, cache_dtype="bf16",
         past_frames=6, capacity_frames=6),
    # INT8 window wrapped, text-only tail group
    dict(heads=2, grid_h=16, grid_w=16, cache_frames_hist=(2, 3), cur_frames=2, n_text=100, cache_dtype="int8",
         past_frames=4, capacity_frames=4),
]


def _variant(i):
    return small_variant(CONFIGS["c2_bf16_hist8"], **CASES[i], seed=300 + i)


def _lists_to_device(kept, width):
    h, g = len(kept), len(kept[0])
    tiles = np.full((h, g, max(1, width)), -1, np.int32)
    counts = np.zeros((h, g), np.int32)
    for a in range(h):
        for b in range(g):
            row = kept[a][b]
            tiles[a, b, :len(row)] = row
            counts[a, b] = len(row)
    return torch.from_numpy(tiles).cuda(), torch.from_numpy(counts).cuda()


def _check_selection(tiles, counts, qbar, kbar, keep):
    kept_ref, scores = o_sparse.select_tiles(qbar, kbar, keep)
    n_t = kbar.shape[1]
    k = o_sparse.keep_count(n_t, keep)
    tl, cn = tiles.cpu().numpy(), counts.cpu().numpy()
    swaps = 0
    for h in range(qbar.shape[0]):
        for g in range(qbar.shape[1]):
            assert cn[h, g] == k
            row = tl[h, g, :k]
            assert np.all((row >= 0) & (row < n_t))
            assert np.all(np.diff(row) > 0), "kept tiles must be increasing"
            if list(row) == kept_ref[h][g]:
                continue
            swaps += 1
            cut = np.sort(scores[h, g])[::-1][k - 1]
            assert np.all(scores[h, g][row] >= cut - SCORE_TOL), (h, g)
    return swaps


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("keep", [0.25, 0.5, 1.0])
def test_select_matches_oracle(case, keep):
    wl = _variant(case)
    gc, oc = build_caches(wl)
    q, _, _ = current_qkv(wl)
    qd = to_dev(q, "bf16")
    tiles, counts = nomas.sparse_select(gc, 0, qd, wl.n_video, wl.n_text, keep)
    kc, _ = oc.cache_kv(0)
    swaps = _check_selection(tiles, counts, o_sparse.group_means(q), o_sparse.tile_means(kc), keep)
    assert swaps <= 1


@pytest.mark.parametrize("name", ["c2_bf16_hist8", "c3_int8_window18", "c4_bf16_hist60"])
def test_select_full_size(name):
    wl = CONFIGS[name]
    gc, oc = build_caches(wl)
    q, _, _ = current_qkv(wl)
    tiles, counts = nomas.sparse_select(gc, 0, to_dev(q, "bf16"), wl.n_video, wl.n_text, 0.25)
    kc, _ = oc.cache_kv(0)
    qbar, kbar = o_sparse.group_means(q), o_sparse.tile_means(kc)
    swaps = _check_selection(tiles, counts, qbar, kbar, 0.25)
    assert swaps <= max(1, qbar.shape[0] * qbar.shape[1] // 50)


def test_select_planted_tile_always_kept_and_empty_cache():
    # 6 frames of 9 x 15 tokens: 810 resident slots, tiles 0..6 (the last partial)
    wl = small_variant(_variant(1), cache_frames_hist=(6,), past_frames=0, capacity_frames=8)
    from synth import segment_kv
    k, v = segment_kv(wl, 0, 6, 0)
    k = k.copy()
    k[5 * 128:6 * 128] += 1.0       # tile 5's keys share a +1 offset
    q, _, _ = current_qkv(wl)
    q = q + 1.0                      # and so do all queries: tile 5 scores ~128
    gc = nomas.KVCache(1, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, 0, wl.cache_dtype)
    tiles, counts = nomas.sparse_select(gc, 0, to_dev(q, "bf16"), wl.n_video, wl.n_text, 0.25)
    assert int(counts.abs().sum()) == 0  # nothing resident yet
    gc.append(to_dev(k, "bf16"), to_dev(v, "bf16"))
    tiles, counts = nomas.sparse_select(gc, 0, to_dev(q, "bf16"), wl.n_video, wl.n_text, 1e-6)
    assert torch.all(counts == 1)
    assert torch.all(tiles[..., 0] == 5)


@pytest.mark.parametrize("cache_dtype", ["bf16", "int8"])
def test_select_exact_ties_go_to_the_lower_tile(cache_dtype):
    # Eight resident tiles (one 8 x 16 frame each) whose keys are identical
    # except that tiles 2 and 6 are scaled up: their mean keys, and so their
    # scores, are exactly equal within each group of equal tiles.  Keeping 4
    # of 8 takes tiles 2 and 6 (the larger scores, given a positive mean query)
    # and then the two lowest of the tied rest, 0 and 1.
    from synth import segment_kv
    wl = small_variant(_variant(1), heads=2, grid_h=8, grid_w=16, cache_frames_hist=(8,), cur_frames=1, n_text=0,
                       cache_dtype=cache_dtype, past_frames=0, capacity_frames=8)
    k1, v1 = segment_kv(wl, 0, 1, 0)
    k = np.concatenate([k1] * 8, axis=0).copy()
    v = np.concatenate([v1] * 8, axis=0)
    k += 0.5                                   # positive mean key in every tile
    k[2 * 128:3 * 128] *= 2.0
    k[6 * 128:7 * 128] *= 2.0
    q, _, _ = current_qkv(wl)
    q = np.abs(q) + 0.1                        # positive mean query: larger keys score higher
    gc = nomas.KVCache(1, wl.heads, wl.grid_h, wl.grid_w, 8, 0, cache_dtype)
    gc.append(to_dev(k, "bf16"), to_dev(v, "bf16"))
    tiles, counts = nomas.sparse_select(gc, 0, to_dev(q, "bf16"), wl.n_video, wl.n_text, 0.5)
    torch.cuda.synchronize()
    assert torch.all(counts == 4)
    for h in range(wl.heads):
        assert tiles[h, 0, :4].tolist() == [0, 1, 2, 6]
    # keep one of eight: the lower of the two largest
    tiles, counts = nomas.sparse_select(gc, 0, to_dev(q, "bf16"), wl.n_video, wl.n_text, 0.125)
    assert torch.all(counts == 1) and torch.all(tiles[..., 0] == 2)


def _oracle_inputs(wl, oc, q, k):
    qr = o_rope.rope3d_segment(q, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    kr = o_rope.rope3d_segment(k, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    kc, vc = oc.cache_kv(0)
    return qr, kr, kc, vc


def _gpu_sparse(wl, gc, q, k, v, tiles, counts, num_splits):
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    nomas.rope3d(qd, kd, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    lse = torch.empty((wl.heads, wl.n_q), dtype=torch.float32, device="cuda")
    nbytes = gc.workspace_bytes(wl.n_video, wl.n_text, num_splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    out = nomas.segment_attn_sparse(gc, 0, qd, kd, vd, wl.n_video, wl.n_text, tiles, counts, lse=lse,
                                    workspace=ws, num_splits=num_splits)
    return out, lse, (qd, kd, vd, ws)


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_sparse_attention_matches_oracle(case, splits):
    wl = _variant(case)
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    qr, kr, kc, vc = _oracle_inputs(wl, oc, q, k)
    kept, _ = o_sparse.select_tiles(o_sparse.group_means(qr), o_sparse.tile_means(kc), 0.25)
    ref_o, ref_lse = o_sparse.sparse_segment_attention(qr, kr, v, kc, vc, o_attn.default_scale(128), kept)
    tiles, counts = _lists_to_device(kept, len(kept[0][0]))
    out, lse, _ = _gpu_sparse(wl, gc, q, k, v, tiles, counts, splits)
    assert_attn_close(out, ref_o, lse, ref_lse)


@pytest.mark.parametrize("splits", [1, 4])
def test_sparse_attention_per_group_lists_of_any_length(splits):
    # every (head, group) keeps a different number of tiles, 0 included
    wl = _variant(0)
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    qr, kr, kc, vc = _oracle_inputs(wl, oc, q, k)
    n_t = -(-kc.shape[0] // 128)
    rng = np.random.default_rng(11)
    groups = -(-wl.n_q // 512)
    kept = [[sorted(rng.choice(n_t, size=int(rng.integers(0, n_t + 1)), replace=False).tolist())
             for _ in range(groups)] for _ in range(wl.heads)]
    kept[0][0] = []
    kept[-1][-1] = list(range(n_t))
    ref_o, ref_lse = o_sparse.sparse_segment_attention(qr, kr, v, kc, vc, o_attn.default_scale(128), kept)
    tiles, counts = _lists_to_device(kept, n_t)
    out, lse, _ = _gpu_sparse(wl, gc, q, k, v, tiles, counts, splits)
    assert_attn_close(out, ref_o, lse, ref_lse)


def test_sparse_full_size_sampled_int8():
    wl = CONFIGS["c3_int8_window18"]
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    qr, kr, kc, vc = _oracle_inputs(wl, oc, q, k)
    kept, _ = o_sparse.select_tiles(o_sparse.group_means(qr), o_sparse.tile_means(kc), 0.25)
    rng = np.random.default_rng(wl.seed)
    rows = np.array(sorted(set(rng.choice(wl.n_q, 64, replace=False).tolist())
                           | {0, 511, 512, wl.n_video - 1, wl.n_video, wl.n_q - 1}))
    ref_o, ref_lse = o_sparse.sparse_segment_attention(qr, kr, v, kc, vc, o_attn.default_scale(128), kept,
                                                       rows=rows)
    tiles, counts = _lists_to_device(kept, len(kept[0][0]))
    out, lse, _ = _gpu_sparse(wl, gc, q, k, v, tiles, counts, 0)
    assert_attn_close(out, ref_o, lse, ref_lse, rows=rows)


@pytest.mark.parametrize("case", [0, 1])
@pytest.mark.parametrize("splits", [1, 4])
def test_keep_all_is_bitwise_dense(case, splits):
    wl = _variant(case)
    gc, _ = build_caches(wl)
    q, k, v = current_qkv(wl)
    n_t = -(-gc.valid_frames * gc.tpf // 128)
    groups = -(-wl.n_q // 512)
    kept = [[list(range(n_t))] * groups] * wl.heads
    tiles, counts = _lists_to_device(kept, n_t)
    out_s, lse_s, (qd, kd, vd, ws) = _gpu_sparse(wl, gc, q, k, v, tiles, counts, splits)
    lse_d = torch.empty_like(lse_s)
    out_d = nomas.segment_attn(gc, 0, qd, kd, vd, wl.n_video, wl.n_text, lse=lse_d, workspace=ws,
                               num_splits=splits)
    assert torch.equal(out_s, out_d) and torch.equal(lse_s, lse_d)


def test_empty_lists_with_empty_splits_attend_current_keys_only():
    # one current key tile, four splits: three splits see no tile at all
    wl = small_variant(_variant(0), cur_frames=1, n_text=20)
    assert wl.n_q <= 128
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    qr, kr, kc, vc = _oracle_inputs(wl, oc, q, k)
    ref_o, ref_lse = o_attn.segment_attention(qr, kr, v, kc[:0], vc[:0], o_attn.default_scale(128))
    tiles, counts = _lists_to_device([[[]]] * wl.heads, 1)
    out, lse, _ = _gpu_sparse(wl, gc, q, k, v, tiles, counts, 4)
    assert_attn_close(out, ref_o, lse, ref_lse)


def test_out_of_range_entry_is_reported_and_contained():
    wl = _variant(1)
    gc, _ = build_caches(wl)
    q, k, v = current_qkv(wl)
    n_t = -(-gc.valid_frames * gc.tpf // 128)
    groups = -(-wl.n_q // 512)
    kept = [[[0, n_t + 7]] * groups] * wl.heads
    tiles, counts = _lists_to_device(kept, 2)
    out, lse, _ = _gpu_sparse(wl, gc, q, k, v, tiles, counts, 1)
    torch.cuda.synchronize()
    assert nomas.device_error(clear=True) == nomas.NOMAS_ERR_INVALID_ARG
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_reused_key_means_give_the_same_lists():
    # the mean keys of an unchanged cache serve every step of a turn
    wl = _variant(2)
    gc, _ = build_caches(wl)
    n_t = -(-gc.valid_frames * gc.tpf // 128)
    ws = torch.empty(max(256, n_t * wl.heads * 512), dtype=torch.uint8, device="cuda")
    for step in range(3):
        q, _, _ = current_qkv(wl, step=step)
        qd = to_dev(q, "bf16")
        fresh = nomas.sparse_select(gc, 0, qd, wl.n_video, wl.n_text, 0.25)
        reused = nomas.sparse_select(gc, 0, qd, wl.n_video, wl.n_text, 0.25, workspace=ws,
                                     reuse_key_means=step > 0)
        assert torch.equal(fresh[0], reused[0]) and torch.equal(fresh[1], reused[1])
