"""CPU-only checks of the C ABI library: it loads without a GPU, exports every
entry point the header declares, and its host-side logic (descriptor checks,
append planning, byte accounting) agrees with the oracle's cache model.
No call here launches a kernel.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import segment_causal_kv_int8_b300 as nomas
from oracle import ring_cache

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "nomas.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nomas_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_are_exported_and_bound():
    names = _declared()
    assert "nomas_segment_attn" in names and "nomas_rope3d_apply" in names
    lib = ctypes.CDLL(nomas.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
        assert n in nomas.EXPORTS, n


def _desc(blocks=1, heads=2, gh=3, gw=4, cap=5, past=0, dtype=nomas.NOMAS_INT8, total=0, valid=0):
    return nomas.nomas_kvcache(blocks, heads, 128, gh, gw, cap, past, dtype, 256, 512, 1024, 2048, total, valid, 0)


def test_descriptor_validation():
    ok = _desc()
    assert nomas.nomas_kvcache_validate(ctypes.byref(ok)) == nomas.NOMAS_OK
    cases = [
        (dict(past=3, cap=5), nomas.NOMAS_ERR_INVALID_ARG),       # window != capacity
        (dict(dtype=7), nomas.NOMAS_ERR_INVALID_ARG),
        (dict(heads=0), nomas.NOMAS_ERR_INVALID_ARG),
        (dict(total=3, valid=2), nomas.NOMAS_ERR_INVALID_ARG),    # inconsistent metadata
    ]
    for kw, want in cases:
        d = _desc(**kw)
        assert nomas.nomas_kvcache_validate(ctypes.byref(d)) == want, kw
    d = _desc()
    d.head_dim = 64
    assert nomas.nomas_kvcache_validate(ctypes.byref(d)) == nomas.NOMAS_ERR_UNSUPPORTED
    d = _desc()
    d.k = 257  # misaligned
    assert nomas.nomas_kvcache_validate(ctypes.byref(d)) == nomas.NOMAS_ERR_INVALID_ARG
    d = _desc()
    d.k_scale = None
    assert nomas.nomas_kvcache_validate(ctypes.byref(d)) == nomas.NOMAS_ERR_INVALID_ARG
    d = _desc(dtype=nomas.NOMAS_BF16)
    d.k_scale = d.v_scale = None
    assert nomas.nomas_kvcache_validate(ctypes.byref(d)) == nomas.NOMAS_OK


def _plan(d, n):
    f, s, t, v = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int32()
    st = nomas.nomas_kvcache_plan_append(ctypes.byref(d), n, f, s, t, v)
    return st, f.value, s.value, t.value, v.value


@pytest.mark.parametrize("window", [0, 1, 4, 18])
def test_plan_append_matches_oracle_ring(window):
    rng = np.random.default_rng(window)
    cap = window if window else 40
    d = _desc(cap=cap, past=window)
    o = ring_cache.RingCache(1, 2, 128, 3, 4, cap, window, "int8", store=False)
    for _ in range(50):
        n = int(rng.integers(0, 3 * cap // 2 + 2))
        st, first, slot, total, valid = _plan(d, n)
        try:
            plan = o.plan_append(n)
        except ring_cache.CapacityError:
            assert st == nomas.NOMAS_ERR_CAPACITY
            continue
        assert st == nomas.NOMAS_OK
        if plan:
            assert first == plan[0][0] and slot == plan[0][2]
        else:
            assert first == n
        o.append(n_frames=n)
        assert (total, valid) == (o.total_frames, o.valid_frames)
        d.total_frames, d.valid_frames = total, valid


def test_kvcache_bytes_matches_oracle_and_archive_arithmetic():
    for dtype, code in (("int8", nomas.NOMAS_INT8), ("bf16", nomas.NOMAS_BF16)):
        d = _desc(blocks=54, heads=16, gh=23, gw=40, cap=30, dtype=code)
        o = ring_cache.RingCache(54, 16, 128, 23, 40, 30, 0, dtype, store=False)
        assert nomas.nomas_kvcache_bytes(ctypes.byref(d)) == o.bytes()
    d = _desc(blocks=54, heads=16, gh=23, gw=40, cap=30)
    # within 0.5% of the 5.881 GiB per 30-frame segment the page logs
    assert abs(nomas.nomas_kvcache_bytes(ctypes.byref(d)) / 2 ** 30 / 5.881 - 1) < 0.005


def test_invalid_calls_return_status_without_launching():
    d = _desc()
    # null q
    assert nomas.nomas_rope3d_apply(None, None, nomas.NOMAS_BF16, 12, 2, 128, 256, 1, 3, 4, 0, 1e4, 32, 48, 48,
                                    None) == nomas.NOMAS_ERR_INVALID_ARG
    # n_video inconsistent with frames*grid
    assert nomas.nomas_rope3d_apply(256, None, nomas.NOMAS_BF16, 11, 2, 128, 256, 1, 3, 4, 0, 1e4, 32, 48, 48,
                                    None) == nomas.NOMAS_ERR_INVALID_ARG
    # odd rotary split
    assert nomas.nomas_rope3d_apply(256, None, nomas.NOMAS_BF16, 12, 2, 128, 256, 1, 3, 4, 0, 1e4, 31, 48, 48,
                                    None) == nomas.NOMAS_ERR_INVALID_ARG
    # more heads than a token row's vector index covers (checked before the row stride)
    heads = 2 ** 19 + 1
    assert nomas.nomas_rope3d_apply(256, None, nomas.NOMAS_BF16, 12, heads, 128, heads * 128, 1, 3, 4, 0, 1e4, 32,
                                    48, 48, None) == nomas.NOMAS_ERR_UNSUPPORTED
    # append: bad dtype, then capacity overflow (checked before any launch)
    assert nomas.nomas_kvcache_append(ctypes.byref(d), 256, 256, 9, 1, 0, None) == nomas.NOMAS_ERR_INVALID_ARG
    assert nomas.nomas_kvcache_append(ctypes.byref(d), 256, 256, nomas.NOMAS_BF16, 6, 0,
                                      None) == nomas.NOMAS_ERR_CAPACITY
    assert d.total_frames == 0
    # attention: block out of range, non-positive scale
    assert nomas.nomas_segment_attn(ctypes.byref(d), 1, 256, 256, 256, 12, 0, 0.1, 256, None, None, 0, 0,
                                    None) == nomas.NOMAS_ERR_INVALID_ARG
    assert nomas.nomas_segment_attn(ctypes.byref(d), 0, 256, 256, 256, 12, 0, 0.0, 256, None, None, 0, 0,
                                    None) == nomas.NOMAS_ERR_INVALID_ARG
    # zero-length work is a no-op that succeeds without touching the device
    assert nomas.nomas_segment_attn(ctypes.byref(d), 0, 256, 256, 256, 0, 0, 0.1, 256, None, None, 0, 0,
                                    None) == nomas.NOMAS_OK
    assert nomas.nomas_kvcache_append(ctypes.byref(d), None, None, nomas.NOMAS_BF16, 0, 0, None) == nomas.NOMAS_OK


def test_expand_validates_before_launching():
    src = _desc(total=2, valid=2)

    def bf16(**kw):
        d = _desc(dtype=nomas.NOMAS_BF16, **kw)
        d.k, d.v, d.k_scale, d.v_scale = 4096, 8192, None, None
        return d

    exp = nomas.nomas_kvcache_expand
    dst = bf16()
    # a one-byte destination, a BF16 source, a geometry mismatch, shared buffers
    assert exp(ctypes.byref(src), ctypes.byref(_desc()), None) == nomas.NOMAS_ERR_INVALID_ARG
    assert exp(ctypes.byref(bf16(total=2, valid=2)), ctypes.byref(dst), None) == nomas.NOMAS_ERR_INVALID_ARG
    for kw in (dict(heads=3), dict(gw=5), dict(cap=6), dict(blocks=2)):
        assert exp(ctypes.byref(src), ctypes.byref(bf16(**kw)), None) == nomas.NOMAS_ERR_INVALID_ARG, kw
    shared = bf16()
    shared.k = src.k
    assert exp(ctypes.byref(src), ctypes.byref(shared), None) == nomas.NOMAS_ERR_INVALID_ARG
    assert exp(ctypes.byref(src), None, None) == nomas.NOMAS_ERR_INVALID_ARG
    # nothing failed, so nothing was copied into the destination's metadata
    assert dst.total_frames == 0 and dst.valid_frames == 0


def test_camera_cross_attention_validates_before_launching():
    cam = nomas.nomas_camera_cross_attn
    # frames, grid_h, grid_w, heads, n_cam, scale; fake 256-aligned pointers never reach a launch
    ok = dict(frames=2, gh=3, gw=4, heads=2, n_cam=4, scale=0.1)

    def call(q=256, k=256, v=256, out=256, **kw):
        a = dict(ok, **kw)
        return cam(q, k, v, a["frames"], a["gh"], a["gw"], a["heads"], a["n_cam"], a["scale"], out, None)

    assert call(n_cam=0) == nomas.NOMAS_ERR_INVALID_ARG
    assert call(n_cam=17) == nomas.NOMAS_ERR_UNSUPPORTED
    assert call(heads=0) == nomas.NOMAS_ERR_INVALID_ARG
    assert call(heads=65536) == nomas.NOMAS_ERR_UNSUPPORTED   # one grid row per head
    assert call(frames=-1) == nomas.NOMAS_ERR_INVALID_ARG
    assert call(frames=65536) == nomas.NOMAS_ERR_UNSUPPORTED
    assert call(scale=0.0) == nomas.NOMAS_ERR_INVALID_ARG
    assert call(scale=float("nan")) == nomas.NOMAS_ERR_INVALID_ARG
    assert call(q=None) == nomas.NOMAS_ERR_INVALID_ARG
    assert call(out=None) == nomas.NOMAS_ERR_INVALID_ARG
    assert call(k=264) == nomas.NOMAS_ERR_INVALID_ARG          # not 16-byte aligned (TMA)
    assert call(frames=0, q=None, k=None, v=None, out=None) == nomas.NOMAS_OK  # nothing to do


def _round256(x):
    return -(-x // 256) * 256


def test_workspace_bytes_for_explicit_splits():
    # INT8 window of 18 frames, 7360 + 256 queries: 30 blocks of 256 rows per
    # head form 15 CTA-pair units, 240 units in all.  Four pieces of every unit
    # keep float32 partial rows of 128 values plus a log-sum-exp per piece, per
    # CTA of the pair, per row of its 256-row block.
    d = _desc(heads=16, gh=23, gw=40, cap=18, past=18, total=24, valid=18)
    out = ctypes.c_size_t()
    assert nomas.nomas_segment_attn_workspace_bytes(ctypes.byref(d), 7360, 256, 1, out) == nomas.NOMAS_OK
    assert out.value == 0
    assert nomas.nomas_segment_attn_workspace_bytes(ctypes.byref(d), 7360, 256, 4, out) == nomas.NOMAS_OK
    rows = 16 * 15 * 4 * 2 * 256
    assert out.value == _round256(rows * 128 * 4) + _round256(rows * 4)
    pl = nomas.nomas_attn_plan()
    assert nomas.nomas_segment_attn_plan(ctypes.byref(d), 7360, 256, 4, ctypes.byref(pl)) == nomas.NOMAS_OK
    assert (pl.units, pl.whole_units, pl.pieces_per_split_unit, pl.ctas_per_unit) == (240, 0, 4, 2)
    assert pl.work_items == 960 and pl.workspace_bytes == out.value


@pytest.mark.parametrize("dtype,frames,cur,slots", [
    (nomas.NOMAS_BF16, 60, 8, 148),   # 60-frame BF16 history: 16 x 30 units of 256 rows
    (nomas.NOMAS_INT8, 18, 8, 74),    # INT8 window of 18 frames: 16 x 15 CTA-pair units
    (nomas.NOMAS_BF16, 8, 4, 148),    # 8-frame BF16 history, 4-frame segment: 16 x 16 units
])
def test_automatic_plan_is_consistent(dtype, frames, cur, slots):
    # Without a GPU the plan assumes a full B300 (148 SMs, 74 CTA pairs).  The
    # whole units fill whole waves; the pieces of the split units make a
    # complete work list; the workspace holds exactly their partial rows.
    past = frames if dtype == nomas.NOMAS_INT8 else 0
    d = _desc(heads=16, gh=23, gw=40, cap=max(frames, 68), dtype=dtype, past=past, total=frames, valid=frames)
    if past:
        d.capacity_frames = frames
    assert nomas.nomas_kvcache_validate(ctypes.byref(d)) == nomas.NOMAS_OK
    nv = cur * 920
    pl = nomas.nomas_attn_plan()
    assert nomas.nomas_segment_attn_plan(ctypes.byref(d), nv, 256, 0, ctypes.byref(pl)) == nomas.NOMAS_OK
    ctas = 2 if dtype == nomas.NOMAS_INT8 else 1
    blocks = -(-(nv + 256) // 256)
    assert pl.ctas_per_unit == ctas and pl.units == 16 * -(-blocks // ctas)
    split_units = pl.units - pl.whole_units
    assert pl.work_items == pl.whole_units + split_units * pl.pieces_per_split_unit
    if pl.pieces_per_split_unit == 1:
        assert split_units == 0 and pl.workspace_bytes == 0
    else:
        assert pl.whole_units % slots == 0
        rows = split_units * pl.pieces_per_split_unit * ctas * 256
        assert pl.workspace_bytes == _round256(rows * 512) + _round256(rows * 4)
    out = ctypes.c_size_t()
    assert nomas.nomas_segment_attn_workspace_bytes(ctypes.byref(d), nv, 256, 0, out) == nomas.NOMAS_OK
    assert out.value == pl.workspace_bytes
    if frames >= 18:
        # the two long-history shapes: 3 whole waves, the 36 (BF16) or 18
        # (pair) units of the fourth wave cut into pieces that run as one wave
        assert pl.whole_units == 3 * slots and split_units * pl.pieces_per_split_unit <= slots
        assert pl.pieces_per_split_unit >= 2


def test_archive_frame_bytes_matches_the_archive_growth_on_the_page():
    # One archived frame holds INT8 K and V codes plus a float32 scale per
    # (block, head, token); 30 frames of a segment at 54 x 16 x 128 on a 23x40
    # grid come within 0.5% of the growth the page logs per segment.
    d = _desc(blocks=54, heads=16, gh=23, gw=40, cap=18)
    d.past_frames = 18
    fb = nomas.nomas_kvcache_archive_frame_bytes(ctypes.byref(d))
    assert fb == 2 * 54 * 16 * 23 * 40 * (128 + 4)
    for gib_logged, segments in ((5.881, 1), (11.763, 2), (17.644, 3)):
        assert abs(segments * 30 * fb / 2 ** 30 / gib_logged - 1) < 0.005
    d16 = _desc(blocks=54, heads=16, gh=23, gw=40, cap=18, dtype=nomas.NOMAS_BF16)
    d16.past_frames = 18
    assert nomas.nomas_kvcache_archive_frame_bytes(ctypes.byref(d16)) == 0


def test_sparse_entry_points_validate_before_launching():
    # 2 heads, 23 x 40 grid, 18 resident frames: 16560 slots -> 130 tiles
    d = _desc(heads=2, gh=23, gw=40, cap=18, past=18, total=24, valid=18)
    out = ctypes.c_size_t()
    assert nomas.nomas_sparse_select_workspace_bytes(ctypes.byref(d), 7360, 256, out) == nomas.NOMAS_OK
    n_tiles = 130
    assert out.value == -(-2 * n_tiles * 512 // 256) * 256
    k = nomas.sparse_keep_count(n_tiles, 0.25)
    assert k == 33  # ceil(32.5)
    ws = 1 << 20
    # keep fraction outside (0, 1]
    for keep in (0.0, -0.5, 1.5, float("nan")):
        assert nomas.nomas_sparse_select(ctypes.byref(d), 0, 256, 7360, 256, keep, 256, 256, k, 0, ws,
                                         out.value, None) == nomas.NOMAS_ERR_INVALID_ARG
    # rows shorter than the kept count, missing workspace, block out of range
    assert nomas.nomas_sparse_select(ctypes.byref(d), 0, 256, 7360, 256, 0.25, 256, 256, k - 1, 0, ws,
                                     out.value, None) == nomas.NOMAS_ERR_INVALID_ARG
    assert nomas.nomas_sparse_select(ctypes.byref(d), 0, 256, 7360, 256, 0.25, 256, 256, k, 0, None,
                                     0, None) == nomas.NOMAS_ERR_INVALID_ARG
    assert nomas.nomas_sparse_select(ctypes.byref(d), 1, 256, 7360, 256, 0.25, 256, 256, k, 0, ws,
                                     out.value, None) == nomas.NOMAS_ERR_INVALID_ARG
    # more than 8192 resident tiles
    big = _desc(heads=2, gh=128, gw=128, cap=70, total=70, valid=70)
    assert nomas.nomas_sparse_select(ctypes.byref(big), 0, 256, 128, 0, 0.25, 256, 256, 9000, 0, ws,
                                     1 << 30, None) == nomas.NOMAS_ERR_UNSUPPORTED
    # sparse attention without lists
    assert nomas.nomas_segment_attn_sparse(ctypes.byref(d), 0, 256, 256, 256, 7360, 256, 0.1, None, 256, k, 256,
                                           None, None, 0, 0, None) == nomas.NOMAS_ERR_INVALID_ARG
    assert nomas.nomas_segment_attn_sparse(ctypes.byref(d), 0, 256, 256, 256, 7360, 256, 0.1, 256, 256, 0, 256,
                                           None, None, 0, 0, None) == nomas.NOMAS_ERR_INVALID_ARG


def test_fp8_descriptor_is_a_quantised_cache():
    d = _desc(dtype=nomas.NOMAS_FP8)
    assert nomas.nomas_kvcache_validate(ctypes.byref(d)) == nomas.NOMAS_OK
    i8 = _desc(dtype=nomas.NOMAS_INT8)
    assert nomas.nomas_kvcache_bytes(ctypes.byref(d)) == nomas.nomas_kvcache_bytes(ctypes.byref(i8))
    assert nomas.nomas_kvcache_archive_frame_bytes(ctypes.byref(d)) == 2 * 1 * 2 * 12 * (128 + 4)
    d.k_scale = None  # scales are required, as for INT8
    assert nomas.nomas_kvcache_validate(ctypes.byref(d)) == nomas.NOMAS_ERR_INVALID_ARG
    # an FP8 input dtype is not an input format
    d = _desc(dtype=nomas.NOMAS_FP8)
    assert nomas.nomas_kvcache_append(ctypes.byref(d), 256, 256, nomas.NOMAS_FP8, 1, 0,
                                      None) == nomas.NOMAS_ERR_INVALID_ARG


def test_descriptor_round_trips_through_its_bytes():
    # the session state's host half is a plain struct: its bytes restore it
    d = _desc(heads=16, gh=23, gw=40, cap=18, past=18, total=40, valid=18)
    r = nomas.nomas_kvcache.from_buffer_copy(bytes(d))
    assert nomas.nomas_kvcache_validate(ctypes.byref(r)) == nomas.NOMAS_OK
    outs = []
    for desc in (d, r):
        ff, sf, vt = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        nt = ctypes.c_int64()
        assert nomas.nomas_kvcache_plan_append(ctypes.byref(desc), 8, ctypes.byref(ff), ctypes.byref(sf),
                                               ctypes.byref(nt), ctypes.byref(vt)) == nomas.NOMAS_OK
        outs.append((ff.value, sf.value, nt.value, vt.value))
    assert outs[0] == outs[1] == (0, 40 % 18, 48, 18)


def test_bench_flop_accounting_is_consistent():
    # the executed-FLOP counts bench.py reports for block-sparse runs
    import bench
    from synth import CONFIGS
    wl = CONFIGS["c3_int8_window18"]
    n_t = -(-wl.n_cache // 128)
    groups = -(-wl.n_q // 512)
    every = np.tile(np.arange(n_t, dtype=np.int32), (wl.heads, groups, 1))
    full = np.full((wl.heads, groups), n_t, np.int32)
    assert bench.sparse_flops(wl, every, full) == wl.attn_flops()
    none = np.zeros((wl.heads, groups), np.int32)
    assert bench.sparse_flops(wl, every, none) == 4.0 * wl.n_q * wl.n_q * 128 * wl.heads
    s5 = CONFIGS["c5_session12"]
    assert bench.session_flops(s5, 12, keep=1.0) == bench.session_flops(s5, 12)
    assert bench.session_flops(s5, 12, keep=0.25) < bench.session_flops(s5, 12)


def test_bench_traffic_provenance_reads_for_every_config():
    # bench.py takes roofline.traffic from the committed ncu summary only while
    # the attention sources hash the same; every config must get an answer
    # (a number, or None with the reason), never an error.
    import bench
    from synth import CONFIG_ORDER
    for name in CONFIG_ORDER:
        traffic, source = bench._load_traffic(name)
        assert traffic is None or traffic > 0
        assert isinstance(source, str) and source
    for rel in bench.ATTN_SOURCES:
        assert os.path.exists(os.path.join(ROOT, rel)), rel
