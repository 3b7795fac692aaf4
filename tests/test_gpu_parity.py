"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Every expected value comes from the oracle on the same seeded inputs; nothing
the GPU produces is fed back into the oracle.
"""
import numpy as np
import pytest
import torch

from synth import CONFIGS, current_qkv, segment_kv, small_variant

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import segment_causal_kv_int8_b300 as nomas
    from _gpu_common import (ROPE_REL, assert_attn_close, build_caches, f64, gpu_segment, oracle_segment,
                             to_dev)
    from oracle import attention as o_attn
    from oracle import int8_codec, ring_cache
    from oracle import rope3d as o_rope


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()
    assert nomas.device_error(clear=True) == 0


# ------------------------------------------------------------------ RoPE
@pytest.mark.parametrize("name", ["c1_tiny", "c2_bf16_hist8", "c3_int8_window18", "c4_bf16_hist60"])
def test_rope3d_matches_oracle(name):
    wl = CONFIGS[name]
    q, k, _ = current_qkv(wl)
    qd, kd = to_dev(q, wl.io_dtype), to_dev(k, wl.io_dtype)
    nomas.rope3d(qd, kd, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    for dev, host in ((qd, q), (kd, k)):
        ref = o_rope.rope3d_segment(host, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
        got = f64(dev)
        nv = wl.n_video
        # text rows untouched, bit for bit
        np.testing.assert_array_equal(got[nv:], host[nv:].astype(np.float64))
        d = np.abs(got[:nv] - ref[:nv])
        vec_inf = np.max(np.abs(ref[:nv]), axis=2, keepdims=True)
        if wl.io_dtype == "f32":
            assert np.max(np.max(d, axis=2, keepdims=True) / vec_inf) <= ROPE_REL
        else:
            # one bf16 rounding of a float32 result within 1e-5 of the exact value
            assert np.all(d <= 2.0 ** -8 * np.abs(ref[:nv]) + ROPE_REL * vec_inf)


@pytest.mark.parametrize("io_dtype", ["bf16", "f32"])
def test_rope3d_padded_token_rows(io_dtype):
    # Token rows farther apart than heads x 128 (Q and K viewed out of wider
    # buffers): the kernel for strided rows, against the oracle; the padding
    # between rows is left untouched.
    wl = small_variant(CONFIGS["c2_bf16_hist8"], heads=3, grid_h=5, grid_w=7, cur_frames=3, n_text=4,
                       io_dtype=io_dtype, seed=77)
    q, k, _ = current_qkv(wl)
    for src in (q, k):
        wide = torch.full((wl.n_q, wl.heads + 2, 128), 7.0, dtype=torch.bfloat16 if io_dtype == "bf16" else
                          torch.float32, device="cuda")
        wide[:, :wl.heads] = to_dev(src, io_dtype)
        view = wide[:, :wl.heads]
        assert view.stride(0) == (wl.heads + 2) * 128
        nomas.rope3d(view, None, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
        ref = o_rope.rope3d_segment(src, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
        got = f64(view)
        nv = wl.n_video
        np.testing.assert_array_equal(got[nv:], src[nv:].astype(np.float64))
        d = np.abs(got[:nv] - ref[:nv])
        vec_inf = np.max(np.abs(ref[:nv]), axis=2, keepdims=True)
        if io_dtype == "f32":
            assert np.max(np.max(d, axis=2, keepdims=True) / vec_inf) <= ROPE_REL
        else:
            assert np.all(d <= 2.0 ** -8 * np.abs(ref[:nv]) + ROPE_REL * vec_inf)
        assert bool((wide[:, wl.heads:] == 7.0).all())


@pytest.mark.parametrize("heads", [8, 32, 64, 65])
def test_rope3d_head_counts(heads):
    # A warp streams one token row of 16 * heads vectors in batches of 256
    # (eight per lane): 8 heads fill half a batch, 32 and 64 heads take two and
    # four full batches, 65 heads five with a ragged last one (16 vectors).
    # 2760 video tokens on a 23 x 40 grid; Q and K both rotated, against the oracle.
    wl = small_variant(CONFIGS["c2_bf16_hist8"], heads=heads, grid_h=23, grid_w=40, cur_frames=3, n_text=5,
                       seed=90 + heads)
    q, k, _ = current_qkv(wl)
    qd, kd = to_dev(q, wl.io_dtype), to_dev(k, wl.io_dtype)
    nomas.rope3d(qd, kd, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    nv = wl.n_video
    for dev, host in ((qd, q), (kd, k)):
        ref = o_rope.rope3d_segment(host, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
        got = f64(dev)
        np.testing.assert_array_equal(got[nv:], host[nv:].astype(np.float64))
        d = np.abs(got[:nv] - ref[:nv])
        vec_inf = np.max(np.abs(ref[:nv]), axis=2, keepdims=True)
        assert np.all(d <= 2.0 ** -8 * np.abs(ref[:nv]) + ROPE_REL * vec_inf)


def test_rope3d_large_frame_index_and_odd_split():
    wl = small_variant(CONFIGS["c1_tiny"], io_dtype="f32", grid_h=3, grid_w=5, cur_frames=3, n_text=2)
    q, k, _ = current_qkv(wl)
    t0 = 1_000_003
    for split in ((32, 48, 48), (16, 24, 24)):
        qd = to_dev(q, "f32")
        nomas.rope3d(qd, None, wl.cur_frames, wl.grid_h, wl.grid_w, t0, 10000.0, split)
        ref = o_rope.rope3d_segment(q, wl.cur_frames, wl.grid_h, wl.grid_w, t0, 10000.0, split)
        got = f64(qd)
        vec_inf = np.max(np.abs(ref[:wl.n_video]), axis=2, keepdims=True)
        rel = np.max(np.abs(got[:wl.n_video] - ref[:wl.n_video]), axis=2, keepdims=True) / vec_inf
        assert rel.max() <= ROPE_REL


# ------------------------------------------------------------------ append
def _check_cache_bits(gc, oc):
    if oc.dtype in ("int8", "fp8"):
        np.testing.assert_array_equal(gc.k.cpu().numpy(), oc.k_codes)
        np.testing.assert_array_equal(gc.v.cpu().numpy(), oc.v_codes)
        np.testing.assert_array_equal(gc.k_scale.cpu().numpy().view(np.uint32), oc.k_scales.view(np.uint32))
        np.testing.assert_array_equal(gc.v_scale.cpu().numpy().view(np.uint32), oc.v_scales.view(np.uint32))
    else:
        np.testing.assert_array_equal(f64(gc.k), oc.k_vals)
        np.testing.assert_array_equal(f64(gc.v), oc.v_vals)
    assert gc.total_frames == oc.total_frames and gc.valid_frames == oc.valid_frames


@pytest.mark.parametrize("name", ["c1_tiny", "c2_bf16_hist8", "c3_int8_window18"])
def test_append_bit_exact(name):
    wl = CONFIGS[name]
    gc, oc = build_caches(wl)
    _check_cache_bits(gc, oc)


@pytest.mark.parametrize("in_dtype,cache_dtype", [("f32", "int8"), ("bf16", "int8"), ("f32", "bf16"),
                                                  ("bf16", "bf16"), ("f32", "fp8"), ("bf16", "fp8")])
def test_append_multi_block_window_wrap_and_long_segment(in_dtype, cache_dtype):
    # 3 blocks, window 4 frames: segments of 3, 2, 6 (longer than the window), 1 frames.
    blocks, heads, gh, gw, W = 3, 2, 3, 5, 4
    wl = small_variant(CONFIGS["c1_tiny"], heads=heads, grid_h=gh, grid_w=gw, io_dtype=in_dtype,
                       outlier_p=0.01)
    gc = nomas.KVCache(blocks, heads, gh, gw, W, W, cache_dtype)
    oc = ring_cache.RingCache(blocks, heads, 128, gh, gw, W, W, cache_dtype)
    for s, f in enumerate((3, 2, 6, 1)):
        kv = [segment_kv(wl, s, f, b) for b in range(blocks)]
        k = np.stack([x[0] for x in kv])
        v = np.stack([x[1] for x in kv])
        if s == 1:
            k[0, 3, 1] = 0.0  # an all-zero row
            v[2, 7, 0, :5] = 0.0
        gc.append(to_dev(k, in_dtype), to_dev(v, in_dtype))
        oc.append(k, v)
        _check_cache_bits(gc, oc)


@pytest.mark.parametrize("cache_dtype", ["int8", "fp8"])
def test_append_codec_edge_rows(cache_dtype):
    heads, gh, gw = 1, 1, 9
    rows = np.zeros((9, 128), np.float32)
    rows[1, :8] = [127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 126.5, -1.5]          # ties (inv = 1)
    rows[2] = np.linspace(-1e-39, 1e-39, 128, dtype=np.float32)              # subnormal, inv overflows
    rows[3] = np.linspace(-3e-37, 2e-37, 128, dtype=np.float32)              # tiny normal
    rows[4] = np.float32(3e38) * np.sin(np.arange(128, dtype=np.float32))    # huge
    rows[5, 17] = -8.0                                                       # single negative spike
    rows[6] = np.arange(-64, 64, dtype=np.float32)
    rows[7] = -rows[6]
    # absmax 448 (inv = 1 for FP8): E4M3 midpoints, subnormal midpoints, signed zero
    rows[8, :10] = [448.0, 1.0625, -1.0625, 7.5 * 2.0 ** -9, 0.5 * 2.0 ** -9, -0.5 * 2.0 ** -9, 1.5 * 2.0 ** -9,
                    232.0, -0.0, 3.0 * 2.0 ** -10]
    k = rows.reshape(1, 9, 1, 128)
    gc = nomas.KVCache(1, heads, gh, gw, 1, 0, cache_dtype)
    oc = ring_cache.RingCache(1, heads, 128, gh, gw, 1, 0, cache_dtype)
    gc.append(to_dev(k, "f32"), to_dev(k, "f32"))
    oc.append(k, k)
    _check_cache_bits(gc, oc)


def test_reset_and_capacity():
    wl = CONFIGS["c1_tiny"]
    gc, oc = build_caches(wl)
    k, v = segment_kv(wl, 9, 2, 0)
    with pytest.raises(nomas.NomasError) as e:
        gc.append(to_dev(k, "f32"), to_dev(v, "f32"))
    assert e.value.status == nomas.NOMAS_ERR_CAPACITY
    assert gc.total_frames == 2
    gc.reset(zero_memory=True)
    torch.cuda.synchronize()
    assert gc.total_frames == 0 and gc.valid_frames == 0
    assert int(gc.k.abs().sum()) == 0 and float(gc.k_scale.abs().sum()) == 0.0


# ------------------------------------------------------------------ attention
def test_attention_tiny_config_full():
    wl = CONFIGS["c1_tiny"]
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    # the attention computes in bf16: round the f32 activations once, on both sides
    from synth import round_to_bf16
    q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    ref_o, ref_lse = oracle_segment(wl, oc, q, k, v)
    for splits in (1, 2):
        out, lse = gpu_segment(wl, gc, q, k, v, num_splits=splits)
        assert_attn_close(out, ref_o, lse, ref_lse)


RAGGED = [
    # heads, grid, cached frames (hist), current frames, text, cache dtype, window
    dict(heads=3, grid_h=5, grid_w=7, cache_frames_hist=(2, 1), cur_frames=2, n_text=9, cache_dtype="int8",
         past_frames=0, capacity_frames=6),
    dict(heads=2, grid_h=5, grid_w=7, cache_frames_hist=(3, 3, 3), cur_frames=3, n_text=5, cache_dtype="int8",
         past_frames=4, capacity_frames=4),
    dict(heads=2, grid_h=9, grid_w=15, cache_frames_hist=(2,), cur_frames=3, n_text=40, cache_dtype="bf16",
         past_frames=0, capacity_frames=5),
    dict(heads=1, grid_h=4, grid_w=4, cache_frames_hist=(), cur_frames=1, n_text=0, cache_dtype="bf16",
         past_frames=0, capacity_frames=2),
    dict(heads=2, grid_h=16, grid_w=16, cache_frames_hist=(1,), cur_frames=1, n_text=0, cache_dtype="int8",
         past_frames=0, capacity_frames=2),
]


@pytest.mark.parametrize("case", range(len(RAGGED)))
@pytest.mark.parametrize("splits", [1, 3])
def test_attention_ragged_shapes(case, splits):
    # N(0,1) inputs: the domain the attention tolerance is stated for
    wl = small_variant(CONFIGS["c2_bf16_hist8"], **RAGGED[case], seed=100 + case)
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    ref_o, ref_lse = oracle_segment(wl, oc, q, k, v)
    out, lse = gpu_segment(wl, gc, q, k, v, num_splits=splits)
    assert_attn_close(out, ref_o, lse, ref_lse)


@pytest.mark.parametrize("case", range(len(RAGGED)))
def test_attention_tail_plans(case):
    # Plans that keep some units whole and cut the rest into pieces (the shape
    # the automatic plan takes on long histories), on ragged shapes.
    wl = small_variant(CONFIGS["c2_bf16_hist8"], **RAGGED[case], seed=200 + case)
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    ref_o, ref_lse = oracle_segment(wl, oc, q, k, v)
    qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
    nomas.rope3d(qd, kd, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    units = gc.attn_plan(wl.n_video, wl.n_text, 1)["units"]
    n_tiles = -(-wl.n_cache // 128) + -(-wl.n_q // 128)
    for whole, pieces in ((units - 1, 2), (max(0, units - 3), min(3, n_tiles)), (1, n_tiles), (0, 2)):
        if whole >= units or pieces < 2 or pieces > n_tiles:
            continue
        lse = torch.empty((wl.heads, wl.n_q), dtype=torch.float32, device="cuda")
        out = nomas.segment_attn_planned(gc, 0, qd, kd, vd, wl.n_video, wl.n_text, whole, pieces, lse=lse)
        assert_attn_close(out, ref_o, lse, ref_lse)


def _tile_rows(n_q, seed, per_tile=6):
    """At least ``per_tile`` query rows from every 128-row tile (its first and last row among them)."""
    rng = np.random.default_rng(seed)
    rows = set()
    for t0 in range(0, n_q, 128):
        t1 = min(n_q, t0 + 128)
        rows |= {t0, t1 - 1}
        rows |= set(rng.integers(t0, t1, size=per_tile - 2).tolist())
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["c2_bf16_hist8", "c3_int8_window18"])
def test_attention_full_size_every_row(name):
    # Every query row of every head, against the oracle, under the automatic
    # plan (a cut last wave on the INT8 window), an uncut plan, and a plan
    # with a cut tail forced on the BF16 history.
    wl = CONFIGS[name]
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    ref_o, ref_lse = oracle_segment(wl, oc, q, k, v)
    out, lse = gpu_segment(wl, gc, q, k, v, num_splits=0)
    assert_attn_close(out, ref_o, lse, ref_lse)
    out1, lse1 = gpu_segment(wl, gc, q, k, v, num_splits=1)
    assert_attn_close(out1, ref_o, lse1, ref_lse)
    if wl.cache_dtype == "bf16":
        qd, kd, vd = (to_dev(x, "bf16") for x in (q, k, v))
        nomas.rope3d(qd, kd, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
        lse2 = torch.empty_like(lse)
        out2 = nomas.segment_attn_planned(gc, 0, qd, kd, vd, wl.n_video, wl.n_text, 148, 4, lse=lse2)
        assert_attn_close(out2, ref_o, lse2, ref_lse)


def test_attention_full_size_every_tile_c4():
    # The 60-frame BF16 history: six rows of every 128-row query tile of every
    # head (the oracle's cost bounds the sample), automatic and uncut plans.
    wl = CONFIGS["c4_bf16_hist60"]
    gc, oc = build_caches(wl)
    q, k, v = current_qkv(wl)
    rows = _tile_rows(wl.n_q, wl.seed)
    ref_o, ref_lse = oracle_segment(wl, oc, q, k, v, rows=rows)
    plan = gc.attn_plan(wl.n_video, wl.n_text, 0)
    assert plan["pieces_per_split_unit"] > 1 and plan["whole_units"] > 0
    out, lse = gpu_segment(wl, gc, q, k, v, num_splits=0)
    assert_attn_close(out, ref_o, lse, ref_lse, rows=rows)
    out1, _ = gpu_segment(wl, gc, q, k, v, num_splits=1)
    assert_attn_close(out1, ref_o, rows=rows)


def test_attention_deterministic():
    wl = CONFIGS["c3_int8_window18"]
    gc, _ = build_caches(wl)
    q, k, v = current_qkv(wl)
    for splits in (1, 4):
        a, la = gpu_segment(wl, gc, q, k, v, num_splits=splits)
        b, lb = gpu_segment(wl, gc, q, k, v, num_splits=splits)
        assert torch.equal(a, b) and torch.equal(la, lb)


def test_invalid_arguments_launch_nothing():
    wl = CONFIGS["c1_tiny"]
    gc, _ = build_caches(wl)
    q = torch.zeros((wl.n_q, wl.heads, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nomas.NomasError) as e:
        nomas.segment_attn(gc, 5, q, q, q, wl.n_video, wl.n_text)
    assert e.value.status == nomas.NOMAS_ERR_INVALID_ARG
    with pytest.raises(nomas.NomasError) as e:
        nomas.segment_attn(gc, 0, q, q, q, wl.n_video, wl.n_text, softmax_scale=-1.0)
    assert e.value.status == nomas.NOMAS_ERR_INVALID_ARG
    with pytest.raises(nomas.NomasError) as e:
        nomas.segment_attn(gc, 0, q, q, q, wl.n_video, wl.n_text, num_splits=3)   # no workspace
    assert e.value.status == nomas.NOMAS_ERR_INVALID_ARG


def test_bounded_wait_reports_timeout_and_context_survives():
    # A kernel waits on a barrier nothing arrives on; after 50 ms it records the
    # timeout status and exits.  The context must stay usable afterwards.
    assert nomas.device_error(clear=True) == 0
    st = nomas.nomas_selftest_wait_timeout(50_000, nomas._stream_ptr())
    assert st == nomas.NOMAS_OK
    torch.cuda.synchronize()
    assert nomas.device_error(clear=True) == nomas.NOMAS_ERR_DEVICE_TIMEOUT
    assert nomas.device_error(clear=False) == 0
    assert nomas.nomas_selftest_wait_timeout(0, nomas._stream_ptr()) == nomas.NOMAS_ERR_INVALID_ARG
    x = torch.arange(16, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 120.0


def _poison(dtype):
    return {torch.int8: -77, torch.uint8: 165}.get(dtype, -12288.0)  # exact in bf16 and fp32


def _guarded(shape, dtype, guard=4096):
    """A tensor viewed out of the middle of a larger one whose ends hold a poison pattern."""
    n = int(np.prod(shape))
    big = torch.empty(n + 2 * guard, dtype=dtype, device="cuda")
    big.fill_(_poison(dtype))
    return big, big[guard:guard + n].view(*shape), guard


def _guards_intact(big, guard, dtype):
    ends = torch.cat([big[:guard], big[-guard:]]).float()
    return bool((ends == float(_poison(dtype))).all())


@pytest.mark.parametrize("case", [0, 1, 2])
def test_no_writes_outside_caller_buffers(case):
    # Ragged shapes (tile tails on both key ranges and on the query side), INT8
    # and BF16 caches, split and unsplit: poison guards around every buffer a
    # kernel writes must survive append, RoPE and attention.
    wl = small_variant(CONFIGS["c2_bf16_hist8"], **RAGGED[case], seed=300 + case)
    hist = [segment_kv(wl, s, f, 0) for s, f in enumerate(wl.cache_frames_hist)]
    slots = wl.capacity_frames * wl.tpf
    kdt = torch.int8 if wl.cache_dtype == "int8" else torch.bfloat16
    kb, kc, g = _guarded((1, wl.heads, slots, 128), kdt)
    vb, vc, _ = _guarded((1, wl.heads, slots, 128), kdt)
    gc = nomas.KVCache(1, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, wl.cache_dtype)
    gc.k, gc.v = kc, vc
    gc.desc.k, gc.desc.v = kc.data_ptr(), vc.data_ptr()
    if wl.cache_dtype == "int8":
        ksb, ksc, _ = _guarded((1, wl.heads, slots), torch.float32)
        vsb, vsc, _ = _guarded((1, wl.heads, slots), torch.float32)
        gc.k_scale, gc.v_scale = ksc, vsc
        gc.desc.k_scale, gc.desc.v_scale = ksc.data_ptr(), vsc.data_ptr()
    for k, v in hist:
        gc.append(to_dev(k, "bf16"), to_dev(v, "bf16"))
    q, k, v = current_qkv(wl)
    qb, qd, _ = _guarded(q.shape, torch.bfloat16)
    kcb, kd, _ = _guarded(k.shape, torch.bfloat16)
    qd.copy_(to_dev(q, "bf16"))
    kd.copy_(to_dev(k, "bf16"))
    vd = to_dev(v, "bf16")
    nomas.rope3d(qd, kd, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
    for splits in (1, 3):
        ob, od, _ = _guarded(q.shape, torch.bfloat16)
        lb, ld, _ = _guarded((wl.heads, wl.n_q), torch.float32)
        nbytes = gc.workspace_bytes(wl.n_video, wl.n_text, splits)
        wb, wd, _ = _guarded((max(nbytes, 256),), torch.uint8)
        nomas.segment_attn(gc, 0, qd, kd, vd, wl.n_video, wl.n_text, out=od, lse=ld, workspace=wd,
                           num_splits=splits)
        torch.cuda.synchronize()
        for big, dt in ((ob, torch.bfloat16), (lb, torch.float32), (wb, torch.uint8)):
            assert _guards_intact(big, g, dt)
    for big, dt in ((kb, kdt), (vb, kdt), (qb, torch.bfloat16), (kcb, torch.bfloat16)):
        assert _guards_intact(big, g, dt)
    if wl.cache_dtype == "int8":
        assert _guards_intact(ksb, g, torch.float32) and _guards_intact(vsb, g, torch.float32)
