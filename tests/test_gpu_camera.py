"""GPU parity of the camera cross-attention against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import segment_causal_kv_int8_b300 as nomas
    from _gpu_common import ATTN_MAX_ABS, ATTN_MEAN_ABS, f64
    from oracle.camera import camera_cross_attention
    from synth import round_to_bf16


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()
    assert nomas.device_error(clear=True) == 0


def _inputs(frames, gh, gw, heads, n_cam, n_text, seed):
    rng = np.random.default_rng(seed)
    nv = frames * gh * gw
    q = round_to_bf16(rng.standard_normal((nv + n_text, heads, 128)).astype(np.float32))
    k = round_to_bf16(rng.standard_normal((frames, n_cam, heads, 128)).astype(np.float32))
    v = round_to_bf16(rng.standard_normal((frames, n_cam, heads, 128)).astype(np.float32))
    return q, k, v


def _dev(x):
    return torch.from_numpy(x).to(torch.bfloat16).cuda()


CASES = [
    # frames, grid_h, grid_w, heads, n_cam, text rows after the video rows
    (8, 23, 40, 16, 4, 256),     # the segment shape of the pages' preset
    (3, 5, 7, 6, 1, 9),          # ragged token and head groups, one camera token
    (2, 4, 6, 3, 16, 0),         # the largest camera group
    (1, 3, 3, 1, 7, 2),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_camera_cross_attention_matches_oracle(case):
    frames, gh, gw, heads, n_cam, n_text = CASES[case]
    q, k, v = _inputs(frames, gh, gw, heads, n_cam, n_text, 40 + case)
    out = nomas.camera_cross_attn(_dev(q), _dev(k), _dev(v), frames, gh, gw)
    ref = camera_cross_attention(q, k, v, frames, gh * gw, 1.0 / np.sqrt(128))
    err = np.abs(f64(out) - ref)
    assert np.isfinite(f64(out)).all()
    assert err.max() <= ATTN_MAX_ABS and err.mean() <= ATTN_MEAN_ABS, (err.max(), err.mean())
    if n_cam == 1:
        # a single camera token: the output is its value, bit for bit
        want = np.repeat(v[:, 0], gh * gw, axis=0)
        np.testing.assert_array_equal(f64(out), want.astype(np.float64))


def test_writes_only_the_video_rows():
    frames, gh, gw, heads, n_cam = 2, 4, 5, 2, 3
    q, k, v = _inputs(frames, gh, gw, heads, n_cam, 0, 77)
    out = torch.full((frames * gh * gw + 8, heads, 128), -7.0, dtype=torch.bfloat16, device="cuda")
    nomas.camera_cross_attn(_dev(q), _dev(k), _dev(v), frames, gh, gw, out=out[:frames * gh * gw])
    assert torch.all(out[frames * gh * gw:] == -7.0)
    with pytest.raises(nomas.NomasError):
        nomas.camera_cross_attn(_dev(q), _dev(np.zeros((frames, 17, heads, 128), np.float32)),
                                _dev(np.zeros((frames, 17, heads, 128), np.float32)), frames, gh, gw)
