"""Pins of the oracle's FP8 (E4M3) row codec (CPU).

The E4M3 value table and the round-to-nearest-even conversion are checked
against PyTorch's own float8_e4m3fn type, an independent implementation;
saturation, NaN and the row rules against closed forms.
"""
import numpy as np
import torch

from oracle import fp8_codec as f


def test_value_table_matches_torch_float8():
    tv = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ov = f.decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(tv), np.isnan(ov)) and np.count_nonzero(np.isnan(ov)) == 2
    ok = ~np.isnan(ov)
    np.testing.assert_array_equal(tv[ok], ov[ok])
    assert ov[0x7E] == 448.0 and ov[0x01] == 2.0 ** -9 and ov[0x08] == 2.0 ** -6


def test_rounding_matches_torch_below_saturation_including_every_midpoint():
    rng = np.random.default_rng(0)
    vals = f.e4m3_values()
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    y = np.concatenate([rng.standard_normal(50000).astype(np.float32) * 60,
                        (rng.standard_normal(5000) * 2.0 ** -8).astype(np.float32),
                        mids, -mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                        np.float32([0.0, -0.0, 448.0, -448.0])])
    y = y[np.abs(y) <= 448]
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(f.round_e4m3(y), want)


def test_ties_go_to_the_even_code_and_saturation_and_nan():
    # 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39)
    assert f.round_e4m3(np.float32([1.0625]))[0] == 0x38
    # 7.5 * 2^-9: halfway between the largest subnormal (0x07) and 2^-6 (0x08)
    assert f.round_e4m3(np.float32([7.5 * 2.0 ** -9]))[0] == 0x08
    # half the smallest subnormal rounds to zero, keeping the sign
    assert list(f.round_e4m3(np.float32([0.5 * 2.0 ** -9, -0.5 * 2.0 ** -9]))) == [0x00, 0x80]
    assert list(f.round_e4m3(np.float32([470.0, -1e30, np.inf, np.nan]))) == [0x7E, 0xFE, 0x7E, 0x00]


def test_row_codec_rules():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 128)).astype(np.float32) * np.float32(3.0)
    codes, scales = f.quantize_rows(x)
    # the absmax element maps to +-448 exactly
    am = np.argmax(np.abs(x), axis=1)
    assert np.all(codes[np.arange(64), am] & 0x7F == 0x7E)
    np.testing.assert_array_equal(scales, (np.max(np.abs(x), axis=1) / np.float32(448)).astype(np.float32))
    # relative round-trip error: half a 3-bit mantissa step for normal codes
    xh = f.dequantize_rows(codes, scales)
    normal = np.abs(x) / scales[:, None] >= 2.0 ** -6
    rel = np.abs(xh - x)[normal] / np.abs(x)[normal]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)
    # zero row: scale 0 and codes 0; a row below 448 / FLT_MAX saturates
    z, zs = f.quantize_rows(np.zeros((1, 128), np.float32))
    assert zs[0] == 0 and not z.any()
    t = np.zeros((1, 128), np.float32)
    t[0, 3], t[0, 5] = 1e-45, -1e-45
    tc, _ = f.quantize_rows(t)
    assert tc[0, 3] == 0x7E and tc[0, 5] == 0xFE and tc[0, 0] == 0


def test_fp8_ring_cache_stores_the_codec_rows_in_their_slots():
    from oracle import ring_cache
    rng = np.random.default_rng(2)
    k = rng.standard_normal((1, 3 * 6, 2, 128)).astype(np.float32)
    v = rng.standard_normal((1, 3 * 6, 2, 128)).astype(np.float32)
    c = ring_cache.RingCache(1, 2, 128, 2, 3, 4, 0, "fp8")
    c.append(k, v)
    codes, scales = f.quantize_rows(np.transpose(k[0], (1, 0, 2)))
    np.testing.assert_array_equal(c.k_codes[0, :, :18], codes)
    np.testing.assert_array_equal(c.k_scales[0, :, :18].view(np.uint32), scales.view(np.uint32))
    kc, _ = c.cache_kv(0)
    # dequantised keys stay within half a mantissa step of the input (normal range)
    rel = np.abs(kc - k[0]) / np.maximum(np.abs(k[0]), 1e-30)
    big = np.abs(k[0]) >= np.max(np.abs(k[0]), axis=2, keepdims=True) * 2.0 ** -6 / 448 * 8
    assert rel[big].max() <= 2.0 ** -4 * (1 + 1e-6)
    assert c.bytes() == 2 * 2 * 24 * (128 + 4)
