"""The per-unit work bench.py divides by: algorithmic bytes of the HBM-bound
kernels and FLOPs of the attention, on the benchmark workloads.

Each expected value is written out from the workload's shape by hand (tokens,
heads, bytes per row), independent of the formulas in bench.py, so a dropped
factor there (a tensor, a read or write, the scale bytes) fails here.
"""
import bench
from synth import CONFIGS

MB = 1e6


def test_rope_bytes():
    # Q and K video rows, 16 heads x 128 bf16 values = 256 B each, read and written
    assert bench.rope_bytes(CONFIGS["c4_bf16_hist60"]) == 7360 * 16 * 256 * 2 * 2  # 120.6 MB
    assert bench.rope_bytes(CONFIGS["c3_int8_window18"]) == 7360 * 16 * 256 * 2 * 2
    assert bench.rope_bytes(CONFIGS["c2_bf16_hist8"]) == 3680 * 16 * 256 * 2 * 2  # 60.3 MB


def test_append_bytes():
    # INT8 row pair: K and V bf16 rows read (2 x 256 B), codes written (2 x 128 B)
    # and their float32 scales (2 x 4 B): 776 B.  Three 8-frame segments of 920 tokens.
    assert bench.append_bytes(CONFIGS["c3_int8_window18"]) == 3 * 8 * 920 * 16 * 776
    # BF16 row pair: 2 x 256 B read, 2 x 256 B written; 60 frames
    assert bench.append_bytes(CONFIGS["c4_bf16_hist60"]) == 60 * 920 * 16 * 1024  # 904.4 MB
    assert abs(bench.append_bytes(CONFIGS["c4_bf16_hist60"]) / MB - 904.4) < 0.05


def test_expand_bytes():
    # resident INT8 window of 18 frames: per row of K and V, 128 code bytes and a
    # 4-byte scale read, 256 bf16 bytes written
    assert bench.expand_bytes(CONFIGS["c3_int8_window18"]) == 2 * 18 * 920 * 16 * (128 + 4 + 256)
    assert abs(bench.expand_bytes(CONFIGS["c3_int8_window18"]) / MB - 205.6) < 0.05


def test_attention_flops():
    # 4 * Nq * Nk * head_dim * heads: QK^T and PV, two FLOPs per multiply-add
    c4 = CONFIGS["c4_bf16_hist60"]
    assert c4.n_q == 7360 + 256 and c4.n_q + 55200 == 62816
    assert c4.attn_flops() == 4.0 * 7616 * 62816 * 128 * 16
    c2 = CONFIGS["c2_bf16_hist8"]
    assert c2.attn_flops() == 4.0 * 3936 * 11296 * 128 * 16
    c3 = CONFIGS["c3_int8_window18"]
    # the window keeps 18 of the 24 appended frames
    assert c3.attn_flops() == 4.0 * 7616 * (7616 + 18 * 920) * 128 * 16


def test_hbm_entry_fractions():
    e = bench.hbm_entry(120586240, 20.0, 6506.9, 1)
    assert abs(e["achieved"] - 120586240 / 20e-6 / 1e9) < 1e-6
    assert abs(e["frac"] - e["achieved"] / 6506.9) < 1e-12
    assert abs(e["frac_of_8tbs"] - e["achieved"] / 8000.0) < 1e-12
