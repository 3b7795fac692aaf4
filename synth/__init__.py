"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the benchmark."""
from .workloads import (CONFIGS, CONFIG_ORDER, Workload, current_qkv, current_qkv_torch, history_segments,
                        round_to_bf16, segment_kv, segment_kv_torch, small_variant)

__all__ = ["CONFIGS", "CONFIG_ORDER", "Workload", "current_qkv", "current_qkv_torch", "history_segments",
           "round_to_bf16", "segment_kv", "segment_kv_torch", "small_variant"]
