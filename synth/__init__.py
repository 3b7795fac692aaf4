"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the benchmark."""
from .workloads import (CONFIGS, CONFIG_ORDER, Workload, current_qkv, history_segments,
                        round_to_bf16, segment_kv, small_variant)

__all__ = ["CONFIGS", "CONFIG_ORDER", "Workload", "current_qkv", "history_segments",
           "round_to_bf16", "segment_kv", "small_variant"]
