"""Seeded synthetic workloads for the segment-causal KV-cache attention path.

This module is shared by the CPU oracle and the CUDA path's tests and benchmark.
It holds only shapes and random draws: no part of the method's arithmetic (no
rotary embedding, no quantisation, no cache indexing, no attention) lives here.

Shapes follow the model the pages describe: 16 heads x 128 dims (hidden 2048),
latent frames of ``grid_h x grid_w`` tokens (720x1280 video through a 32x
spatial / 4x temporal latent codec gives a 23x40 grid), 8 latent frames per
segment plus 256 text tokens (Hy-Nomas auf einer RTX 4090, "Modell und Dateien"
and "Das Single-GPU-Preset"; Hy-Nomas: Was Tencent ... tatsaechlich macht,
"Die Schleife").

Every draw uses ``numpy.random.Generator(PCG64(...))`` seeded from a fixed
integer tuple, so the CPU oracle and the GPU tests see identical values.
Values destined for bf16 tensors are rounded to bf16-representable float32 here
(round-to-nearest-even on the bit pattern), so both sides consume the same
numbers exactly.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic configuration of the hot path.

    ``cache_frames_hist`` lists the latent-frame counts of the segments that were
    appended to the cache before the measured segment (in order); the measured
    segment starts at absolute latent frame ``t0 = sum(cache_frames_hist)``.
    ``past_frames`` is the sliding window in latent frames (0 = no window).
    """

    name: str
    heads: int
    head_dim: int
    grid_h: int
    grid_w: int
    cur_frames: int
    n_text: int
    cache_frames_hist: Tuple[int, ...]
    cache_dtype: str          # "int8" or "bf16"
    past_frames: int          # 0 = no window
    capacity_frames: int
    io_dtype: str             # "f32" or "bf16"
    seed: int
    blocks: int = 1
    outlier_p: float = 0.0    # probability an element of K/V is replaced by +-outlier_mag
    outlier_mag: float = 8.0
    theta: float = 10000.0
    rope_split: Tuple[int, int, int] = (32, 48, 48)
    turns: int = 1
    steps: int = 1

    @property
    def tpf(self) -> int:
        return self.grid_h * self.grid_w

    @property
    def n_video(self) -> int:
        return self.cur_frames * self.tpf

    @property
    def n_q(self) -> int:
        return self.n_video + self.n_text

    @property
    def t0(self) -> int:
        return int(sum(self.cache_frames_hist))

    @property
    def window(self) -> int:
        return self.past_frames if self.past_frames > 0 else self.capacity_frames

    @property
    def resident_frames(self) -> int:
        return min(self.t0, self.window)

    @property
    def n_cache(self) -> int:
        return self.resident_frames * self.tpf

    @property
    def n_k(self) -> int:
        return self.n_cache + self.n_q

    def attn_flops(self) -> float:
        """4 * Nq * Nk * D * H: two GEMMs (QK^T and PV) of 2 flops per MAC."""
        return 4.0 * self.n_q * self.n_k * self.head_dim * self.heads


# The five configurations of the hot path (tiny correctness case, single block
# with a BF16 history, the low-memory INT8 window, the full BF16 history, and
# a 12-turn session).  Config 3's history is three appended 8-frame segments,
# so the 18-frame window has wrapped around the ring when the segment runs.
CONFIGS = {
    "c1_tiny": Workload(
        name="c1_tiny", heads=2, head_dim=128, grid_h=4, grid_w=6, cur_frames=1,
        n_text=16, cache_frames_hist=(2,), cache_dtype="int8", past_frames=0,
        capacity_frames=3, io_dtype="f32", seed=1),
    "c2_bf16_hist8": Workload(
        name="c2_bf16_hist8", heads=16, head_dim=128, grid_h=23, grid_w=40,
        cur_frames=4, n_text=256, cache_frames_hist=(8,), cache_dtype="bf16",
        past_frames=0, capacity_frames=12, io_dtype="bf16", seed=2),
    "c3_int8_window18": Workload(
        name="c3_int8_window18", heads=16, head_dim=128, grid_h=23, grid_w=40,
        cur_frames=8, n_text=256, cache_frames_hist=(8, 8, 8),
        cache_dtype="int8", past_frames=18, capacity_frames=18, io_dtype="bf16",
        seed=3, outlier_p=0.01, outlier_mag=8.0),
    "c4_bf16_hist60": Workload(
        name="c4_bf16_hist60", heads=16, head_dim=128, grid_h=23, grid_w=40,
        cur_frames=8, n_text=256, cache_frames_hist=(60,), cache_dtype="bf16",
        past_frames=0, capacity_frames=68, io_dtype="bf16", seed=4),
    "c5_session12": Workload(
        name="c5_session12", heads=16, head_dim=128, grid_h=23, grid_w=40,
        cur_frames=8, n_text=256, cache_frames_hist=(), cache_dtype="int8",
        past_frames=18, capacity_frames=18, io_dtype="bf16", seed=5, blocks=54,
        turns=12, steps=8),
}

CONFIG_ORDER = ["c1_tiny", "c2_bf16_hist8", "c3_int8_window18", "c4_bf16_hist60", "c5_session12"]


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even), kept as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def _normal(rng: np.random.Generator, shape, outlier_p: float, outlier_mag: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if outlier_p > 0.0:
        hit = rng.random(size=shape, dtype=np.float32) < outlier_p
        sign = np.where(rng.random(size=shape, dtype=np.float32) < 0.5, -1.0, 1.0).astype(np.float32)
        x = np.where(hit, sign * np.float32(outlier_mag), x).astype(np.float32)
    return x


def _finish(wl: Workload, x: np.ndarray) -> np.ndarray:
    return round_to_bf16(x) if wl.io_dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


# Stream tags keep the draws of different tensors independent.
_TAG_Q, _TAG_K, _TAG_V, _TAG_HK, _TAG_HV = 11, 12, 13, 21, 22


def current_qkv(wl: Workload, turn: int = 0, step: int = 0, block: int = 0,
                rows: Optional[int] = None):
    """Q, K, V of the current segment, each float32 ``[n_q][heads][head_dim]``.

    Rows ``[0, n_video)`` are video tokens in (frame, h, w) row-major order and
    rows ``[n_video, n_q)`` are text tokens.  Q is N(0,1); K and V are N(0,1)
    with the workload's outlier mix.
    """
    n = wl.n_q if rows is None else rows
    shape = (n, wl.heads, wl.head_dim)
    q = _normal(_rng(wl.seed, _TAG_Q, turn, step, block), shape, 0.0, 0.0)
    k = _normal(_rng(wl.seed, _TAG_K, turn, step, block), shape, wl.outlier_p, wl.outlier_mag)
    v = _normal(_rng(wl.seed, _TAG_V, turn, step, block), shape, wl.outlier_p, wl.outlier_mag)
    return _finish(wl, q), _finish(wl, k), _finish(wl, v)


def segment_kv(wl: Workload, segment: int, frames: int, block: int):
    """K and V of a finished segment of ``frames`` latent frames for one block.

    Float32 ``[frames * tpf][heads][head_dim]``, video tokens only, standing for
    the keys and values that the KV-write pass produces for the segment's final
    latents (already position-encoded).
    """
    shape = (frames * wl.tpf, wl.heads, wl.head_dim)
    k = _normal(_rng(wl.seed, _TAG_HK, segment, block), shape, wl.outlier_p, wl.outlier_mag)
    v = _normal(_rng(wl.seed, _TAG_HV, segment, block), shape, wl.outlier_p, wl.outlier_mag)
    return _finish(wl, k), _finish(wl, v)


def history_segments(wl: Workload, block: int = 0) -> List[Tuple[np.ndarray, np.ndarray]]:
    """The segments appended before the measured one, oldest first, for one block."""
    return [segment_kv(wl, s, f, block) for s, f in enumerate(wl.cache_frames_hist)]


def small_variant(wl: Workload, **changes) -> Workload:
    """A copy of ``wl`` with some fields replaced (used for ragged / edge shapes)."""
    return dataclasses.replace(wl, **changes)


# ---------------------------------------------------------------- device-side draws
# The session workload (54 blocks x 12 turns x 8 steps) is too large to draw
# on the host for every call.  These draws use torch's counter-based
# generator on the given device, seeded from the same integer tuples; they are
# a different stream of numbers from the NumPy draws above, but serve the CUDA
# path and the oracle alike (the oracle receives copies of them).
def _torch_seed(*key: int) -> int:
    ss = np.random.SeedSequence([int(k) for k in key])
    return int(ss.generate_state(1, dtype=np.uint64)[0] & 0x7FFFFFFFFFFFFFFF)


def _torch_normal(shape, seed: int, device, outlier_p: float, outlier_mag: float):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if outlier_p > 0.0:
        hit = torch.rand(shape, generator=g, device=device) < outlier_p
        sign = torch.where(torch.rand(shape, generator=g, device=device) < 0.5, -1.0, 1.0)
        x = torch.where(hit, sign * outlier_mag, x)
    return x.to(torch.bfloat16)


def current_qkv_torch(wl: Workload, turn: int, step: int, block: int, device):
    """Q, K, V of the current segment as bf16 tensors on ``device``, ``[n_q][heads][head_dim]``."""
    shape = (wl.n_q, wl.heads, wl.head_dim)
    return tuple(_torch_normal(shape, _torch_seed(wl.seed, tag, turn, step, block), device,
                               0.0 if tag == _TAG_Q else wl.outlier_p, wl.outlier_mag)
                 for tag in (_TAG_Q, _TAG_K, _TAG_V))


def segment_kv_torch(wl: Workload, segment: int, frames: int, blocks: int, device):
    """K and V of a finished segment for ``blocks`` blocks, bf16 ``[blocks][frames*tpf][heads][head_dim]``."""
    shape = (blocks, frames * wl.tpf, wl.heads, wl.head_dim)
    return tuple(_torch_normal(shape, _torch_seed(wl.seed, tag, segment, blocks), device, wl.outlier_p,
                               wl.outlier_mag) for tag in (_TAG_HK, _TAG_HV))
