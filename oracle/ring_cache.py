"""Persistent, optionally windowed KV cache of latent frames (oracle; test infrastructure only).

What the pages fix:

* each segment is conditioned on a lifelong cache of the earlier latents' keys
  and values (Hy-Nomas: Was Tencent ... tatsaechlich macht, section "Die
  Schleife");
* the single-GPU preset keeps a sliding window of ``past_frames: 18`` latent
  frames on the GPU and moves older frames out (Hy-Nomas auf einer RTX 4090,
  sections "Das Single-GPU-Preset" and "System-RAM": ``total_frames``
  30/60/90 with 18 latent frames kept on the GPU);
* a new session starts from an empty cache, and the service keeps the cache
  between calls (same page, section "Setup": ``preserve_kv_cache=True``).

Reading used here (the plainest the rest supports):

* the cache holds video tokens only, one row of ``head_dim`` values per
  (block, head, token);
* ``W = past_frames`` if a window is set, else the capacity; a windowed cache
  has ``capacity_frames == past_frames``;
* absolute latent frame ``f`` lives in ring frame-slot ``f mod capacity``, its
  token ``(h, w)`` at slot ``(f mod capacity) * tpf + h * grid_w + w``;
* appending frames ``[T, T + F)`` leaves frames ``[max(0, T + F - W), T + F)``
  resident; frames of the new segment older than that are never written;
  ``valid_frames = min(T + F, W)``, so the resident slots are exactly
  ``[0, valid_frames * tpf)`` (the ring fills from slot 0);
* without a window, appending past the capacity is an error.

INT8 caches store codes and per-row scales from :mod:`oracle.int8_codec`, FP8
caches (the comparison format) E4M3 codes and scales from
:mod:`oracle.fp8_codec`; BF16
caches store the values rounded to bf16 (round to nearest even).
"""
from __future__ import annotations

import numpy as np

from . import fp8_codec, int8_codec
from .rope3d import rope3d_segment


class CapacityError(RuntimeError):
    """Appending would exceed the capacity of a cache without a window."""


def _bf16_round(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


class RingCache:
    """Model of the KV cache of ``blocks`` transformer blocks."""

    def __init__(self, blocks: int, heads: int, head_dim: int, grid_h: int, grid_w: int,
                 capacity_frames: int, past_frames: int, dtype: str, store: bool = True):
        if blocks <= 0 or heads <= 0 or head_dim <= 0 or grid_h <= 0 or grid_w <= 0:
            raise ValueError("shape arguments must be positive")
        if capacity_frames <= 0 or past_frames < 0:
            raise ValueError("bad capacity / window")
        if past_frames > 0 and capacity_frames != past_frames:
            raise ValueError("a windowed cache must have capacity_frames == past_frames")
        if dtype not in ("int8", "fp8", "bf16"):
            raise ValueError("dtype must be 'int8', 'fp8' or 'bf16'")
        self.blocks, self.heads, self.head_dim = blocks, heads, head_dim
        self.grid_h, self.grid_w = grid_h, grid_w
        self.tpf = grid_h * grid_w
        self.capacity_frames, self.past_frames, self.dtype = capacity_frames, past_frames, dtype
        self.slots = capacity_frames * self.tpf
        self.total_frames = 0
        self.valid_frames = 0
        self.frame_of_slot = np.full(capacity_frames, -1, dtype=np.int64)
        self.store = store
        if store:
            shape = (blocks, heads, self.slots, head_dim)
            if dtype in ("int8", "fp8"):
                self.k_codes = np.zeros(shape, np.int8 if dtype == "int8" else np.uint8)
                self.v_codes = np.zeros(shape, np.int8 if dtype == "int8" else np.uint8)
                self.k_scales = np.zeros(shape[:3], np.float32)
                self.v_scales = np.zeros(shape[:3], np.float32)
            else:
                self.k_vals = np.zeros(shape, np.float64)
                self.v_vals = np.zeros(shape, np.float64)

    @property
    def window(self) -> int:
        return self.past_frames if self.past_frames > 0 else self.capacity_frames

    def plan_append(self, n_frames: int):
        """Frames an append of ``n_frames`` would write.

        Returns a list of ``(segment_frame, absolute_frame, ring_frame_slot)`` in
        increasing order.  Raises :class:`CapacityError` when a cache without a
        window would overflow.
        """
        if n_frames < 0:
            raise ValueError("n_frames must be >= 0")
        t, w = self.total_frames, self.window
        if self.past_frames == 0 and t + n_frames > self.capacity_frames:
            raise CapacityError("append exceeds capacity of a cache without a window")
        first = max(0, n_frames - w)
        return [(fs, t + fs, (t + fs) % self.capacity_frames) for fs in range(first, n_frames)]

    def append(self, k=None, v=None, n_frames: int = None):
        """Append a finished segment's K/V (``[blocks][F * tpf][heads][D]``).

        With ``store=False`` only ``n_frames`` is needed and only the metadata
        advances.  Returns the plan of :meth:`plan_append`.
        """
        if k is not None:
            k = np.asarray(k)
            v = np.asarray(v)
            if k.ndim == 3:
                k, v = k[None], v[None]
            if k.shape[0] != self.blocks or k.shape[2:] != (self.heads, self.head_dim):
                raise ValueError("K/V shape does not match the cache")
            if k.shape[1] % self.tpf:
                raise ValueError("token count is not a whole number of frames")
            n_frames = k.shape[1] // self.tpf
        plan = self.plan_append(n_frames)
        for fs, fa, sf in plan:
            if self.store and k is not None:
                rows = slice(fs * self.tpf, (fs + 1) * self.tpf)
                dst = slice(sf * self.tpf, (sf + 1) * self.tpf)
                kk = np.transpose(k[:, rows], (0, 2, 1, 3))        # [blocks][heads][tpf][D]
                vv = np.transpose(v[:, rows], (0, 2, 1, 3))
                if self.dtype in ("int8", "fp8"):
                    codec = int8_codec if self.dtype == "int8" else fp8_codec
                    self.k_codes[:, :, dst], self.k_scales[:, :, dst] = codec.quantize_rows(kk)
                    self.v_codes[:, :, dst], self.v_scales[:, :, dst] = codec.quantize_rows(vv)
                else:
                    self.k_vals[:, :, dst] = _bf16_round(kk)
                    self.v_vals[:, :, dst] = _bf16_round(vv)
            self.frame_of_slot[sf] = fa
        self.total_frames += n_frames
        self.valid_frames = min(self.total_frames, self.window)
        return plan

    def append_rope(self, k, v, theta: float = 10000.0, split=(32, 48, 48)):
        """Append a finished segment whose keys still lack their 3D RoPE.

        After a segment is generated its keys and values are written to the
        cache (the KV-write stage, Hy-Nomas auf einer RTX 4090, section
        "Zeiten"), and later segments see them at their own positions, which
        continue from the cached frames.  Reading: frame ``f`` of the segment is
        rotated at ``(total_frames + f, h, w)`` (as :func:`rope3d_segment` with
        ``t0 = total_frames``) in float64, rounded once to float32 (the
        precision in which a stored row is quantised or rounded to bf16), and
        then appended as by :meth:`append`; V is appended unchanged.  Frames
        the window drops at once keep their absolute positions: only the
        resident ones are written.
        """
        k = np.asarray(k, dtype=np.float64)
        if k.ndim == 3:
            k = k[None]
        if k.shape[1] % self.tpf:
            raise ValueError("token count is not a whole number of frames")
        frames = k.shape[1] // self.tpf
        rot = np.stack([rope3d_segment(k[b], frames, self.grid_h, self.grid_w, self.total_frames, theta, split)
                        for b in range(k.shape[0])])
        v = np.asarray(v)
        return self.append(rot.astype(np.float32), v[None] if v.ndim == 3 else v)

    def resident_frames(self):
        """Absolute latent frames resident on the device, oldest first."""
        lo = max(0, self.total_frames - self.window)
        return list(range(lo, self.total_frames))

    def n_resident_tokens(self) -> int:
        return self.valid_frames * self.tpf

    def cache_kv(self, block: int):
        """Dequantised K and V of the resident slots ``[0, valid_frames * tpf)``.

        Returns float64 ``[n_resident_tokens][heads][D]`` each, in slot order.
        """
        n = self.n_resident_tokens()
        if self.dtype in ("int8", "fp8"):
            codec = int8_codec if self.dtype == "int8" else fp8_codec
            k = codec.dequantize_rows(self.k_codes[block, :, :n], self.k_scales[block, :, :n])
            v = codec.dequantize_rows(self.v_codes[block, :, :n], self.v_scales[block, :, :n])
        else:
            k = self.k_vals[block, :, :n]
            v = self.v_vals[block, :, :n]
        return np.transpose(k, (1, 0, 2)), np.transpose(v, (1, 0, 2))

    def reset(self, zero_memory: bool = False):
        """Start a new session: metadata to zero, storage optionally cleared."""
        self.total_frames = 0
        self.valid_frames = 0
        self.frame_of_slot[:] = -1
        if zero_memory and self.store:
            for name in ("k_codes", "v_codes", "k_scales", "v_scales", "k_vals", "v_vals"):
                if hasattr(self, name):
                    getattr(self, name)[...] = 0

    def bytes(self) -> int:
        """Device bytes of the cache storage (K and V, codes or bf16, plus scales)."""
        per = self.blocks * self.heads * self.slots
        if self.dtype in ("int8", "fp8"):
            return 2 * per * (self.head_dim + 4)
        return 2 * per * self.head_dim * 2
