"""Python binding of the segment-causal KV-cache attention library (``libnomas.so``).

Argument marshalling only: every step of the hot path runs in the CUDA kernels
behind the C ABI declared in ``include/nomas.h``.  PyTorch supplies device
memory and streams.  The functions ``nomas_*`` mirror the C entry points one to
one (ctypes); :class:`KVCache`, :func:`rope3d`, :func:`segment_attn` are thin
conveniences over them that take torch tensors and raise :class:`NomasError`
on any status other than ``NOMAS_OK``.

There is no CPU fallback: importing this package loads the shared library and
fails loudly when it has not been built (``python
segment_causal_kv_int8_b300/_build.py``).  With ``NOMAS_LIBRARY=checked`` in the
environment it loads ``libnomas_checked.so`` instead: the same kernels with every
computed global-memory index range-checked (a bad index is recorded in the
device error word as NOMAS_ERR_INVALID_ARG and its access skipped).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
_VARIANT = os.environ.get("NOMAS_LIBRARY", "")
if _VARIANT not in ("", "checked"):
    raise ImportError(f"NOMAS_LIBRARY={_VARIANT!r}: expected unset or 'checked'")
LIB_PATH = os.path.join(_PKG, "libnomas_checked.so" if _VARIANT == "checked" else "libnomas.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python segment_causal_kv_int8_b300/_build.py` "
        "(there is no fallback implementation)")

_lib = ctypes.CDLL(LIB_PATH)

# ---------------------------------------------------------------- enums
NOMAS_OK = 0
NOMAS_ERR_INVALID_ARG = 1
NOMAS_ERR_UNSUPPORTED = 2
NOMAS_ERR_CAPACITY = 3
NOMAS_ERR_CUDA = 4
NOMAS_ERR_DEVICE_TIMEOUT = 5

NOMAS_F32 = 0
NOMAS_BF16 = 1
NOMAS_INT8 = 2
NOMAS_FP8 = 3


class nomas_kvcache(ctypes.Structure):
    """Mirror of the C ``nomas_kvcache`` descriptor."""

    _fields_ = [
        ("num_blocks", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("grid_h", ctypes.c_int32),
        ("grid_w", ctypes.c_int32),
        ("capacity_frames", ctypes.c_int32),
        ("past_frames", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("total_frames", ctypes.c_int64),
        ("valid_frames", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class nomas_attn_plan(ctypes.Structure):
    """Mirror of the C ``nomas_attn_plan`` (how nomas_segment_attn divides its work)."""

    _fields_ = [
        ("units", ctypes.c_int32),
        ("whole_units", ctypes.c_int32),
        ("pieces_per_split_unit", ctypes.c_int32),
        ("ctas_per_unit", ctypes.c_int32),
        ("work_items", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_size_t),
    ]


_P = ctypes.POINTER
_c_int, _i32, _i64, _f32, _vp, _sz = (ctypes.c_int, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                      ctypes.c_void_p, ctypes.c_size_t)

# name -> (restype, argtypes); the declarations of include/nomas.h
EXPORTS = {
    "nomas_version": (_i32, []),
    "nomas_status_string": (ctypes.c_char_p, [_c_int]),
    "nomas_kvcache_validate": (_c_int, [_P(nomas_kvcache)]),
    "nomas_kvcache_bytes": (_sz, [_P(nomas_kvcache)]),
    "nomas_kvcache_plan_append": (_c_int, [_P(nomas_kvcache), _i32, _P(_i32), _P(_i32), _P(_i64), _P(_i32)]),
    "nomas_rope3d_apply": (_c_int, [_vp, _vp, _c_int, _i32, _i32, _i32, _i64, _i32, _i32, _i32, _i64, _f32,
                                    _i32, _i32, _i32, _vp]),
    "nomas_kvcache_append": (_c_int, [_P(nomas_kvcache), _vp, _vp, _c_int, _i32, _i64, _vp]),
    "nomas_kvcache_append_rope": (_c_int, [_P(nomas_kvcache), _vp, _vp, _c_int, _i32, _i64, _f32, _i32, _i32, _i32,
                                           _vp]),
    "nomas_kvcache_archive_frame_bytes": (_sz, [_P(nomas_kvcache)]),
    "nomas_kvcache_append_archive": (_c_int, [_P(nomas_kvcache), _vp, _vp, _c_int, _i32, _i64, _vp, _sz, _P(_sz),
                                              _vp]),
    "nomas_segment_attn_workspace_bytes": (_c_int, [_P(nomas_kvcache), _i32, _i32, _i32, _P(_sz)]),
    "nomas_segment_attn_plan": (_c_int, [_P(nomas_kvcache), _i32, _i32, _i32, _P(nomas_attn_plan)]),
    "nomas_segment_attn": (_c_int, [_P(nomas_kvcache), _i32, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _vp, _vp,
                                    _sz, _i32, _vp]),
    "nomas_segment_attn_planned": (_c_int, [_P(nomas_kvcache), _i32, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _vp,
                                            _vp, _sz, _P(nomas_attn_plan), _vp]),
    "nomas_segment_attn_noalloc": (_c_int, [_P(nomas_kvcache), _i32, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _vp,
                                            _i32, _vp]),
    "nomas_sparse_select_workspace_bytes": (_c_int, [_P(nomas_kvcache), _i32, _i32, _P(_sz)]),
    "nomas_sparse_select": (_c_int, [_P(nomas_kvcache), _i32, _vp, _i32, _i32, _f32, _vp, _vp, _i32, _i32, _vp,
                                     _sz, _vp]),
    "nomas_segment_attn_sparse": (_c_int, [_P(nomas_kvcache), _i32, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _vp,
                                           _i32, _vp, _vp, _vp, _sz, _i32, _vp]),
    "nomas_camera_cross_attn": (_c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp]),
    "nomas_kvcache_reset": (_c_int, [_P(nomas_kvcache), _c_int, _vp]),
    "nomas_kvcache_expand": (_c_int, [_P(nomas_kvcache), _P(nomas_kvcache), _vp]),
    "nomas_selftest_wait_timeout": (_c_int, [ctypes.c_uint32, _vp]),
    "nomas_bounds_checked": (_i32, []),
    "nomas_selftest_bounds_check": (_c_int, [_vp]),
    "nomas_device_error": (_c_int, [_P(_c_int), _c_int]),
}

for _name, (_res, _args) in EXPORTS.items():
    try:
        _fn = getattr(_lib, _name)
    except AttributeError as _e:
        raise ImportError(f"{LIB_PATH} lacks {_name}: rebuild it with "
                          "`python segment_causal_kv_int8_b300/_build.py`") from _e
    _fn.restype = _res
    _fn.argtypes = _args
    globals()[_name] = _fn


class NomasError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {nomas_status_string(status).decode()}")


def _check(status: int, what: str) -> None:
    if status != NOMAS_OK:
        raise NomasError(status, what)


# ---------------------------------------------------------------- torch conveniences
def _torch():
    import torch
    return torch


def _stream_ptr(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dt_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return NOMAS_F32
    if t.dtype == torch.bfloat16:
        return NOMAS_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def rope3d(q, k, frames: int, grid_h: int, grid_w: int, t0: int, theta: float = 10000.0,
           split=(32, 48, 48), stream=None) -> None:
    """In-place 3D RoPE on the first ``frames * grid_h * grid_w`` rows of q (and k).

    ``q``/``k``: CUDA tensors ``[tokens][heads][128]`` (float32 or bfloat16),
    token rows contiguous; ``k`` may be None.
    """
    if not q.is_cuda or (k is not None and (not k.is_cuda or k.dtype != q.dtype or k.shape != q.shape)):
        raise ValueError("q and k must be CUDA tensors of the same dtype and shape")
    if q.dim() != 3 or q.stride(2) != 1 or q.stride(1) != q.shape[2] or (k is not None and k.stride() != q.stride()):
        raise ValueError("expected [tokens][heads][head_dim] with contiguous heads")
    n_video = frames * grid_h * grid_w
    _check(nomas_rope3d_apply(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr() if k is not None else 0),
                              _dt_code(q), n_video, q.shape[1], q.shape[2], q.stride(0), frames, grid_h, grid_w,
                              t0, theta, split[0], split[1], split[2], _stream_ptr(stream)), "nomas_rope3d_apply")


class KVCache:
    """A persistent ring KV cache whose device buffers are torch tensors.

    ``dtype``: "int8" (codes + float32 per-(block, head, token) scales), "fp8" (E4M3 codes
    as uint8 + scales; the comparison format) or "bf16".
    """

    def __init__(self, num_blocks: int, heads: int, grid_h: int, grid_w: int, capacity_frames: int,
                 past_frames: int = 0, dtype: str = "int8", device="cuda", head_dim: int = 128):
        torch = _torch()
        slots = capacity_frames * grid_h * grid_w
        shape = (num_blocks, heads, slots, head_dim)
        if dtype in ("int8", "fp8"):
            code_t = torch.int8 if dtype == "int8" else torch.uint8
            self.k = torch.zeros(shape, dtype=code_t, device=device)
            self.v = torch.zeros(shape, dtype=code_t, device=device)
            self.k_scale = torch.zeros(shape[:3], dtype=torch.float32, device=device)
            self.v_scale = torch.zeros(shape[:3], dtype=torch.float32, device=device)
            code = NOMAS_INT8 if dtype == "int8" else NOMAS_FP8
        elif dtype == "bf16":
            self.k = torch.zeros(shape, dtype=torch.bfloat16, device=device)
            self.v = torch.zeros(shape, dtype=torch.bfloat16, device=device)
            self.k_scale = self.v_scale = None
            code = NOMAS_BF16
        else:
            raise ValueError("dtype must be 'int8', 'fp8' or 'bf16'")
        self.dtype = dtype
        self.desc = nomas_kvcache(num_blocks, heads, head_dim, grid_h, grid_w, capacity_frames, past_frames, code,
                                  self.k.data_ptr(), self.v.data_ptr(),
                                  self.k_scale.data_ptr() if self.k_scale is not None else None,
                                  self.v_scale.data_ptr() if self.v_scale is not None else None, 0, 0, 0)
        _check(nomas_kvcache_validate(ctypes.byref(self.desc)), "nomas_kvcache_validate")

    @property
    def total_frames(self) -> int:
        return int(self.desc.total_frames)

    @property
    def valid_frames(self) -> int:
        return int(self.desc.valid_frames)

    @property
    def tpf(self) -> int:
        return self.desc.grid_h * self.desc.grid_w

    def nbytes(self) -> int:
        return int(nomas_kvcache_bytes(ctypes.byref(self.desc)))

    def expand_into(self, dst: "KVCache", stream=None) -> None:
        """Write this one-byte cache's resident window as BF16 values into ``dst`` (a "bf16"
        KVCache of the same geometry) and give ``dst`` this cache's frame counts."""
        _check(nomas_kvcache_expand(ctypes.byref(self.desc), ctypes.byref(dst.desc), _stream_ptr(stream)),
               "nomas_kvcache_expand")

    def append(self, k, v, stream=None) -> None:
        """Append a finished segment: ``k``, ``v`` ``[blocks][F*tpf][heads][128]`` (or 3-D for one block)."""
        k, v = self._check_segment(k, v)
        _check(nomas_kvcache_append(ctypes.byref(self.desc), ctypes.c_void_p(k.data_ptr()),
                                    ctypes.c_void_p(v.data_ptr()), _dt_code(k), k.shape[1] // self.tpf,
                                    k.stride(0), _stream_ptr(stream)), "nomas_kvcache_append")

    def append_rope(self, k, v, theta: float = 10000.0, split=(32, 48, 48), stream=None) -> None:
        """Append a segment whose keys are not yet position-encoded: K is rotated by 3D RoPE at
        (total_frames + f, h, w) on the way into the cache."""
        k, v = self._check_segment(k, v)
        _check(nomas_kvcache_append_rope(ctypes.byref(self.desc), ctypes.c_void_p(k.data_ptr()),
                                         ctypes.c_void_p(v.data_ptr()), _dt_code(k), k.shape[1] // self.tpf,
                                         k.stride(0), theta, split[0], split[1], split[2], _stream_ptr(stream)),
               "nomas_kvcache_append_rope")

    def _check_segment(self, k, v):
        if k.dim() == 3:
            k, v = k.unsqueeze(0), v.unsqueeze(0)
        if k.shape != v.shape or k.dtype != v.dtype or not k.is_cuda:
            raise ValueError("k and v must be CUDA tensors of equal shape and dtype")
        if k.shape[0] != self.desc.num_blocks or k.shape[2] != self.desc.heads or k.shape[3] != self.desc.head_dim:
            raise ValueError("K/V shape does not match the cache")
        if k.shape[1] % self.tpf:
            raise ValueError("token count is not a whole number of frames")
        for t in (k, v):
            if t.stride(3) != 1 or t.stride(2) != t.shape[3] or t.stride(1) != t.shape[2] * t.shape[3]:
                raise ValueError("K/V rows must be contiguous within a block")
        if k.stride() != v.stride():
            raise ValueError("k and v must share strides")
        return k, v

    def archive_frame_bytes(self) -> int:
        return int(nomas_kvcache_archive_frame_bytes(ctypes.byref(self.desc)))

    def append_archive(self, k, v, archive, used: int = 0, stream=None) -> int:
        """Append like :meth:`append` (INT8 or FP8 cache) and copy every frame of the segment to ``archive``
        (a host uint8 tensor, pinned for asynchronous copies) from byte ``used`` on; returns the new
        byte count.  Synchronise the stream before reading the archive."""
        if k.dim() == 3:
            k, v = k.unsqueeze(0), v.unsqueeze(0)
        if k.shape != v.shape or k.dtype != v.dtype or not k.is_cuda:
            raise ValueError("k and v must be CUDA tensors of equal shape and dtype")
        if k.shape[0] != self.desc.num_blocks or k.shape[2] != self.desc.heads or k.shape[1] % self.tpf:
            raise ValueError("K/V shape does not match the cache")
        if archive.is_cuda or archive.dtype.itemsize != 1 or not archive.is_contiguous():
            raise ValueError("archive must be a contiguous host byte tensor")
        n = ctypes.c_size_t(used)
        _check(nomas_kvcache_append_archive(ctypes.byref(self.desc), ctypes.c_void_p(k.data_ptr()),
                                            ctypes.c_void_p(v.data_ptr()), _dt_code(k), k.shape[1] // self.tpf,
                                            k.stride(0), ctypes.c_void_p(archive.data_ptr()), archive.numel(),
                                            ctypes.byref(n), _stream_ptr(stream)), "nomas_kvcache_append_archive")
        return int(n.value)

    def reset(self, zero_memory: bool = False, stream=None) -> None:
        _check(nomas_kvcache_reset(ctypes.byref(self.desc), int(bool(zero_memory)), _stream_ptr(stream)),
               "nomas_kvcache_reset")

    def attn_plan(self, n_video: int, n_text: int, num_splits: int = 0) -> dict:
        """The work plan nomas_segment_attn runs for these arguments (see ``nomas_segment_attn_plan``)."""
        pl = nomas_attn_plan()
        _check(nomas_segment_attn_plan(ctypes.byref(self.desc), n_video, n_text, num_splits, ctypes.byref(pl)),
               "nomas_segment_attn_plan")
        return {name: int(getattr(pl, name)) for name, _ in nomas_attn_plan._fields_ if name != "reserved"}

    def workspace_bytes(self, n_video: int, n_text: int, num_splits: int = 0) -> int:
        out = ctypes.c_size_t(0)
        _check(nomas_segment_attn_workspace_bytes(ctypes.byref(self.desc), n_video, n_text, num_splits,
                                                  ctypes.byref(out)), "nomas_segment_attn_workspace_bytes")
        return int(out.value)


def segment_attn(cache: KVCache, block: int, q, k_cur, v_cur, n_video: int, n_text: int,
                 softmax_scale: Optional[float] = None, out=None, lse=None, workspace=None,
                 num_splits: int = 0, stream=None):
    """Segment attention of one block; returns ``out`` (bf16 ``[Nq][heads][128]``).

    ``workspace``: optional CUDA uint8 tensor (see :meth:`KVCache.workspace_bytes`).
    """
    torch = _torch()
    for t in (q, k_cur, v_cur):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k_cur, v_cur must be contiguous bfloat16 CUDA tensors")
    nq = n_video + n_text
    if q.shape[0] != nq or q.shape != k_cur.shape or q.shape != v_cur.shape:
        raise ValueError("q/k_cur/v_cur must be [n_video + n_text][heads][128]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[2])
    if out is None:
        out = torch.empty_like(q)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(nomas_segment_attn(ctypes.byref(cache.desc), block, ctypes.c_void_p(q.data_ptr()),
                              ctypes.c_void_p(k_cur.data_ptr()), ctypes.c_void_p(v_cur.data_ptr()), n_video, n_text,
                              softmax_scale, ctypes.c_void_p(out.data_ptr()),
                              ctypes.c_void_p(lse.data_ptr() if lse is not None else 0), ctypes.c_void_p(ws_ptr),
                              ws_bytes, num_splits, _stream_ptr(stream)), "nomas_segment_attn")
    return out


def plan_workspace_bytes(units: int, whole_units: int, pieces: int, ctas_per_unit: int) -> int:
    """Scratch bytes of a work plan (float32 partial rows and log-sum-exps of every piece)."""
    rows = (units - whole_units) * pieces * ctas_per_unit * 256 if pieces > 1 and whole_units < units else 0
    return -(-rows * 512 // 256) * 256 + -(-rows * 4 // 256) * 256


def segment_attn_planned(cache: KVCache, block: int, q, k_cur, v_cur, n_video: int, n_text: int,
                         whole_units: int, pieces: int, softmax_scale: Optional[float] = None, out=None, lse=None,
                         workspace=None, stream=None):
    """Segment attention with a caller-chosen plan: the first ``whole_units`` units whole, the rest in
    ``pieces`` pieces each (see ``nomas_segment_attn_planned``); allocates the workspace when not given."""
    torch = _torch()
    base = cache.attn_plan(n_video, n_text, 1)
    pl = nomas_attn_plan(base["units"], whole_units, pieces, base["ctas_per_unit"], 0, 0, 0)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        need = plan_workspace_bytes(base["units"], whole_units, pieces, base["ctas_per_unit"])
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[2])
    _check(nomas_segment_attn_planned(ctypes.byref(cache.desc), block, ctypes.c_void_p(q.data_ptr()),
                                      ctypes.c_void_p(k_cur.data_ptr()), ctypes.c_void_p(v_cur.data_ptr()), n_video,
                                      n_text, softmax_scale, ctypes.c_void_p(out.data_ptr()),
                                      ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
                                      ctypes.c_void_p(workspace.data_ptr()),
                                      workspace.numel() * workspace.element_size(), ctypes.byref(pl),
                                      _stream_ptr(stream)), "nomas_segment_attn_planned")
    return out


def _check_lists(torch, tiles, counts, heads: int, groups: int) -> None:
    if tiles.dtype != torch.int32 or counts.dtype != torch.int32 or not tiles.is_contiguous() \
            or not counts.is_contiguous() or not tiles.is_cuda or not counts.is_cuda:
        raise ValueError("tiles and counts must be contiguous int32 CUDA tensors")
    if tiles.dim() != 3 or tuple(tiles.shape[:2]) != (heads, groups) or tiles.shape[2] < 1 \
            or tuple(counts.shape) != (heads, groups):
        raise ValueError(f"tiles must be [{heads}][{groups}][max_keep] and counts [{heads}][{groups}]")


def sparse_keep_count(n_tiles: int, keep_fraction: float) -> int:
    """Tiles kept per (head, query group) out of ``n_tiles`` resident cache tiles."""
    return min(n_tiles, max(0, math.ceil(keep_fraction * n_tiles - 1e-9)))


def sparse_select(cache: KVCache, block: int, q, n_video: int, n_text: int, keep_fraction: float = 0.25,
                  tiles=None, counts=None, workspace=None, reuse_key_means: bool = False, stream=None):
    """Kept cache tiles of block-sparse attention; returns ``(tiles, counts)``.

    ``tiles``: int32 ``[heads][groups][max_keep]`` (first ``counts[h, g]``
    entries of a row valid, increasing), ``counts``: int32 ``[heads][groups]``,
    groups = ceil((n_video + n_text) / 512).  Allocated when not given.
    ``reuse_key_means``: ``workspace`` still holds the mean keys of an earlier
    call on this block with the cache unchanged since.
    """
    torch = _torch()
    if not q.is_cuda or q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise ValueError("q must be a contiguous bfloat16 CUDA tensor")
    nq = n_video + n_text
    heads = cache.desc.heads
    groups = (nq + 511) // 512
    n_tiles = (cache.valid_frames * cache.tpf + 127) // 128
    if tiles is None:
        tiles = torch.zeros((heads, groups, max(1, sparse_keep_count(n_tiles, keep_fraction))),
                            dtype=torch.int32, device=q.device)
    if counts is None:
        counts = torch.zeros((heads, groups), dtype=torch.int32, device=q.device)
    _check_lists(torch, tiles, counts, heads, groups)
    need = ctypes.c_size_t(0)
    _check(nomas_sparse_select_workspace_bytes(ctypes.byref(cache.desc), n_video, n_text, ctypes.byref(need)),
           "nomas_sparse_select_workspace_bytes")
    if workspace is None:
        if reuse_key_means:
            raise ValueError("reuse_key_means needs the workspace of the earlier call")
        workspace = torch.empty(max(256, need.value), dtype=torch.uint8, device=q.device)
    _check(nomas_sparse_select(ctypes.byref(cache.desc), block, ctypes.c_void_p(q.data_ptr()), n_video, n_text,
                               keep_fraction, ctypes.c_void_p(tiles.data_ptr()), ctypes.c_void_p(counts.data_ptr()),
                               tiles.shape[-1], int(bool(reuse_key_means)), ctypes.c_void_p(workspace.data_ptr()),
                               workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "nomas_sparse_select")
    return tiles, counts


def segment_attn_sparse(cache: KVCache, block: int, q, k_cur, v_cur, n_video: int, n_text: int, tiles, counts,
                        softmax_scale: Optional[float] = None, out=None, lse=None, workspace=None,
                        num_splits: int = 0, stream=None):
    """Block-sparse segment attention over the kept tiles of :func:`sparse_select`; returns ``out``."""
    torch = _torch()
    for t in (q, k_cur, v_cur):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k_cur, v_cur must be contiguous bfloat16 CUDA tensors")
    nq = n_video + n_text
    if q.shape[0] != nq or q.shape != k_cur.shape or q.shape != v_cur.shape:
        raise ValueError("q/k_cur/v_cur must be [n_video + n_text][heads][128]")
    _check_lists(torch, tiles, counts, cache.desc.heads, (nq + 511) // 512)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[2])
    if out is None:
        out = torch.empty_like(q)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(nomas_segment_attn_sparse(ctypes.byref(cache.desc), block, ctypes.c_void_p(q.data_ptr()),
                                     ctypes.c_void_p(k_cur.data_ptr()), ctypes.c_void_p(v_cur.data_ptr()), n_video,
                                     n_text, softmax_scale, ctypes.c_void_p(tiles.data_ptr()),
                                     ctypes.c_void_p(counts.data_ptr()), tiles.shape[-1],
                                     ctypes.c_void_p(out.data_ptr()),
                                     ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
                                     ctypes.c_void_p(ws_ptr), ws_bytes, num_splits, _stream_ptr(stream)),
           "nomas_segment_attn_sparse")
    return out


def camera_cross_attn(q, k_cam, v_cam, frames: int, grid_h: int, grid_w: int, softmax_scale: Optional[float] = None,
                      out=None, stream=None):
    """Cross-attention of the video rows of ``q`` to their latent frame's camera tokens.

    ``q``: bf16 ``[>= frames*grid_h*grid_w][heads][128]`` (video rows first);
    ``k_cam``/``v_cam``: bf16 ``[frames][n_cam][heads][128]``.  Returns ``out``,
    bf16 ``[frames*grid_h*grid_w][heads][128]``.
    """
    torch = _torch()
    for t in (q, k_cam, v_cam):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k_cam, v_cam must be contiguous bfloat16 CUDA tensors")
    nv = frames * grid_h * grid_w
    heads = q.shape[1]
    if q.dim() != 3 or q.shape[0] < nv or q.shape[2] != 128:
        raise ValueError("q must be [tokens][heads][128] with at least frames*grid_h*grid_w rows")
    if k_cam.dim() != 4 or tuple(k_cam.shape[::2]) != (frames, heads) or k_cam.shape[3] != 128 \
            or k_cam.shape != v_cam.shape:
        raise ValueError("k_cam/v_cam must be [frames][n_cam][heads][128]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(128)
    if out is None:
        out = torch.empty((nv, heads, 128), dtype=torch.bfloat16, device=q.device)
    _check(nomas_camera_cross_attn(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_cam.data_ptr()),
                                   ctypes.c_void_p(v_cam.data_ptr()), frames, grid_h, grid_w, heads, k_cam.shape[1],
                                   softmax_scale, ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream)),
           "nomas_camera_cross_attn")
    return out


def device_error(clear: bool = True) -> int:
    """The device-side error word (0 = none), read synchronously."""
    st = ctypes.c_int(0)
    _check(nomas_device_error(ctypes.byref(st), int(bool(clear))), "nomas_device_error")
    return int(st.value)


__all__ = ["KVCache", "rope3d", "segment_attn", "segment_attn_planned", "plan_workspace_bytes", "sparse_select", "segment_attn_sparse", "sparse_keep_count",
           "camera_cross_attn",
           "device_error", "NomasError", "nomas_kvcache", "nomas_attn_plan", "EXPORTS",
           "LIB_PATH"] + list(EXPORTS)
