#!/usr/bin/env python
"""Benchmark of the segment-causal KV-cache attention hot path.

One step = one pass of the whole path over one batch of synthetic input:
reset the cache (metadata), append the history segment(s) of K/V (INT8
quantise or BF16 copy into the ring), 3D RoPE of the current segment's Q and K,
segment attention of the current segment over [cache ; current].  The metric is
the attention's FLOPs (4 * Nq * Nk * 128 * heads) per step time, in TFLOP/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

The headline workload is the 60-frame BF16 history (``c4_bf16_hist60``, the
largest single-block call).  The same JSON line carries, under ``configs``, the
other single-block workloads (the INT8 window of 18 frames and the 8-frame
BF16 history) measured the same way, the INT8 window attended through its BF16
copy, block-sparse steps keeping a quarter of the cache tiles on the INT8
window and the 60-frame history, and one whole simulated 12-turn session
(8 denoising steps x 54 blocks per turn), each with attention TFLOP/s, its
fraction of the measured dense BF16 peak, query tokens per second per block
call, and the RoPE / append bandwidth against the measured HBM copy rate and
against 8 TB/s.

Under torchrun (N > 1) every rank runs the same-shaped workload on its own
seeded data (independent blocks; no collective on the data path) and rank 0
prints one JSON line with the whole-job throughput (weak scaling).

``--impl reference`` times the CPU oracle (the plain float64 reference the
tests check against) on a bounded sample of the same workload, on this host's
cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "segment-causal KV-cache attention TFLOP/s (% of B300 dense BF16 peak)"
UNIT = "TFLOP/s"
DEFAULT_CONFIG = "c4_bf16_hist60"
EXTRA_CONFIGS = ("c3_int8_window18", "c2_bf16_hist8")
SESSION_CONFIG = "c5_session12"
SPARSE_KEEP = 0.25  # kept fraction of cache tiles in the block-sparse entries
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
HBM_NOMINAL_GBS = 8000.0  # the "about 8 TB/s" HBM figure the RoPE / append targets are quoted against


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU work of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads and the session (only the --config workload)")
    ap.add_argument("--extra-seconds", type=float, default=0.5,
                    help="timed device time per extra single-block workload (at least --steps steps)")
    ap.add_argument("--turns", type=int, default=12, help="turns of the session workload (c5_session12)")
    ap.add_argument("--cache-dtype", choices=["int8", "fp8", "bf16"], default=None,
                    help="override the config's cache format (fp8: the E4M3 comparison variant)")
    ap.add_argument("--camera", type=int, default=0,
                    help="add the camera cross-attention with this many camera tokens per latent frame to the step")
    ap.add_argument("--bf16-shadow", action="store_true",
                    help="one-byte caches: expand the resident window to a BF16 copy after the appends "
                         "(nomas_kvcache_expand) and attend over the copy")
    ap.add_argument("--append-rope", action="store_true",
                    help="write the history with the fused RoPE + append (keys rotated on the way into the cache)")
    ap.add_argument("--sparse", type=float, default=0.0,
                    help="block-sparse attention keeping this fraction of cache tiles (0 = dense)")
    ap.add_argument("--archive", action="store_true",
                    help="session workload: also copy every appended frame to a host archive")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ------------------------------------------------------------------ multi-rank host logic
def rank_block(rank: int) -> int:
    """Seed block of a rank: every rank runs an independent block's workload (no data exchange)."""
    return rank


def max_over_ranks(x: float, world: int, device) -> float:
    """Maximum of a per-rank timing over all ranks (the job ends when the slowest rank does)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flops_per_step: float, world: int, steps: int, total_ms: float) -> float:
    """Whole-job TFLOP/s: the work of all ranks' timed steps over the slowest rank's time."""
    return flops_per_step * world * steps / (total_ms * 1e-3) / 1e12


def hbm_entry(nbytes: float, us: float, hbm_gbs: float, launches: int, **extra) -> dict:
    """Bandwidth summary of an HBM-bound kernel group: algorithmic bytes over its event time (inside
    the step unless ``timing`` says otherwise)."""
    gbs = nbytes / (us * 1e-6) / 1e9 if us > 0 else None
    d = {"bound": "hbm", "algorithmic_bytes": int(nbytes), "us": us, "achieved": gbs, "peak": hbm_gbs,
         "unit": "GB/s", "frac": gbs / hbm_gbs if gbs else None,
         "frac_of_8tbs": gbs / HBM_NOMINAL_GBS if gbs else None, "launches_per_step": launches}
    d.update(extra)
    return d


def append_bytes(wl) -> int:
    """Algorithmic bytes of the history appends of one step: per written (token, head) row pair, the
    K and V rows read plus the codes and scales (one-byte caches) or the bf16 rows written."""
    in_esz = 2 if wl.io_dtype == "bf16" else 4
    one_byte = wl.cache_dtype in ("int8", "fp8")
    row = 2 * (wl.head_dim * in_esz + (wl.head_dim + 4 if one_byte else 2 * wl.head_dim))
    return sum(min(f, wl.window) for f in wl.cache_frames_hist) * wl.tpf * wl.heads * row


def expand_bytes(wl) -> int:
    """Algorithmic bytes of the BF16 expansion of the resident window: per row of K and V, the codes
    and the scale read and the bf16 row written."""
    resident = min(sum(wl.cache_frames_hist), wl.window) * wl.tpf
    return 2 * resident * wl.heads * (wl.head_dim + 4 + 2 * wl.head_dim)


def rope_bytes(wl) -> int:
    """Algorithmic bytes of RoPE of one step: the video rows of Q and K, read and written."""
    in_esz = 2 if wl.io_dtype == "bf16" else 4
    return wl.n_video * wl.heads * wl.head_dim * in_esz * 2 * 2


# ------------------------------------------------------------------ CPU oracle timing
def oracle_setup(wl, block: int = 0):
    """The oracle's inputs for one block call of ``wl`` (cache built by the oracle's own append)."""
    from oracle import ring_cache as o_cache
    from synth import current_qkv, history_segments

    oc = o_cache.RingCache(1, wl.heads, wl.head_dim, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames,
                           wl.cache_dtype)
    for k, v in history_segments(wl, block):
        oc.append(k[None], v[None])
    q, k, v = current_qkv(wl, block=block)
    kc, vc = oc.cache_kv(0)
    return q, k, v, kc, vc


def oracle_sample(wl, seconds: float, block: int = 0, inputs=None, rows: int = 64):
    """Time the oracle's RoPE + segment attention on a sample of query rows.

    Returns (flops_per_second, description, threads, seconds, rows).  The
    sample grows from ``rows`` until it takes at least ``seconds`` (capped at
    the whole segment).  ``inputs``: a reused ``oracle_setup`` result.
    """
    import numpy as np

    from oracle import attention as o_attn
    from oracle import rope3d as o_rope

    q, k, v, kc, vc = inputs if inputs is not None else oracle_setup(wl, block)
    scale = o_attn.default_scale(wl.head_dim)
    while True:
        sel = np.linspace(0, wl.n_q - 1, rows).astype(np.int64)
        t0 = time.perf_counter()
        kr = o_rope.rope3d_segment(k, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
        qr = o_rope.rope3d_segment(q, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)[sel]
        o_attn.segment_attention(qr, kr, v, kc, vc, scale)
        dt = time.perf_counter() - t0
        if dt >= seconds or rows >= wl.n_q:
            break
        rows = min(wl.n_q, max(rows * 2, int(rows * seconds / max(dt, 1e-3) * 1.1)))
    flops = 4.0 * rows * wl.n_k * wl.head_dim * wl.heads
    threads = _blas_threads()
    desc = (f"oracle RoPE + segment attention (float64 numpy) on {rows} of {wl.n_q} query rows x all "
            f"{wl.heads} heads x {wl.n_k} keys of {wl.name}; {dt:.1f} s")
    return flops / dt, desc, threads, dt, rows


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from synth import CONFIGS

    wl = CONFIGS[args.config]
    per_step = max(2.0, min(args.cpu_seconds, 60.0 / max(1, args.steps + args.warmup)))
    inputs = oracle_setup(wl)  # built once; every step times RoPE + attention on a sample of rows
    rows = 64
    for _ in range(args.warmup):
        _, _, _, _, rows = oracle_sample(wl, per_step, inputs=inputs, rows=rows)
    vals, times = [], []
    for _ in range(args.steps):
        v, desc, threads, dt, rows = oracle_sample(wl, per_step, inputs=inputs, rows=rows)
        vals.append(v)
        times.append(dt)
    value = statistics.median(vals) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config_dict(wl, args.gpus, "oracle sample per step"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def _config_dict(wl, n_gpus, l2_policy):
    return {"workload": f"{wl.name}: {wl.heads} heads x {wl.head_dim}, grid {wl.grid_h}x{wl.grid_w}, "
                        f"{wl.cur_frames} latent frames + {wl.n_text} text queries (Nq={wl.n_q}), "
                        f"{wl.cache_dtype} cache of {wl.n_cache} tokens (window {wl.past_frames or 'none'}), "
                        f"Nk={wl.n_k}",
            "heads": wl.heads, "head_dim": wl.head_dim, "n_q": wl.n_q, "n_k": wl.n_k, "n_cache": wl.n_cache,
            "cache_dtype": wl.cache_dtype, "parallelism": f"replica x{n_gpus} (independent blocks per GPU)",
            "l2": l2_policy}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """SM clock, power, busy % and throttle reasons sampled in a background thread while a timed
    region runs: NVML every 10 ms (short regions still get samples), else nvidia-smi every 200 ms."""

    SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40), ("sw_thermal_slowdown", 0x20),
               ("sw_power_cap", 0x4), ("hw_power_brake_slowdown", 0x80))

    def __init__(self, device):
        self.device = device
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.samples = []   # (sm_mhz, max_mhz, busy_pct, reasons_mask)
        self.source = None
        self.nvml_error = None

    class _Nvml:
        """The few NVML calls the sampler needs, through ctypes on the driver's libnvidia-ml."""

        def __init__(self):
            import ctypes
            self.ct = ctypes
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit_v2 failed")

        def _ok(self, rc, what):
            if rc != 0:
                raise RuntimeError(f"{what} returned {rc}")

        def handle(self, device):
            ct = self.ct
            h = ct.c_void_p()
            errors = []
            try:
                import torch
                uuid = str(torch.cuda.get_device_properties(device).uuid)
                if uuid:
                    u = (uuid if uuid.startswith("GPU-") else "GPU-" + uuid).encode()
                    if self.lib.nvmlDeviceGetHandleByUUID(ct.c_char_p(u), ct.byref(h)) == 0:
                        return h
                    errors.append("uuid " + uuid)
            except Exception as e:  # fall back to the index
                errors.append(repr(e))
            n = ct.c_uint(0)
            self._ok(self.lib.nvmlDeviceGetCount_v2(ct.byref(n)), "nvmlDeviceGetCount_v2")
            if n.value == 1 or "CUDA_VISIBLE_DEVICES" not in os.environ:
                self._ok(self.lib.nvmlDeviceGetHandleByIndex_v2(ct.c_uint(device.index or 0), ct.byref(h)),
                         "nvmlDeviceGetHandleByIndex_v2")
                return h
            raise RuntimeError("no NVML handle: " + "; ".join(errors))

        def sample(self, h):
            ct = self.ct
            sm, smax = ct.c_uint(0), ct.c_uint(0)
            util = (ct.c_uint * 2)()
            reasons = ct.c_ulonglong(0)
            self._ok(self.lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(sm)), "nvmlDeviceGetClockInfo")  # 1 = SM clock
            self._ok(self.lib.nvmlDeviceGetMaxClockInfo(h, 1, ct.byref(smax)), "nvmlDeviceGetMaxClockInfo")
            self._ok(self.lib.nvmlDeviceGetUtilizationRates(h, util), "nvmlDeviceGetUtilizationRates")
            fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self._ok(fn(h, ct.byref(reasons)), "clock event reasons")
            return float(sm.value), float(smax.value), float(util[0]), int(reasons.value)

    def start(self):
        try:
            nv = self._Nvml()
            h = nv.handle(self.device)
            nv.sample(h)

            def loop():
                while not self.stop_flag.is_set():
                    try:
                        self.samples.append(nv.sample(h))
                    except Exception:
                        pass
                    self.stop_flag.wait(0.01)

            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            self.source = "nvml, 10 ms"
            return
        except Exception as e:
            self.thread = None
            self.nvml_error = repr(e)[:200]
        try:
            idx = self.device.index or 0
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={idx}", f"--query-gpu={self.SMI_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, 200 ms"
        except OSError:
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join(timeout=5)
        elif self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            names = [n for n, _ in self.REASONS[:4]]
            for line in out.strip().splitlines():
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm, smax = float(parts[1]), float(parts[2])
                except ValueError:
                    continue
                mask = 0
                for (n, bit), v in zip(self.REASONS[:4], parts[5:9]):
                    if v.lower() == "active":
                        mask |= bit
                self.samples.append((sm, smax, 100.0, mask))
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"], "samples": 0}
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        loaded = [s for s in self.samples if s[2] >= 50.0] or self.samples
        reasons = sorted({n for n, bit in self.REASONS for s in loaded if s[3] & bit})
        out = {"sm_mhz": statistics.median(s[0] for s in loaded), "sm_max_mhz": max(s[1] for s in self.samples),
               "reasons": reasons, "samples": len(self.samples), "samples_under_load": len(loaded),
               "source": self.source}
        if self.nvml_error:
            out["nvml_error"] = self.nvml_error
        return out


# ------------------------------------------------------------------ GPU arm: one block call per step
def _workspace_plan(nomas, cache, wl, num_splits):
    """Work plan and workspace bytes the library uses once the history is resident."""
    import ctypes
    d = nomas.nomas_kvcache.from_buffer_copy(cache.desc)
    total = sum(wl.cache_frames_hist)
    d.total_frames = total
    d.valid_frames = min(total, wl.window)
    pl = nomas.nomas_attn_plan()
    if nomas.nomas_segment_attn_plan(ctypes.byref(d), wl.n_video, wl.n_text, num_splits, ctypes.byref(pl)) != 0:
        raise RuntimeError("attention plan query failed")
    plan = {name: int(getattr(pl, name)) for name, _ in nomas.nomas_attn_plan._fields_ if name != "reserved"}
    return plan


def measure_block_call(args, wl, dev, block, steps, warmup, world, with_sampler=False, target_s=0.0):
    """Time ``steps`` steps (reset, history append, RoPE, attention [, selection, camera]) of one
    block call on workload ``wl``; returns raw per-step event timings and the step's accounting.
    With ``target_s`` the step count grows (up to 1000) until the timed steps take about that long."""
    import numpy as np
    import torch

    import segment_causal_kv_int8_b300 as nomas
    from synth import current_qkv, history_segments

    hist = history_segments(wl, block)
    q_h, k_h, v_h = current_qkv(wl, block=block)

    def dev_t(x):
        return torch.from_numpy(x).to(torch.bfloat16 if wl.io_dtype == "bf16" else torch.float32).to(dev)

    hist_d = [(dev_t(k), dev_t(v)) for k, v in hist]
    q0, k0, v0 = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (q_h, k_h, v_h))
    q, k, v = q0.clone(), k0.clone(), v0.clone()
    cache = nomas.KVCache(1, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, wl.cache_dtype,
                          device=dev)
    shadow = None
    if getattr(args, "bf16_shadow", False) and wl.cache_dtype in ("int8", "fp8"):
        shadow = nomas.KVCache(1, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, "bf16",
                               device=dev)
    att_cache = shadow if shadow is not None else cache  # the cache the attention reads
    lse = torch.empty((wl.heads, wl.n_q), dtype=torch.float32, device=dev)
    out = torch.empty_like(q)
    plan = _workspace_plan(nomas, att_cache, wl, args.num_splits)
    ws = torch.empty(max(plan["workspace_bytes"], 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)  # > 126 MB L2
    stream = torch.cuda.current_stream(dev)
    camera = args.camera
    if camera:
        g = torch.Generator(device=dev)
        g.manual_seed(wl.seed)
        cam_k = torch.randn((wl.cur_frames, camera, wl.heads, wl.head_dim), generator=g, device=dev).to(
            torch.bfloat16)
        cam_v = torch.randn(cam_k.shape, generator=g, device=dev).to(torch.bfloat16)
        cam_out = torch.empty((wl.n_video, wl.heads, wl.head_dim), dtype=torch.bfloat16, device=dev)
    keep = args.sparse
    if keep:
        import ctypes
        n_tiles = (wl.n_cache + 127) // 128
        groups = (wl.n_q + 511) // 512
        sel_tiles = torch.zeros((wl.heads, groups, max(1, nomas.sparse_keep_count(n_tiles, keep))),
                                dtype=torch.int32, device=dev)
        sel_counts = torch.zeros((wl.heads, groups), dtype=torch.int32, device=dev)
        b = ctypes.c_size_t()
        d = nomas.nomas_kvcache.from_buffer_copy(cache.desc)
        d.total_frames = sum(wl.cache_frames_hist)
        d.valid_frames = min(d.total_frames, wl.window)
        nomas.nomas_sparse_select_workspace_bytes(ctypes.byref(d), wl.n_video, wl.n_text, ctypes.byref(b))
        sel_ws = torch.empty(max(256, b.value), dtype=torch.uint8, device=dev)

    def evict_l2():
        # Write a buffer twice the L2 size, then read it back: the inputs leave
        # L2 and the flush's own dirty lines are written back here, outside the
        # timed step, instead of during it.
        flush.zero_()
        flush.view(torch.int32).sum()

    def step(ev=None):
        # ev: None or events bracketing append, RoPE, attention, (sparse) tile selection and camera
        cache.reset(zero_memory=False)
        if ev is not None:
            ev[0].record(stream)
        for kh, vh in hist_d:
            if args.append_rope:
                cache.append_rope(kh, vh, wl.theta, wl.rope_split)
            else:
                cache.append(kh, vh)
        if ev is not None:
            ev[1].record(stream)
        if shadow is not None:
            if ev is not None:
                ev[10].record(stream)
            cache.expand_into(shadow)
            if ev is not None:
                ev[11].record(stream)
        if ev is not None:
            ev[2].record(stream)
        nomas.rope3d(q, k, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
        if ev is not None:
            ev[3].record(stream)
        if keep:
            if ev is not None:
                ev[6].record(stream)
            nomas.sparse_select(att_cache, 0, q, wl.n_video, wl.n_text, keep, tiles=sel_tiles, counts=sel_counts,
                                workspace=sel_ws)
            if ev is not None:
                ev[7].record(stream)
        if ev is not None:
            ev[4].record(stream)
        if keep:
            nomas.segment_attn_sparse(att_cache, 0, q, k, v, wl.n_video, wl.n_text, sel_tiles, sel_counts,
                                      out=out, lse=lse, workspace=ws, num_splits=args.num_splits)
        else:
            nomas.segment_attn(att_cache, 0, q, k, v, wl.n_video, wl.n_text, out=out, lse=lse, workspace=ws,
                               num_splits=args.num_splits)
        if ev is not None:
            ev[5].record(stream)
        if camera:
            if ev is not None:
                ev[8].record(stream)
            nomas.camera_cross_attn(q, cam_k, cam_v, wl.cur_frames, wl.grid_h, wl.grid_w, out=cam_out)
            if ev is not None:
                ev[9].record(stream)

    def restage():
        q.copy_(q0)  # RoPE works in place: fresh un-rotated inputs for every step (untimed)
        k.copy_(k0)

    for _ in range(warmup):
        restage()
        step()
    torch.cuda.synchronize(dev)
    if target_s > 0:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        restage()
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        per = max(1e-6, e0.elapsed_time(e1) * 1e-3)
        steps = max(steps, min(1000, int(target_s / per)))
        steps = int(max_over_ranks(steps, world, dev))

    import torch.distributed as dist
    sampler = ClockSampler(dev) if with_sampler else None
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(14)] for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
        time.sleep(0.05)
    # Steps are enqueued back to back (one synchronisation after the last).  A
    # GPU-side sleep queued first holds the stream while the host enqueues all
    # steps, so no host launch latency lands between a step's events.  Each
    # step is bracketed by its own events; the L2 flush and the restaging copy
    # sit between steps, outside them, and the sleep precedes the first step.
    torch.cuda._sleep(int(2e6) * steps)
    for i in range(steps):
        restage()   # untimed, between steps: fresh inputs, then L2 evicted so they start in HBM
        evict_l2()
        evs[i][0].record(stream)
        step(evs[i][2:])
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    # The append group and RoPE each on their own after an L2 eviction (their
    # inputs in HBM, no other kernel's dirty lines to write back): the
    # kernels' own bandwidth, next to their times inside the step.
    iso = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(min(steps, 50))]
    torch.cuda._sleep(int(2e6) * len(iso))  # hold the stream while the host enqueues, as for the steps
    for ev in iso:
        restage()
        cache.reset(zero_memory=False)
        evict_l2()
        ev[0].record(stream)
        for kh, vh in hist_d:
            if args.append_rope:
                cache.append_rope(kh, vh, wl.theta, wl.rope_split)
            else:
                cache.append(kh, vh)
        ev[1].record(stream)
        evict_l2()
        ev[2].record(stream)
        nomas.rope3d(q, k, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split)
        ev[3].record(stream)
    torch.cuda.synchronize(dev)
    r = {
        "step_ms": [e[0].elapsed_time(e[1]) for e in evs],
        "append_ms": [e[2].elapsed_time(e[3]) for e in evs],
        "rope_ms": [e[4].elapsed_time(e[5]) for e in evs],
        "attn_ms": [e[6].elapsed_time(e[7]) for e in evs],
        "select_ms": [e[8].elapsed_time(e[9]) for e in evs] if keep else None,
        "camera_ms": [e[10].elapsed_time(e[11]) for e in evs] if camera else None,
        "expand_ms": [e[12].elapsed_time(e[13]) for e in evs] if shadow is not None else None,
        "clocks": clocks, "plan": plan, "hist": hist, "qkv": (q_h, k_h, v_h), "steps": steps,
        "append_iso_ms": [e[0].elapsed_time(e[1]) for e in iso],
        "rope_iso_ms": [e[2].elapsed_time(e[3]) for e in iso],
    }
    r["flops"] = sparse_flops(wl, sel_tiles.cpu().numpy(), sel_counts.cpu().numpy()) if keep else wl.attn_flops()
    r["launches_per_step"] = (len(hist) + 1 + 1 + (1 if plan["pieces_per_split_unit"] > 1 else 0)
                              + (2 if keep and wl.n_cache else 0) + (1 if camera else 0)
                              + (1 if shadow is not None else 0))
    del cache, shadow, att_cache, hist_d, flush, ws
    return r


def summarize_block_call(wl, m, world, steps, peaks, append_rope=False, camera=0):
    """Per-workload summary: attention TFLOP/s and roofline fractions, query tokens/s, step time,
    RoPE and append bandwidth (fractions of the measured copy rate and of 8 TB/s)."""
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_s = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    attn_avg = statistics.mean(m["attn_ms"])
    step_avg = statistics.mean(m["step_ms"])
    achieved = m["flops"] / (attn_avg * 1e-3) / 1e12
    el = {}
    name = "kvcache_append_rope" if append_rope else "kvcache_append"
    el[name] = hbm_entry(append_bytes(wl), 1e3 * statistics.mean(m["append_ms"]), hbm, len(wl.cache_frames_hist),
                         isolated=hbm_entry(append_bytes(wl), 1e3 * statistics.mean(m["append_iso_ms"]), hbm,
                                            len(wl.cache_frames_hist), timing="alone after an L2 eviction"))
    el["rope3d"] = hbm_entry(rope_bytes(wl), 1e3 * statistics.mean(m["rope_ms"]), hbm, 1,
                             isolated=hbm_entry(rope_bytes(wl), 1e3 * statistics.mean(m["rope_iso_ms"]), hbm, 1,
                                                timing="alone after an L2 eviction"))
    if m.get("expand_ms"):
        el["kvcache_expand"] = hbm_entry(expand_bytes(wl), 1e3 * statistics.mean(m["expand_ms"]), hbm, 1)
    if camera:
        nbytes = 2 * wl.n_video * wl.heads * wl.head_dim * 2 + 2 * wl.cur_frames * camera * wl.heads * wl.head_dim * 2
        el["camera_cross_attn"] = hbm_entry(nbytes, 1e3 * statistics.mean(m["camera_ms"]), hbm, 1,
                                            camera_tokens_per_frame=camera)
    return {
        "workload": _config_dict(wl, world, "")["workload"],
        "attention": {"tflops": achieved, "frac": achieved / peak, "frac_of_sustained": achieved / peak_s,
                      "us": 1e3 * attn_avg, "q_tokens_per_s": wl.n_q / (attn_avg * 1e-3),
                      "plan": m["plan"]},
        "step": {"ms": step_avg, "tflops": m["flops"] / (step_avg * 1e-3) / 1e12,
                 "q_tokens_per_s": wl.n_q / (step_avg * 1e-3), "steps": steps},
        "elementwise": el,
    }


def run_ours(args):
    import torch
    import torch.distributed as dist

    import segment_causal_kv_int8_b300 as nomas
    from synth import CONFIGS

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    wl = CONFIGS[args.config]
    if args.cache_dtype:
        import dataclasses
        wl = dataclasses.replace(wl, cache_dtype=args.cache_dtype)
    block = rank_block(rank)  # each rank owns an independent block's data
    peaks, src = load_peaks()

    m = measure_block_call(args, wl, dev, block, args.steps, args.warmup, world, with_sampler=True)
    total_ms = max_over_ranks(sum(m["step_ms"]), world, dev)
    ms_per_step = total_ms / args.steps
    flops = m["flops"]
    value = whole_job_value(flops, world, args.steps, total_ms)
    keep = args.sparse
    summary = summarize_block_call(wl, m, world, args.steps, peaks, args.append_rope, args.camera)
    att = summary["attention"]

    e2e = None
    if not args.no_e2e and not keep and not args.append_rope:
        e2e = _e2e(args, torch, nomas, wl, m["hist"], *m["qkv"], dev, world)
    m["hist"] = m["qkv"] = None

    configs = {}
    if not args.no_extras and not keep and not args.append_rope and not args.camera and not args.cache_dtype:
        configs = run_extras(args, wl, dev, world, peaks)

    traffic, traffic_source = _load_traffic(args.config)
    if wl.cache_dtype != CONFIGS[args.config].cache_dtype or keep:
        traffic, traffic_source = None, "not captured for this variant"
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": _config_dict(wl, world, "256 MiB buffer written then read between timed steps (L2 flush, untimed)"),
            "roofline": {"bound": "tensor", "achieved": att["tflops"], "peak": float(peaks.get("bf16_tflops", 0)),
                         "unit": UNIT, "frac": att["frac"], "frac_of_sustained": att["frac_of_sustained"],
                         "traffic": traffic, "traffic_source": traffic_source,
                         "kernel": "segment_attn_kernel" + (" + combine" if m["plan"]["pieces_per_split_unit"] > 1
                                                            else ""),
                         "attn_ms": att["us"] / 1e3, "plan": m["plan"],
                         "peak_source": f"bf16_tflops (burst) of {src} peaks"},
            "q_tokens_per_s": att["q_tokens_per_s"],
            "q_tokens_per_s_step": summary["step"]["q_tokens_per_s"],
            "elementwise": summary["elementwise"],
            "e2e": e2e,
            "gpu_launches": m["launches_per_step"] * args.steps,
            "clocks": m["clocks"],
        }
        if configs:
            line["configs"] = configs
        if args.append_rope:
            line["config"]["workload"] += "; history written by the fused RoPE + append"
        if args.bf16_shadow and wl.cache_dtype in ("int8", "fp8"):
            line["config"]["workload"] += ("; the resident window expanded to a BF16 copy after the appends "
                                           "(nomas_kvcache_expand), attention over the copy")
        if keep:
            # Executed FLOPs count each query group's kept keys; the dense
            # equivalent is the full-attention FLOPs over the same step time.
            line["config"]["workload"] += f"; block-sparse, keep {keep} of the cache tiles"
            line["sparse"] = {"keep": keep, "select_us": 1e3 * statistics.mean(m["select_ms"]),
                              "executed_flops": flops, "dense_flops": wl.attn_flops(),
                              "dense_equivalent_tflops": whole_job_value(wl.attn_flops(), world, args.steps,
                                                                         total_ms)}
            line["roofline"]["kernel"] += " (tile lists)"
        if not args.no_cpu_baseline and world == 1:
            v_cpu, desc, threads, _, _ = oracle_sample(wl, args.cpu_seconds)
            line["cpu_baseline"] = {"value": v_cpu / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
                                    "sample": desc}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_extras(args, main_wl, dev, world, peaks):
    """The other single-block workloads (timed like the headline, at least --steps steps and about
    --extra-seconds of device time each) and one whole session, for the ``configs`` key."""
    import copy

    import torch

    from synth import CONFIGS

    rank, _, _ = dist_env()
    out = {}

    def block_entry(a, wl):
        m = measure_block_call(a, wl, dev, rank_block(rank), args.steps, max(3, args.warmup), world,
                               with_sampler=True, target_s=args.extra_seconds)
        steps = m["steps"]
        m["hist"] = m["qkv"] = None
        total = max_over_ranks(sum(m["step_ms"]), world, dev)
        s = summarize_block_call(wl, m, world, steps, peaks)
        s["step"]["ms"] = total / steps
        s["step"]["whole_job_tflops"] = whole_job_value(m["flops"], world, steps, total)
        s["clocks"] = m["clocks"]
        s["gpu_launches"] = m["launches_per_step"] * steps
        if m["select_ms"]:
            # executed FLOPs count each query group's kept keys plus the current keys
            s["sparse"] = {"keep": a.sparse, "select_us": 1e3 * statistics.mean(m["select_ms"]),
                           "executed_flops": m["flops"], "dense_flops": wl.attn_flops(),
                           "dense_equivalent_tflops": whole_job_value(wl.attn_flops(), world, steps, total)}
        torch.cuda.empty_cache()
        return s

    for name in EXTRA_CONFIGS:
        if name != main_wl.name:
            out[name] = block_entry(args, CONFIGS[name])
    # The INT8 window with its BF16 copy: once per step here (the step re-appends the history), once
    # per turn in the session (the copy serves that turn's 8 steps of every block).
    sh_args = copy.copy(args)
    sh_args.bf16_shadow = True
    s = block_entry(sh_args, CONFIGS["c3_int8_window18"])
    s["note"] = "attention over the BF16 copy of the INT8 window (nomas_kvcache_expand after the appends)"
    out["c3_int8_window18_bf16_shadow"] = s
    # Block-sparse steps (tile selection + tile-list attention) keeping a quarter of the cache tiles.
    sp_args = copy.copy(args)
    sp_args.sparse = SPARSE_KEEP
    for name in ("c3_int8_window18", "c4_bf16_hist60"):
        s = block_entry(sp_args, CONFIGS[name])
        s["note"] = f"block-sparse: tile selection, then attention over the kept {SPARSE_KEEP} of the cache tiles"
        out[f"{name}_sparse{int(round(100 * SPARSE_KEEP))}"] = s
    sess = measure_session(args, CONFIGS[SESSION_CONFIG], dev, world, rank, args.turns, steps=1, warmup=[1],
                           keep=0.0, archive=False)
    out[SESSION_CONFIG] = session_summary(CONFIGS[SESSION_CONFIG], sess, world, peaks)
    torch.cuda.empty_cache()
    sess = measure_session(args, CONFIGS[SESSION_CONFIG], dev, world, rank, args.turns, steps=1, warmup=[1],
                           keep=0.0, archive=False, shadow_bf16=True)
    ss = session_summary(CONFIGS[SESSION_CONFIG], sess, world, peaks)
    ss["note"] = "the INT8 window expanded to a BF16 copy of all 54 blocks after each turn's append"
    out[SESSION_CONFIG + "_bf16_shadow"] = ss
    torch.cuda.empty_cache()
    return out


def sparse_flops(wl, tiles, counts) -> float:
    """4 * D * sum over (head, query group) of rows x (kept cache keys + current keys)."""
    total = 0.0
    for h in range(wl.heads):
        for g in range(counts.shape[1]):
            rows = min(wl.n_q, 512 * (g + 1)) - 512 * g
            kept = sum(min(128, wl.n_cache - 128 * int(t)) for t in tiles[h, g, :counts[h, g]])
            total += 4.0 * wl.head_dim * rows * (kept + wl.n_q)
    return total


def _e2e(args, torch, nomas, wl, hist, q_h, k_h, v_h, dev, world):
    """Same step through the public API with host (pinned) inputs and a host read of the output.

    ``value``: the whole step, its history segments and Q, K, V uploaded every
    step.  ``per_call_resident_cache``: the pages' serving pattern, where the
    cache stays resident between calls and each block call uploads only the
    current segment's Q, K, V and reads back O (RoPE + attention per call).
    Both run as a serving loop would: two sets of device buffers, the uploads
    on a copy stream, so the next step's inputs travel while this step
    computes, and this step's output returns while the next one computes.
    Every step's copies lie inside the timed region.
    """
    import torch.distributed as dist

    def pin(x, bf16):
        t = torch.from_numpy(x)
        t = t.to(torch.bfloat16) if bf16 else t
        return t.pin_memory()

    hist_h = [(pin(k, wl.io_dtype == "bf16"), pin(v, wl.io_dtype == "bf16")) for k, v in hist]
    qkv_h = [pin(x, True) for x in (q_h, k_h, v_h)]
    out_h = torch.empty(qkv_h[0].shape, dtype=torch.bfloat16).pin_memory()
    bufs = []
    for _ in range(2):
        bufs.append({"hist": [(torch.empty_like(a, device=dev), torch.empty_like(b, device=dev)) for a, b in hist_h],
                     "qkv": [torch.empty_like(x, device=dev) for x in qkv_h],
                     "out": torch.empty(qkv_h[0].shape, dtype=torch.bfloat16, device=dev)})
    cache = nomas.KVCache(1, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames, wl.cache_dtype,
                          device=dev)
    plan = _workspace_plan(nomas, cache, wl, args.num_splits)
    ws = torch.empty(max(plan["workspace_bytes"], 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(device=dev)
    qkv_bytes = sum(x.numel() * x.element_size() for x in qkv_h)
    hist_bytes = sum(a.numel() * a.element_size() * 2 for a, _ in hist_h)
    d2h = out_h.numel() * out_h.element_size()

    def upload(b, with_hist):
        with torch.cuda.stream(copy):
            if with_hist:
                for (a, bb), (ad, bd) in zip(hist_h, bufs[b]["hist"]):
                    ad.copy_(a, non_blocking=True)
                    bd.copy_(bb, non_blocking=True)
            for x, xd in zip(qkv_h, bufs[b]["qkv"]):
                xd.copy_(x, non_blocking=True)

    def compute(b, with_hist):
        qd, kd, vd = bufs[b]["qkv"]
        if with_hist:
            cache.reset(zero_memory=False)
            for ad, bd in bufs[b]["hist"]:
                cache.append(ad, bd)
        nomas.rope3d(qd, kd, wl.cur_frames, wl.grid_h, wl.grid_w, wl.t0, wl.theta, wl.rope_split, stream=comp)
        nomas.segment_attn(cache, 0, qd, kd, vd, wl.n_video, wl.n_text, out=bufs[b]["out"], workspace=ws,
                           num_splits=args.num_splits, stream=comp)

    def pipeline(n, with_hist):
        """n steps; returns elapsed ms from the first upload to the last output's arrival on the host."""
        up = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        flush.view(torch.int32).sum()
        copy.wait_stream(comp)
        e0.record(copy)
        upload(0, with_hist)
        up[0].record(copy)
        for i in range(n):
            b = i % 2
            comp.wait_event(up[b])
            compute(b, with_hist)
            done[b].record(comp)
            if i + 1 < n:
                if i >= 1:
                    copy.wait_event(done[1 - b])  # buffers of step i - 1 are free again
                upload(1 - b, with_hist)
                up[1 - b].record(copy)
            copy.wait_event(done[b])
            with torch.cuda.stream(copy):
                out_h.copy_(bufs[b]["out"], non_blocking=True)
        e1.record(copy)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    pipeline(max(2, args.warmup), True)
    if world > 1:
        dist.barrier()
    total = max_over_ranks(pipeline(args.steps, True), world, dev)
    val = whole_job_value(wl.attn_flops(), world, args.steps, total)
    # The cache now holds the history (resident from the last step).
    pipeline(max(2, args.warmup), False)
    total_pc = max_over_ranks(pipeline(args.steps, False), world, dev)
    res = {"value": val, "unit": UNIT, "h2d_bytes_per_step": int(hist_bytes + qkv_bytes),
           "d2h_bytes_per_step": int(d2h), "ms_per_step": total / args.steps,
           "pipelining": "two buffer sets; uploads and read-backs on a copy stream overlap the kernels",
           "per_call_resident_cache": {"value": whole_job_value(wl.attn_flops(), world, args.steps, total_pc),
                                       "unit": UNIT, "ms_per_call": total_pc / args.steps,
                                       "h2d_bytes_per_call": int(qkv_bytes), "d2h_bytes_per_call": int(d2h)}}
    del cache, bufs, ws, flush
    return res


_CSRC = "segment_causal_kv_int8_b300/csrc/"
ATTN_SOURCES = tuple(_CSRC + f for f in ("segment_attn.cu", "attn_common.cuh", "sm100.cuh", "checks.cuh"))


def attn_source_hash() -> str:
    """sha256 over the attention kernel's sources (decides whether committed counters still apply)."""
    import hashlib
    h = hashlib.sha256()
    for rel in ATTN_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _load_traffic(config):
    """DRAM bytes per attention launch from the committed ncu summary of this config.

    ``profiles/attention_<config>.md`` records ``dram_bytes_per_launch`` (an
    ncu capture of that launch) and the ``kernel_source_sha256`` of the sources
    it was captured from; the value is used only while the sources still hash
    the same.  Returns ``(bytes or None, description of the source)``.
    """
    rel = os.path.join("profiles", f"attention_{config}.md")
    fields = {}
    try:
        with open(os.path.join(ROOT, rel)) as f:
            for line in f:
                if ":" in line:
                    k, _, v = line.strip().lstrip("-* `").partition(":")
                    fields[k.strip(" `")] = v.strip(" `")
    except OSError:
        return None, f"no ncu capture committed ({rel} missing)"
    if fields.get("kernel_source_sha256") != attn_source_hash():
        return None, f"{rel} was captured from other kernel sources (hash differs)"
    try:
        return int(float(fields["dram_bytes_per_launch"])), (
            f"ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch, {rel} (same kernel sources)")
    except (KeyError, ValueError):
        return None, f"{rel} holds no dram_bytes_per_launch"


# ------------------------------------------------------------------ session workload
def session_flops(wl, turns: int, keep: float = 0.0, dense_steps: int = 2) -> float:
    """Attention FLOPs of a session: every turn runs steps x blocks calls over the cache resident then.

    With ``keep`` (block-sparse after ``dense_steps`` dense steps) the sparse
    calls count ceil(keep * T) kept tiles of 128 keys per query group (capped
    at the resident keys): an upper bound, since a kept partial last tile
    holds fewer keys.
    """
    import math
    total = 0.0
    for t in range(turns):
        n_c = min(t * wl.cur_frames, wl.window) * wl.tpf
        dense = 4.0 * wl.n_q * (n_c + wl.n_q) * wl.head_dim * wl.heads
        if not keep:
            total += wl.steps * wl.blocks * dense
            continue
        n_t = -(-n_c // 128)
        kept = min(n_c, 128 * min(n_t, math.ceil(keep * n_t - 1e-9)))
        sparse = 4.0 * wl.n_q * (kept + wl.n_q) * wl.head_dim * wl.heads
        n_dense = min(dense_steps, wl.steps)
        total += wl.blocks * (n_dense * dense + (wl.steps - n_dense) * sparse)
    return total


def measure_session(args, wl, dev, world, rank, turns, steps, warmup, keep, archive, shadow_bf16=False):
    """Time ``steps`` whole sessions of ``turns`` turns: per turn, steps x blocks calls of RoPE +
    segment attention (each block against its own window of the shared INT8 cache), then one append
    of the finished segment's K/V for all blocks.  ``warmup`` lists the turn counts of the untimed
    sessions run first.  ``shadow_bf16``: after each append, expand the window to a BF16 copy of all
    blocks (nomas_kvcache_expand) and run the next turn's attention over the copy."""
    import ctypes

    import torch
    import torch.distributed as dist

    import segment_causal_kv_int8_b300 as nomas
    from synth import current_qkv_torch, segment_kv_torch

    turns = min(turns, wl.turns)
    seed_block = rank_block(rank)
    cache = nomas.KVCache(wl.blocks, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames,
                          wl.cache_dtype, device=dev)
    shadow = None
    if shadow_bf16 and wl.cache_dtype in ("int8", "fp8"):
        shadow = nomas.KVCache(wl.blocks, wl.heads, wl.grid_h, wl.grid_w, wl.capacity_frames, wl.past_frames,
                               "bf16", device=dev)
    att_cache = shadow if shadow is not None else cache  # the cache the attention reads
    # A pool of current-segment inputs (values do not change the work) and one
    # finished segment per turn, drawn on the device before timing.
    pool = [current_qkv_torch(wl, seed_block, s, b, dev) for s, b in ((0, 0), (1, 1), (2, 2), (3, 3))]
    seg_k, seg_v = segment_kv_torch(wl, seed_block, wl.cur_frames, wl.blocks, dev)
    out = torch.empty_like(pool[0][0])
    ws_bytes = 0
    for vf in range(0, wl.window + 1):
        d = nomas.nomas_kvcache.from_buffer_copy(att_cache.desc)
        d.total_frames, d.valid_frames = vf, vf
        b = ctypes.c_size_t()
        nomas.nomas_segment_attn_workspace_bytes(ctypes.byref(d), wl.n_video, wl.n_text, 0, ctypes.byref(b))
        ws_bytes = max(ws_bytes, int(b.value))
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    calls = [0]
    if keep:
        # Block-sparse after two dense steps: per block a kept-tile list and
        # the mean keys of its window (computed at the first sparse step of a
        # turn, reused by the later ones while the cache is unchanged).
        n_tiles_max = -(-wl.window * wl.tpf // 128)
        groups = -(-wl.n_q // 512)
        sel_tiles = torch.zeros((wl.heads, groups, max(1, nomas.sparse_keep_count(n_tiles_max, keep))),
                                dtype=torch.int32, device=dev)
        sel_counts = torch.zeros((wl.heads, groups), dtype=torch.int32, device=dev)
        kbar_bytes = -(-wl.heads * n_tiles_max * 128 * 4 // 256) * 256
        kbar = torch.empty((wl.blocks, kbar_bytes), dtype=torch.uint8, device=dev)
    host_archive = None
    if archive:
        # Host KV archive of every appended frame (pinned, one session's worth).
        host_archive = torch.empty(turns * wl.cur_frames * cache.archive_frame_bytes(),
                                   dtype=torch.uint8).pin_memory()

    def session(n_turns):
        cache.reset(zero_memory=False)
        if shadow is not None:
            shadow.reset(zero_memory=False)
        used = 0
        for t in range(n_turns):
            # the plan (and so whether a merge pass follows) depends on the resident frames
            merge = 1 if att_cache.attn_plan(wl.n_video, wl.n_text)["pieces_per_split_unit"] > 1 else 0
            for s in range(wl.steps):
                for blk in range(wl.blocks):
                    q, k, v = pool[(s * wl.blocks + blk) % len(pool)]
                    nomas.rope3d(q, k, wl.cur_frames, wl.grid_h, wl.grid_w, cache.total_frames, wl.theta,
                                 wl.rope_split)
                    if keep and s >= 2 and cache.valid_frames > 0:
                        nomas.sparse_select(att_cache, blk, q, wl.n_video, wl.n_text, keep, tiles=sel_tiles,
                                            counts=sel_counts, workspace=kbar[blk], reuse_key_means=s > 2)
                        nomas.segment_attn_sparse(att_cache, blk, q, k, v, wl.n_video, wl.n_text, sel_tiles,
                                                  sel_counts, out=out, workspace=ws)
                        calls[0] += 3 + (1 if s == 2 else 0)
                    else:
                        nomas.segment_attn(att_cache, blk, q, k, v, wl.n_video, wl.n_text, out=out, workspace=ws)
                        calls[0] += 1 + merge
                    calls[0] += 1
            if host_archive is not None:
                used = cache.append_archive(seg_k, seg_v, host_archive, used)
            else:
                cache.append(seg_k, seg_v)
            calls[0] += 1
            if shadow is not None:
                cache.expand_into(shadow)
                calls[0] += 1

    for n in warmup:
        session(min(n, turns))
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.05)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    calls[0] = 0
    for i in range(steps):
        evs[i][0].record(stream)
        session(turns)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), world, dev)
    del cache, shadow, att_cache, ws, pool
    return {"total_ms": total_ms, "steps": steps, "turns": turns, "calls": calls[0], "clocks": clocks,
            "flops": session_flops(wl, turns, keep), "keep": keep, "archive": archive, "shadow_bf16": shadow_bf16}


def session_summary(wl, s, world, peaks):
    peak_s = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    tf = whole_job_value(s["flops"], world, s["steps"], s["total_ms"]) / world
    calls = s["turns"] * wl.steps * wl.blocks
    return {"workload": f"{wl.name}: {s['turns']} turns x {wl.steps} steps x {wl.blocks} blocks of RoPE + segment "
                        f"attention (Nq={wl.n_q}, INT8 window {wl.window} frames), one 54-block append per turn",
            "session_s": s["total_ms"] / s["steps"] / 1e3, "attention_calls": calls,
            "tflops": tf, "frac_of_sustained": tf / peak_s,
            "q_tokens_per_s": calls * wl.n_q / (s["total_ms"] / s["steps"] / 1e3),
            "peak": peak_s, "peak_source": "bf16_tflops_sustained (a seconds-long step)",
            "gpu_launches": s["calls"], "clocks": s["clocks"]}


def run_session(args):
    """The simulated multi-turn session as the headline workload (``--config c5_session12``):
    one timed step = one whole session of ``--turns`` turns."""
    import torch
    import torch.distributed as dist

    from synth import CONFIGS

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    wl = CONFIGS[args.config]
    keep = args.sparse
    s = measure_session(args, wl, dev, world, rank, args.turns, args.steps, [args.turns] * args.warmup, keep,
                        args.archive, shadow_bf16=args.bf16_shadow)
    turns = s["turns"]
    total_ms = s["total_ms"]
    flops = s["flops"]
    value = whole_job_value(flops, world, args.steps, total_ms)
    peaks, src = load_peaks()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{wl.name}: {turns} turns x {wl.steps} steps x {wl.blocks} blocks of RoPE + "
                                   f"segment attention ({wl.heads} heads x {wl.head_dim}, Nq={wl.n_q}, INT8 cache "
                                   f"window {wl.window} frames), one 54-block append per turn; one step = one session",
                       "turns": turns, "attention_calls": turns * wl.steps * wl.blocks,
                       "host_archive": bool(args.archive),
                       "bf16_shadow": bool(args.bf16_shadow),
                       "l2": "working set (54 blocks' caches, input pool) far larger than L2",
                       "parallelism": f"replica x{world} (independent sessions per GPU)"},
            "roofline": {"bound": "tensor", "achieved": value / world, "peak": float(peaks["bf16_tflops_sustained"]),
                         "unit": UNIT, "frac": value / world / float(peaks["bf16_tflops_sustained"]),
                         "traffic": None, "traffic_source": "not captured (thousands of launches per step)",
                         "kernel": "whole session (attention dominant)",
                         "peak_source": f"bf16_tflops_sustained of {src} peaks (a seconds-long step)"},
            "q_tokens_per_s": turns * wl.steps * wl.blocks * wl.n_q * args.steps / (total_ms * 1e-3),
            "gpu_launches": s["calls"], "clocks": s["clocks"],
        }
        if keep:
            line["config"]["workload"] += (f"; steps 0-1 dense, steps 2-{wl.steps - 1} block-sparse keeping {keep} "
                                           "of the cache tiles (mean keys computed once per turn and block)")
            line["sparse"] = {"keep": keep, "executed_flops_upper_bound": flops,
                              "dense_flops": session_flops(wl, turns),
                              "dense_equivalent_tflops": whole_job_value(session_flops(wl, turns), world,
                                                                         args.steps, total_ms)}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.config == SESSION_CONFIG:
        return run_session(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
