// attn_common.cuh - pieces shared by both forms of the segment-attention
// kernel (one CTA per work item with a BF16 cache; CTA pairs with a one-byte
// cache): tile sizes, the key-tile walk (dense or block-sparse), the decoding
// of a work item of the plan, and the softmax / epilogue role of warps 0-7.
//
// What the kernels compute (the "segment-wise causal joint attention" of the
// madebyagents.com model page over the lifelong KV cache of the orcarouter.ai
// explainer, section "Die Schleife"): per head, O = softmax(s Q K^T) V where
// the queries are the current segment's video + text tokens and the keys are
// the resident cache slots followed by the current segment's own tokens.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "checks.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace nomas {
namespace attn {

constexpr int kThreads = 512;
constexpr int kTileBytes = 128 * 128 * 2;   // one bf16 tile: [2 panels][128 rows][128 B]
constexpr int kPanelBytes = 128 * 128;      // 64 bf16 columns x 128 rows, 128B-swizzled
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);  // S = Q K^T (both K-major)
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 128, true);   // O += P V (V is N-major)
constexpr float kLazyRescale = 8.0f;        // log2 of the tolerated growth of exp terms
constexpr float kLn2 = 0.69314718055994531f;
// Register budget per warpgroup after the role split (launch: 128 per thread x
// 512 threads).  The softmax warpgroups hold a whole 128-column score row;
// 2 x 128 x 184 + 2 x 128 x 72 = 65536, the CTA's launch allocation.
constexpr uint32_t kSoftmaxRegs = 184;
constexpr uint32_t kControlRegs = 72;   // warps 8-11: TMA producer, MMA issuer
constexpr uint32_t kFillerRegs = 72;    // warps 12-15: INT8 ring fillers

struct TileInfo {
  bool cache;
  int row0;
  int valid;
};

// The key tiles a CTA visits, in order: n_cache cache tiles (all resident
// ones, or the kept list of block-sparse attention), then every current tile.
struct KeyTiles {
  int n_cache;
  const int* list;  // null: cache tiles 0 .. n_cache-1
};

__device__ __forceinline__ KeyTiles key_tiles(const AttnParams& p, int head, int qblk) {
  KeyTiles kt;
  if (p.sparse_tiles == nullptr) {
    kt.n_cache = p.n_cache_tiles;
    kt.list = nullptr;
  } else {
    // Query group = two consecutive 256-query blocks (one CTA pair for INT8).
    const size_t hg = static_cast<size_t>(head) * p.n_groups + (qblk >> 1);
    kt.n_cache = min(max(p.sparse_counts[hg], 0), min(p.max_keep, p.n_cache_tiles));
    kt.list = p.sparse_tiles + hg * p.max_keep;
  }
  return kt;
}

__device__ __forceinline__ TileInfo tile_info(int j, const AttnParams& p, const KeyTiles& kt) {
  TileInfo t;
  if (j < kt.n_cache) {
    int c = kt.list ? kt.list[j] : j;
    if (c < 0 || c >= p.n_cache_tiles) {
      // A bad list entry: stay inside the cache and report it.
      if (p.err) atomicCAS(p.err, 0u, 1u /* NOMAS_ERR_INVALID_ARG */);
      c = min(max(c, 0), p.n_cache_tiles - 1);
    }
    t.cache = true;
    t.row0 = c * 128;
    t.valid = min(128, p.nc - t.row0);
  } else {
    t.cache = false;
    t.row0 = (j - kt.n_cache) * 128;
    t.valid = min(128, p.nq - t.row0);
  }
  return t;
}

// A work item of the plan: whole unit (items < n_full) or one piece of a
// split unit.  For CTA pairs (one-byte caches) CTA r of the pair takes query
// block 2 * (unit's block pair) + r.  Pieces keep their partial rows at
// [pieces][ctas per unit][256 rows] of the workspace.
struct WorkItem {
  int unit, split, nsplit, head, qblk, q_row0;
  size_t piece_row0;
};

__device__ __forceinline__ WorkItem decode_item(const AttnParams& p, int item, int pair_rank, bool pair) {
  WorkItem w;
  if (item < p.n_full) {
    w.unit = item;
    w.split = 0;
    w.nsplit = 1;
  } else {
    const int j = item - p.n_full;
    w.unit = p.n_full + j / p.tail_splits;
    w.split = j - (j / p.tail_splits) * p.tail_splits;
    w.nsplit = p.tail_splits;
  }
  w.head = w.unit / p.units_per_head;
  const int ublk = w.unit - w.head * p.units_per_head;
  w.qblk = pair ? 2 * ublk + pair_rank : ublk;
  w.q_row0 = w.qblk * 256;
  w.piece_row0 = w.nsplit > 1 ? (static_cast<size_t>(item - p.n_full) * (pair ? 2 : 1) + pair_rank) * 256 : 0;
  return w;
}

// Warps 0-7 (softmax and epilogue).  Warpgroup t owns query tile t (rows
// 128 t .. 128 t + 127 of the work item's 256), one thread per row, its scores
// in tensor-memory columns 128 t .. 128 t + 127 and its output accumulator in
// columns 256 + 128 t .. 256 + 128 t + 127.  s_full[t] / pv_done[t] complete
// when S_t of the next key tile / the last P_t V are in tensor memory;
// arrive_p(t) (lane 0 of each warp) reports that P_t is stored.
template <typename ArriveP>
__device__ __forceinline__ void softmax_role(const AttnParams& p, const KeyTiles& kt, const WorkItem& wi,
                                             int t_begin, int n_iter, uint32_t tmem, uint64_t* s_full,
                                             uint64_t* pv_done, AbortState* ab, ArriveP arrive_p) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // ------------------------------------------------------------ softmax
  // One thread per query row.  Per key tile: the whole 128-column score row
  // comes out of tensor memory in one batch, the row maximum is a tree of
  // three-input maxima, and the exponentials use packed f32x2 FMAs with four
  // independent packed accumulators for the row sum.  The running maximum m
  // (log2 domain) only moves when the tile maximum exceeds it by more than
  // kLazyRescale; O and l are then rescaled by exp2(m_old - m_new).
  regs_grow<kSoftmaxRegs>();
  const int t = warp >> 2;
  const int quad = warp & 3;
  const int row = quad * 32 + lane;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const uint32_t s_col = t * 128;
  const uint32_t o_col = 256 + t * 128;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  float m = -INFINITY;
  uint64_t lacc[4] = {0ull, 0ull, 0ull, 0ull};  // packed partial row sums (0.0f bits are 0)
  bool ok = true;
  for (int it = 0; it < n_iter; ++it) {
    const int valid = tile_info(t_begin + it, p, kt).valid;
    if (!warp_wait(&s_full[t], it & 1, ab, p.err)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t v[128];
    tmem_ld_x64_nowait(lane_base + s_col, v);
    tmem_ld_x64_nowait(lane_base + s_col + 64, v + 64);
    tmem_wait_ld();
    if (valid < 128) {
#pragma unroll
      for (int i = 0; i < 128; ++i)
        if (i >= valid) v[i] = __float_as_uint(-INFINITY);
    }
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 128; i += 8) {
      m0 = fmax3(m0, __uint_as_float(v[i + 0]), __uint_as_float(v[i + 1]));
      m1 = fmax3(m1, __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
      m2 = fmax3(m2, __uint_as_float(v[i + 4]), __uint_as_float(v[i + 5]));
      m3 = fmax3(m3, __uint_as_float(v[i + 6]), __uint_as_float(v[i + 7]));
    }
    const float m_tile = fmax3(m0, m1, fmaxf(m2, m3)) * sl2;
    const bool need = m_tile > m + kLazyRescale;  // always true on the first tile (m = -inf)
    const bool any_need = __any_sync(0xffffffffu, need);
    float alpha = 1.0f;
    if (any_need) {
      const float m_new = need ? m_tile : m;
      alpha = fast_exp2(m - m_new);  // 0 on the first tile, 1 where nothing moves
      const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
      for (int k = 0; k < 4; ++k) lacc[k] = f2_mul(lacc[k], a2);
      m = m_new;
    }
    const uint64_t negm = f2_pack(-m, -m);
    uint32_t pk[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const uint64_t x = f2_fma(f2_pack(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), sl2x2, negm);
      float x0, x1;
      f2_unpack(x, x0, x1);
      const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
      lacc[i & 3] = f2_add(lacc[i & 3], f2_pack(p0, p1));
      pk[i] = pack_bf16x2(p0, p1);
    }
    tmem_st_x64(lane_base + s_col, pk);
    if (any_need && it > 0) {
      // O_t holds the previous tiles' P.V (complete: S_t of this tile was
      // issued after it); bring it to the new reference maximum.
      const uint64_t a2 = f2_pack(alpha, alpha);
      uint32_t o[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld_x32(lane_base + o_col + 32 * c, o);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const uint64_t x = f2_mul(f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2);
          float x0, x1;
          f2_unpack(x, x0, x1);
          o[i] = __float_as_uint(x0);
          o[i + 1] = __float_as_uint(x1);
        }
        tmem_st_x32(lane_base + o_col + 32 * c, o);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive_p(t);
  }
  float l;
  {
    const uint64_t s01 = f2_add(lacc[0], lacc[1]), s23 = f2_add(lacc[2], lacc[3]);
    float a, b;
    f2_unpack(f2_add(s01, s23), a, b);
    l = a + b;
  }
  if (ok && n_iter > 0 && warp_wait(&pv_done[t], 0, ab, p.err)) {
    tc_fence_after();
    const int grow = wi.q_row0 + t * 128 + row;
    bool live = grow < p.nq;
    const float inv_l = 1.0f / l;
    const float lse_val = (m + log2f(l)) * kLn2;
    uint32_t v[32];
    if (wi.nsplit == 1) {
      __nv_bfloat16* dst = p.out + (static_cast<size_t>(grow) * p.heads + wi.head) * 128;
      live = live && in_bounds((static_cast<long long>(grow) * p.heads + wi.head) * 128, 128,
                               static_cast<long long>(p.nq) * p.heads * 128, p.err);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld_x32(lane_base + o_col + 32 * c, v);
        if (live) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[8 * g + 0]) * inv_l, __uint_as_float(v[8 * g + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(v[8 * g + 2]) * inv_l, __uint_as_float(v[8 * g + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(v[8 * g + 4]) * inv_l, __uint_as_float(v[8 * g + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(v[8 * g + 6]) * inv_l, __uint_as_float(v[8 * g + 7]) * inv_l);
            *reinterpret_cast<uint4*>(dst + 32 * c + 8 * g) = w;
          }
        }
      }
      if (live && p.lse) p.lse[static_cast<size_t>(wi.head) * p.nq + grow] = lse_val;
    } else {
      const size_t prow = wi.piece_row0 + t * 128 + row;
      float* dst = p.ws_o + prow * 128;
      live = live && in_bounds(static_cast<long long>(prow), 1, p.ws_rows, p.err);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld_x32(lane_base + o_col + 32 * c, v);
        if (live) {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            float4 w = make_float4(__uint_as_float(v[4 * g + 0]) * inv_l, __uint_as_float(v[4 * g + 1]) * inv_l,
                                   __uint_as_float(v[4 * g + 2]) * inv_l, __uint_as_float(v[4 * g + 3]) * inv_l);
            *reinterpret_cast<float4*>(dst + 32 * c + 4 * g) = w;
          }
        }
      }
      if (live) p.ws_lse[prow] = lse_val;
    }
  } else if (ok && n_iter == 0 && wi.nsplit > 1) {
    // A piece with no key tile (a block-sparse list shorter than the piece
    // count) contributes weight zero to the combine: O = 0, LSE = -inf.
    const int grow = wi.q_row0 + t * 128 + row;
    if (grow < p.nq && in_bounds(static_cast<long long>(wi.piece_row0 + t * 128 + row), 1, p.ws_rows, p.err)) {
      const size_t prow = wi.piece_row0 + t * 128 + row;
      float4* dst = reinterpret_cast<float4*>(p.ws_o + prow * 128);
#pragma unroll 4
      for (int c = 0; c < 32; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      p.ws_lse[prow] = -INFINITY;
    }
  }
}

}  // namespace attn
}  // namespace nomas
