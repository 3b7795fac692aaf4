// segment_attn.cu - segment-causal attention over [resident KV cache ; current
// segment] for one transformer block, on B300 tensor cores (tcgen05 + TMEM +
// TMA), with the INT8 cache dequantised to BF16 in shared memory.
//
// What it computes (the "segment-wise causal joint attention" of the
// madebyagents.com model page over the lifelong KV cache of the orcarouter.ai
// explainer, section "Die Schleife"): per head, O = softmax(s Q K^T) V where
// the queries are the current segment's video + text tokens and the keys are
// the resident cache slots followed by the current segment's own tokens.
//
// Design (one CTA = one head x 256 query rows x its whole key range or one
// piece of it, as the work plan says):
//   warps 0-3   softmax for query tile 0 (rows   0..127), one thread per row
//   warps 4-7   softmax for query tile 1 (rows 128..255)
//   warp  8     TMA producer: Q once, then K/V tiles of 128 keys (into the
//               4-slot ring for a BF16 cache, into int8 staging slots for INT8)
//   warp  9     TMEM allocator + tcgen05.mma issuer (one elected lane)
//   warps 12-15 (INT8 cache) fill the ring: dequantise staged int8 tiles,
//               fetch current-segment tiles by TMA
// One-byte caches launch clusters of two CTAs on adjacent query blocks of the
// same head: each dequantises its 64-row half of every cache tile and copies
// it into the partner's ring slot, so both see the whole tile.
// Tensor memory (512 columns): S0 | S1 | O0 | O1, 128 f32 columns each; the
// bf16 probabilities P_t overwrite the first 64 columns of S_t and feed the
// P.V product straight from tensor memory.  Softmax is online in the log2
// domain with a lazy rescale of O (only when the running max grows by more
// than 8, i.e. a factor 256), which is exact up to rounding.  Splits of the
// key range write f32 partial outputs and log-sum-exps that a second kernel
// combines in a fixed order, so results are reproducible bit for bit.
//
// Every wait on an mbarrier is bounded (about one second); on timeout the CTA
// records an error, waits briefly for its own copies and MMAs, frees tensor
// memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn_common.cuh"
#include "checks.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace nomas {
namespace attn {

constexpr int kI8HalfBytes = 64 * 128;      // one CTA's half of an int8 tile: [64 rows][128 B], 128B-swizzled
constexpr int kWarpRowBytes = 16 * 128;     // 16 rows of one bf16 panel (one filler warp's share of a half)

template <bool kInt8>
struct Layout {
  // bf16 ring slots (K and V tiles alternate).  Four measured faster than five
  // for the BF16 cache too (c2 266 -> 260 us, c4 2305 -> 2272 us).
  static constexpr int NS = 4;
  static constexpr int NI = kInt8 ? 4 : 0;  // int8 staging slots (half tiles)
  static constexpr int kQ = 0;
  static constexpr int kRing = 2 * kTileBytes;
  static constexpr int kStage = kRing + NS * kTileBytes;
  static constexpr int kBars = kStage + NI * kI8HalfBytes;
  // barrier indices
  static constexpr int bQ = 0;
  static constexpr int bRingFull = 1;
  static constexpr int bRingEmpty = bRingFull + NS;
  static constexpr int bStageFull = bRingEmpty + NS;
  static constexpr int bStageEmpty = bStageFull + NI;
  static constexpr int bSFull = bStageEmpty + NI;  // [2]
  static constexpr int bPFull = bSFull + 2;         // [2]
  static constexpr int bPVDone = bPFull + 2;        // [2]
  static constexpr int bFinal = bPVDone + 2;
  static constexpr int kNumBars = bFinal + 1;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;  // slack for aligning the base to 1024 B
};
static_assert(Layout<false>::kAlloc <= 232448, "bf16 layout exceeds shared memory");
static_assert(Layout<true>::kAlloc <= 232448, "int8 layout exceeds shared memory");

template <bool kInt8, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    segment_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kcur,
                        const __grid_constant__ CUtensorMap tm_vcur, const __grid_constant__ CUtensorMap tm_kc,
                        const __grid_constant__ CUtensorMap tm_vc, const AttnParams p) {
  using L = Layout<kInt8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  AbortState* ab = reinterpret_cast<AbortState*>(smem + L::kMisc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Work item -> (unit, piece).  One-byte caches launch clusters of two CTAs
  // along x, both on the same item.
  const int item = kInt8 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int pair_rank = kInt8 ? static_cast<int>(blockIdx.x & 1u) : 0;
  const WorkItem wi = decode_item(p, item, pair_rank, kInt8);
  const int split = wi.split, nsplit = wi.nsplit, head = wi.head, qblk = wi.qblk, q_row0 = wi.q_row0;
  const KeyTiles kt = key_tiles(p, head, qblk);
  const int n_tiles = kt.n_cache + p.n_cur_tiles;
  const int t_begin = static_cast<int>((static_cast<long long>(split) * n_tiles) / nsplit);
  const int t_end = static_cast<int>((static_cast<long long>(split + 1) * n_tiles) / nsplit);
  const int n_iter = t_end - t_begin;
  const int bh = p.block_head_base + head;

  if (threadIdx.x == 0) {
    mbar_init(&bars[L::bQ], 1);
    for (int s = 0; s < L::NS; ++s) {
      // INT8: one arrival per local filler warp, plus the transaction bytes
      // of the partner's half tile; both CTAs' MMA warps release every slot
      // (multicast commit).
      mbar_init(&bars[L::bRingFull + s], kInt8 ? 4 : 1);
      mbar_init(&bars[L::bRingEmpty + s], kInt8 ? 2 : 1);
    }
    for (int s = 0; s < L::NI; ++s) {
      mbar_init(&bars[L::bStageFull + s], 1);
      mbar_init(&bars[L::bStageEmpty + s], 4);  // one arrival per filler warp
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[L::bSFull + t], 1);
      mbar_init(&bars[L::bPFull + t], 4);  // one arrival per softmax warp
      mbar_init(&bars[L::bPVDone + t], 1);
    }
    mbar_init(&bars[L::bFinal], 1);
    ab->flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // INT8: the pair's barriers must be initialised before either CTA signals the other.
  if constexpr (kInt8) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t rank = kInt8 ? cluster_ctarank() : 0u;  // position in the CTA pair

  uint8_t* sQ = smem + L::kQ;
  uint8_t* sRing = smem + L::kRing;
  uint8_t* sStage = smem + L::kStage;

  if (warp >= 8 && warp < 12) regs_shrink<kControlRegs>();
  if (warp >= 12) regs_shrink<kFillerRegs>();

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // BF16 cache: fills every ring slot.  INT8 cache: loads int8 cache tiles
    // into the staging slots only; the dequantising warps fill the ring (each
    // ring has exactly one filler, so a filler never waits on an empty-barrier
    // more than one phase ahead of it).
    int r_done = 0, ri_done = 0;  // ring / staging uses issued so far
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_kcur);
      tma_prefetch_desc(&tm_vcur);
      if (p.n_cache_tiles > 0) {
        tma_prefetch_desc(&tm_kc);
        tma_prefetch_desc(&tm_vc);
      }
      mbar_arrive_expect_tx(&bars[L::bQ], 2 * kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int pn = 0; pn < 2; ++pn)
          tma_load_3d(sQ + t * kTileBytes + pn * kPanelBytes, &tm_q, &bars[L::bQ], pn * 64, head,
                      q_row0 + t * 128);
    }
    __syncwarp();
    for (int it = 0; it < n_iter && ok; ++it) {
      const TileInfo ti = tile_info(t_begin + it, p, kt);
      for (int kv = 0; kv < 2 && ok; ++kv) {
        const int r = 2 * it + kv;
        if constexpr (kInt8) {
          if (!ti.cache) continue;
          const int si = ri_done % L::NI, ui = ri_done / L::NI;
          if (ui > 0 && !warp_wait(&bars[L::bStageEmpty + si], (ui - 1) & 1, ab, p.err)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            uint64_t* fb = &bars[L::bStageFull + si];
            (void)(in_bounds(ti.row0, 1, p.nc, p.err) && in_bounds(bh, 1, p.block_heads, p.err));
            mbar_arrive_expect_tx(fb, kI8HalfBytes);
            tma_load_3d(sStage + si * kI8HalfBytes, kv ? &tm_vc : &tm_kc, fb, 0, ti.row0 + 64 * static_cast<int>(rank),
                        bh);
          }
          ++ri_done;
        } else {
          const int s = r % L::NS, u = r / L::NS;
          if (u > 0 && !warp_wait(&bars[L::bRingEmpty + s], (u - 1) & 1, ab, p.err)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            uint64_t* fb = &bars[L::bRingFull + s];
            (void)(ti.cache ? in_bounds(ti.row0, 1, p.nc, p.err) && in_bounds(bh, 1, p.block_heads, p.err)
                            : in_bounds(ti.row0, 1, p.nq, p.err));
            mbar_arrive_expect_tx(fb, kTileBytes);
            uint8_t* dst = sRing + s * kTileBytes;
            for (int pn = 0; pn < 2; ++pn) {
              if (ti.cache)
                tma_load_3d(dst + pn * kPanelBytes, kv ? &tm_vc : &tm_kc, fb, pn * 64, ti.row0, bh);
              else
                tma_load_3d(dst + pn * kPanelBytes, kv ? &tm_vcur : &tm_kcur, fb, pn * 64, head, ti.row0);
            }
          }
          r_done = r + 1;
        }
        __syncwarp();
      }
    }
    if (!ok) {
      // Abort: let our own copies land before the CTA's shared memory goes away.
      warp_wait_teardown(&bars[L::bQ], 0, 20000000ull);
      for (int r = r_done - 1; r >= 0 && r >= r_done - L::NS; --r)
        warp_wait_teardown(&bars[L::bRingFull + r % L::NS], (r / L::NS) & 1, 20000000ull);
      if constexpr (kInt8) {
        for (int ri = ri_done - 1; ri >= 0 && ri >= ri_done - L::NI; --ri)
          warp_wait_teardown(&bars[L::bStageFull + ri % L::NI], (ri / L::NI) & 1, 20000000ull);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (operands stay warp-uniform) and an
    // elected lane issues each tcgen05.mma and commit.  Order on the tensor
    // pipe:
    //   S0(0) S1(0) | PV0(0) S0(1) PV1(0) S1(1) | PV0(1) S0(2) PV1(1) S1(2) | ...
    // so the softmax of tile t for key tile j overlaps PV of the other query
    // tile and S of the next key tile (1024 MMA cycles).  S_t(j+1) overwrites
    // the columns P_t(j) lives in without waiting for PV_t(j): tcgen05.mma
    // operations issued by one thread execute in issue order, so PV_t(j) has
    // read P_t(j) before S_t(j+1) writes there.  A commit after S_t(j+1)
    // therefore also covers PV_t(j), which is what lets the softmax rescale
    // O_t once it sees S_t(j+1).
    bool ok = warp_wait(&bars[L::bQ], 0, ab, p.err);
    tc_fence_after();
    // Descriptors of offset 0; adding (byte offset >> 4) advances the start
    // address field (shared addresses stay below 256 KB, so it never carries).
    const uint64_t q_desc = smem_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t k_desc = smem_desc_sw128(smem_u32(sRing), 16, 1024);           // K-major (K tiles)
    const uint64_t v_desc = smem_desc_sw128(smem_u32(sRing), kPanelBytes, 1024);  // N-major (V tiles)
    auto commit = [=](int bar) {
      if (elect_one()) mma_commit(&bars[bar]);
      __syncwarp();
    };
    // A ring slot is released in both CTAs of an INT8 pair (both fill it).
    auto release = [=](int bar) {
      if (elect_one()) {
        if constexpr (kInt8)
          mma_commit_multicast(&bars[bar], 0x3);
        else
          mma_commit(&bars[bar]);
      }
      __syncwarp();
    };
    auto issue_s = [=](int t, int slot) {
      const uint32_t d = tmem + t * 128;
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t koff = (k >> 2) * kPanelBytes + (k & 3) * 32;
          const uint64_t a = q_desc + ((t * kTileBytes + koff) >> 4);
          const uint64_t b = k_desc + ((slot * kTileBytes + koff) >> 4);
          mma_ss(d, a, b, kIdescS, k > 0 ? 1u : 0u);
        }
      }
      __syncwarp();
      commit(L::bSFull + t);
    };
    auto issue_pv = [=](int t, int slot, bool accumulate) {
      const uint32_t d = tmem + 256 + t * 128;
      const uint32_t a_tm = tmem + t * 128;
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t b = v_desc + ((slot * kTileBytes + k * 2048) >> 4);
          mma_ts(d, a_tm + k * 8, b, kIdescO, (accumulate || k > 0) ? 1u : 0u);
        }
      }
      __syncwarp();

    };
    // K of key tile j sits in ring use 2j, V in ring use 2j + 1.
    if (ok && n_iter > 0) {
      ok = warp_wait(&bars[L::bRingFull + 0], 0, ab, p.err);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        release(L::bRingEmpty + 0);
      }
    }
    for (int j = 0; j < n_iter && ok; ++j) {
      const bool last = (j + 1 == n_iter);
      const int rv = 2 * j + 1, sv = rv % L::NS;
      const int rk = 2 * j + 2, sk = rk % L::NS;
      if (!warp_wait(&bars[L::bRingFull + sv], (rv / L::NS) & 1, ab, p.err) ||
          !warp_wait(&bars[L::bPFull + 0], j & 1, ab, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_pv(0, sv, j > 0);
      if (last) commit(L::bPVDone + 0);
      if (!last) {
        if (!warp_wait(&bars[L::bRingFull + sk], (rk / L::NS) & 1, ab, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(0, sk);
      }
      if (!warp_wait(&bars[L::bPFull + 1], j & 1, ab, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_pv(1, sv, j > 0);
      release(L::bRingEmpty + sv);
      if (last) {
        commit(L::bPVDone + 1);
      } else {
        issue_s(1, sk);
        release(L::bRingEmpty + sk);
      }
    }
    // Drain: all MMAs issued by this warp complete before tensor memory is freed.
    commit(L::bFinal);
    warp_wait_teardown(&bars[L::bFinal], 0, ok ? 2000000000ull : 20000000ull);
  } else if (warp < 8) {
    softmax_role(p, kt, wi, t_begin, n_iter, tmem, &bars[L::bSFull], &bars[L::bPVDone], ab,
                 [&](int t) { mbar_arrive(&bars[L::bPFull + t]); });
  } else if (warp >= 12) {
    // ------------------------------------------------------------ ring filler (INT8 cache)
    // The two CTAs of a pair work on the same head and key range (adjacent
    // query blocks) and share every dequantised tile: each CTA dequantises
    // its half (64 rows) of each int8 cache tile, x_hat = bf16(code * scale),
    // into its own ring slot, and the copy engine then moves that half into
    // the partner's slot: each filler warp copies the 16 rows of each panel it
    // wrote (2 KB shared-to-shared bulk copies that complete transactions on
    // the partner's full-barrier) as soon as it wrote them.  Current-segment bf16
    // tiles are fetched by TMA into the local ring (issued by warp 12).  Each
    // local filler warp arrives once on a slot's full-barrier (count 4), and a
    // slot is reused only after both CTAs' MMA warps released it, so neither
    // a copy nor a dequantising thread writes into a slot still being read.
    if constexpr (kInt8) {
      const int ft = threadIdx.x - 384;  // 0..127
      const int hrow = ft >> 1;          // row of this CTA's half tile (0..63)
      const int half = ft & 1;           // bf16 panel written: columns 64*half .. 64*half+63
      const int trow = 64 * static_cast<int>(rank) + hrow;  // row of the 128-row tile
      const int sw_src = hrow & 7, sw_dst = trow & 7;
      const uint32_t peer = rank ^ 1u;
      int ri = 0, r_tma = 0;
      bool ok = true;
      // This row's K and V scales of a cache tile (0 past its valid rows).
      // They are loaded one tile ahead, so the global-load latency overlaps
      // the conversion of the tile before instead of stalling it.
      const long long scale_end = static_cast<long long>(p.block_heads) * p.scale_stride;
      const auto load_scales = [&](int it_x, float& sk, float& sv) {
        sk = sv = 0.0f;
        if (it_x >= n_iter) return;
        const TileInfo tx = tile_info(t_begin + it_x, p, kt);
        if (!tx.cache || trow >= tx.valid) return;
        const long long sidx = static_cast<long long>(bh) * p.scale_stride + tx.row0 + trow;
        if (!in_bounds(sidx, 1, scale_end, p.err)) return;
        sk = p.k_scale[sidx];
        sv = p.v_scale[sidx];
      };
      float sc_next[2];
      load_scales(0, sc_next[0], sc_next[1]);
      for (int it = 0; it < n_iter && ok; ++it) {
        const TileInfo ti = tile_info(t_begin + it, p, kt);
        const float sc_tile[2] = {sc_next[0], sc_next[1]};
        load_scales(it + 1, sc_next[0], sc_next[1]);
        for (int kv = 0; kv < 2; ++kv) {
          const int r = 2 * it + kv, s = r % L::NS, u = r / L::NS;
          uint64_t* fb = &bars[L::bRingFull + s];
          if (!ti.cache) {
            if (u > 0 && !warp_wait(&bars[L::bRingEmpty + s], (u - 1) & 1, ab, p.err)) {
              ok = false;
              break;
            }
            if (lane == 0) {
              if (warp == 12) {
                mbar_expect_tx(fb, kTileBytes);
                uint8_t* dst = sRing + s * kTileBytes;
                for (int pn = 0; pn < 2; ++pn)
                  tma_load_3d(dst + pn * kPanelBytes, kv ? &tm_vcur : &tm_kcur, fb, pn * 64, head, ti.row0);
              }
              mbar_arrive(fb);
            }
            r_tma = r + 1;
            __syncwarp();
            continue;
          }
          const int si = ri % L::NI, ui = ri / L::NI;
          const float sc = sc_tile[kv];
          if (!warp_wait(&bars[L::bStageFull + si], ui & 1, ab, p.err)) {
            ok = false;
            break;
          }
          if (u > 0 && !warp_wait(&bars[L::bRingEmpty + s], (u - 1) & 1, ab, p.err)) {
            ok = false;
            break;
          }
          const uint8_t* src = sStage + si * kI8HalfBytes + hrow * 128;
          uint8_t* dst = sRing + s * kTileBytes + half * kPanelBytes + trow * 128;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int c = 4 * half + cc;  // int8 chunk: columns 16c .. 16c+15
            const uint4 w = *reinterpret_cast<const uint4*>(src + ((c ^ sw_src) << 4));
            uint32_t o[8];
            if constexpr (kFp8) {
              // E4M3 pairs -> f16 pairs (exact) -> float32, times the row scale.
              const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                    static_cast<__nv_fp8x2_storage_t>(wd[e] & 0xFFFFu), __NV_E4M3);
                const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wd[e] >> 16),
                                                                  __NV_E4M3);
                const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
                const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
                o[2 * e] = pack_bf16x2(a.x * sc, a.y * sc);
                o[2 * e + 1] = pack_bf16x2(b.x * sc, b.y * sc);
              }
            } else {
              // int8 code byte -> float via the 2^23 magic number: the biased
              // byte c + 128 in the low mantissa bits of 2^23 gives the float
              // 2^23 + 128 + c, and subtracting 2^23 + 128 leaves c exactly;
              // then one rounded multiply by the row scale.  Packed f32x2 pairs.
              const uint32_t wd[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
              const uint64_t bias2 = f2_pack(-8388736.0f, -8388736.0f);
              const uint64_t sc2 = f2_pack(sc, sc);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const uint64_t c01 = f2_add(f2_pack(__uint_as_float(__byte_perm(wd[e], 0x4B000000u, 0x7540u)),
                                                    __uint_as_float(__byte_perm(wd[e], 0x4B000000u, 0x7541u))),
                                            bias2);
                const uint64_t c23 = f2_add(f2_pack(__uint_as_float(__byte_perm(wd[e], 0x4B000000u, 0x7542u)),
                                                    __uint_as_float(__byte_perm(wd[e], 0x4B000000u, 0x7543u))),
                                            bias2);
                float f0, f1, f2, f3;
                f2_unpack(f2_mul(c01, sc2), f0, f1);
                f2_unpack(f2_mul(c23, sc2), f2, f3);
                o[2 * e] = pack_bf16x2(f0, f1);
                o[2 * e + 1] = pack_bf16x2(f2, f3);
              }
            }
            // 16 int8 columns -> 16-byte chunks 2cc and 2cc+1 of bf16 panel `half`
            *reinterpret_cast<uint4*>(dst + ((((2 * cc) ^ sw_dst)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + ((((2 * cc + 1) ^ sw_dst)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // This warp wrote rows 16 (warp - 12) .. + 15 of this CTA's half in
            // both panels (2 KB each, contiguous): copy them into the partner's
            // slot at once, and expect the partner's matching 4 KB here.  Each
            // warp raises the expected bytes before its own arrival, so the
            // phase cannot complete before all 16 KB of the partner's half land.
            mbar_expect_tx(fb, 2 * kWarpRowBytes);
            const uint32_t peer_fb = mapa_shared(smem_u32(fb), peer);
            for (int pn = 0; pn < 2; ++pn) {
              const uint8_t* rows_src =
                  sRing + s * kTileBytes + pn * kPanelBytes + (64 * rank + 16 * (warp - 12)) * 128;
              bulk_copy_to_cluster(mapa_shared(smem_u32(rows_src), peer), rows_src, kWarpRowBytes, peer_fb);
            }
            mbar_arrive(fb);
            mbar_arrive(&bars[L::bStageEmpty + si]);
          }
          ++ri;
        }
      }
      if (!ok && warp == 12) {
        // Abort: give the current-tile copies this warp issued time to land.
        for (int r = r_tma - 1; r >= 0 && r >= r_tma - L::NS; --r) {
          const TileInfo ti = tile_info(t_begin + r / 2, p, kt);
          if (ti.cache) continue;
          warp_wait_teardown(&bars[L::bRingFull + r % L::NS], (r / L::NS) & 1, 20000000ull);
        }
      }
      if (warp == 12) {
        // Both MMA warps release every slot in both CTAs: wait until the last
        // release of each slot has arrived here, so no release is still in
        // flight toward this CTA when the pair meets at the final barrier.
        const int uses = 2 * n_iter;
        for (int sl = 0; sl < L::NS && sl < uses; ++sl) {
          const int n_s = (uses - sl + L::NS - 1) / L::NS;
          warp_wait_teardown(&bars[L::bRingEmpty + sl], (n_s - 1) & 1, ok ? 2000000000ull : 20000000ull);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // INT8: neither CTA of a pair leaves while the other may still write into
  // its shared memory or arrive on its barriers.
  if constexpr (kInt8) cluster_sync();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Combine the pieces of every split unit in piece order: O = sum_s w_s O_s /
// sum_s w_s, w_s = exp(lse_s - max lse), LSE = max + log(sum w_s).  One warp
// per (split unit, CTA of the unit, query row).
__global__ void __launch_bounds__(256) combine_kernel(const AttnParams p, int n_split_units, int ctas) {
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= static_cast<long long>(n_split_units) * ctas * 256) return;
  const int r = static_cast<int>(gw & 255);
  const int c = static_cast<int>((gw >> 8) % ctas);
  const int su = static_cast<int>((gw >> 8) / ctas);
  const int unit = p.n_full + su;
  const int head = unit / p.units_per_head;
  const int ublk = unit - head * p.units_per_head;
  const int grow = (ctas == 2 ? 2 * ublk + c : ublk) * 256 + r;
  if (grow >= p.nq) return;
  const int S = p.tail_splits;
  auto prow = [&](int s) { return ((static_cast<size_t>(su) * S + s) * ctas + c) * 256 + r; };
  if (!in_bounds(static_cast<long long>(prow(S - 1)), 1, p.ws_rows, p.err) ||
      !in_bounds((static_cast<long long>(grow) * p.heads + head) * 128, 128, static_cast<long long>(p.nq) * p.heads * 128,
                 p.err))
    return;
  float mx = -INFINITY;
  for (int s = 0; s < S; ++s) mx = fmaxf(mx, p.ws_lse[prow(s)]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.0f;
  for (int s = 0; s < S; ++s) {
    const size_t row = prow(s);
    const float w = expf(p.ws_lse[row] - mx);
    const float4 o = *reinterpret_cast<const float4*>(p.ws_o + row * 128 + 4 * lane);
    acc.x += w * o.x;
    acc.y += w * o.y;
    acc.z += w * o.z;
    acc.w += w * o.w;
    wsum += w;
  }
  const float inv = 1.0f / wsum;
  uint2 pk;
  pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(grow) * p.heads + head) * 128 + 4 * lane) = pk;
  if (p.lse && lane == 0) p.lse[static_cast<size_t>(head) * p.nq + grow] = mx + logf(wsum);
}

template <bool kInt8, bool kFp8>
static cudaError_t configure(int dev) {
  using L = Layout<kInt8>;
  static int configured[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(segment_attn_kernel<kInt8, kFp8>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return cudaSuccess;
}

template <bool kInt8, bool kFp8>
static cudaError_t launch_impl(const AttnTensorMaps& tm, const AttnParams& p, int n_items, cudaStream_t stream) {
  using L = Layout<kInt8>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure<kInt8, kFp8>(dev);
  if (e != cudaSuccess) return e;
  if constexpr (kInt8) {
    // CTA pairs (clusters of two adjacent query blocks) share the dequantised
    // tiles; the second block of a pair may lie past the end (no live rows).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2u * static_cast<unsigned>(n_items), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, segment_attn_kernel<kInt8, kFp8>, tm.q, tm.kcur, tm.vcur, tm.kc, tm.vc, p);
    if (e != cudaSuccess) return e;
  } else {
    segment_attn_kernel<kInt8, kFp8><<<static_cast<unsigned>(n_items), kThreads, L::kAlloc, stream>>>(
        tm.q, tm.kcur, tm.vcur, tm.kc, tm.vc, p);
  }
  return cudaGetLastError();
}

// Co-resident work items: one CTA per SM (BF16), or the number of clusters of
// two CTAs that fit at once (one-byte caches).
template <bool kInt8, bool kFp8>
static int concurrent_items() {
  using L = Layout<kInt8>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cached[64] = {0};
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 0;
  int n = sms;
  if constexpr (kInt8) {
    n = sms / 2;
    if (configure<kInt8, kFp8>(dev) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2u * static_cast<unsigned>(sms), 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = L::kAlloc;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, segment_attn_kernel<kInt8, kFp8>, &cfg) == cudaSuccess &&
          clusters > 0)
        n = clusters;
      else
        (void)cudaGetLastError();
    }
  }
  cached[dev] = n;
  return n;
}

}  // namespace attn

cudaError_t launch_segment_attn(int kind, const AttnTensorMaps& tm, const AttnParams& p, int n_items,
                                cudaStream_t stream) {
  if (kind == kCacheInt8) return attn::launch_impl<true, false>(tm, p, n_items, stream);
  if (kind == kCacheFp8) return attn::launch_impl<true, true>(tm, p, n_items, stream);
  if (kind == kCacheBF16) return attn::launch_impl<false, false>(tm, p, n_items, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_combine(const AttnParams& p, int units, int ctas_per_unit, cudaStream_t stream) {
  const int n_split_units = units - p.n_full;
  if (p.tail_splits <= 1 || n_split_units <= 0) return cudaSuccess;
  const long long warps = static_cast<long long>(n_split_units) * ctas_per_unit * 256;
  const long long blocks = (warps * 32 + 255) / 256;
  attn::combine_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p, n_split_units, ctas_per_unit);
  return cudaGetLastError();
}

int attn_concurrent_items(int kind) {
  if (kind == kCacheInt8) return attn::concurrent_items<true, false>();
  if (kind == kCacheFp8) return attn::concurrent_items<true, true>();
  return attn::concurrent_items<false, false>();
}

int attn_smem_bytes(bool int8_cache) {
  return int8_cache ? attn::Layout<true>::kAlloc : attn::Layout<false>::kAlloc;
}

}  // namespace nomas
