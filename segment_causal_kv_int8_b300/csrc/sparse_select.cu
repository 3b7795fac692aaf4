// sparse_select.cu - choose the cache key tiles of block-sparse segment
// attention.
//
// The single-GPU preset's backend list mentions a sparse attention mode that
// attends to a quarter of the candidate video key blocks after two dense
// denoising steps (Hy-Nomas auf einer RTX 4090, section "Das
// Single-GPU-Preset").  The selection rule is not given; the reading used
// here: for head h and query group g (512 rows) the score of cache key tile t
// (128 resident slots) is mean_query(g) . mean_key(t), and the ceil(keep * T)
// highest scores are kept (ties: lower tile first), listed in increasing
// tile order.
//
// Two HBM-bound kernels.  tile_means_kernel reads the resident cache K once
// (16-byte coalesced loads, INT8 or FP8 codes dequantised with their row
// scale) and writes the float32 mean key of every (head, tile); the means
// depend only on the cache, so callers may keep them across the denoising
// steps of a turn.  select_kernel, one CTA per (query group, head), streams
// the group's queries and then the head's mean keys through a per-thread
// cp.async ring in shared memory, scores every tile, selects the k best by a
// radix selection on the scores' bits and writes the kept list in tile order
// with block-wide prefix counts.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "checks.cuh"
#include "kernels.h"

namespace nomas {
namespace {

constexpr int kSelThreads = 256;

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& w) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    acc[2 * e] += __uint_as_float(v[e] << 16);
    acc[2 * e + 1] += __uint_as_float(v[e] & 0xFFFF0000u);
  }
}

// One CTA per (tile, head).  BF16: 16 lanes cover a 256-byte key row, so the
// 256 threads take 16 rows at a time (8 passes for a full tile).  INT8: 8
// lanes cover a 128-byte row, 32 rows at a time (4 passes); each code is
// multiplied by its row scale before it is summed.  Every pass's loads are
// issued before any is summed.  Partial sums (one per row lane) are added in
// a fixed order in shared memory.
template <int K>
__global__ void __launch_bounds__(kSelThreads) tile_means_kernel(const SparseSelectParams p) {
  constexpr bool kCodes = K != kCacheBF16;        // one-byte codes (INT8 or FP8) with row scales
  constexpr int kLanesPerRow = kCodes ? 8 : 16;   // 16-byte vectors per row
  constexpr int kDims = 128 / kLanesPerRow;       // dims per thread
  constexpr int kRowSlots = kSelThreads / kLanesPerRow;
  constexpr int kPasses = 128 / kRowSlots;
  __shared__ float part[kRowSlots][129];
  const int t = blockIdx.x, h = blockIdx.y;
  const int c = threadIdx.x % kLanesPerRow, rs = threadIdx.x / kLanesPerRow;
  const long long plane = static_cast<long long>(p.block_head_base + h) * p.cap_slots;
  const int r0 = t * 128, n = min(128, p.nc - r0);
  uint4 w[kPasses];
  float sc[kPasses];
#pragma unroll
  for (int pass = 0; pass < kPasses; ++pass) {
    const int r = pass * kRowSlots + rs;
    w[pass] = make_uint4(0u, 0u, 0u, 0u);
    sc[pass] = 0.0f;
    if (r < n && in_bounds(plane + r0 + r, 1, p.cache_rows, p.err)) {
      const long long row = plane + r0 + r;
      if constexpr (kCodes) {
        w[pass] = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.kcache) + row * 128)[c];
        sc[pass] = p.kscale[row];
      } else {
        w[pass] = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.kcache) + row * 128)[c];
      }
    }
  }
  float acc[kDims];
#pragma unroll
  for (int e = 0; e < kDims; ++e) acc[e] = 0.0f;
#pragma unroll
  for (int pass = 0; pass < kPasses; ++pass) {
    // rows past the tile's end hold zero codes and a zero scale: they add 0
    if constexpr (K == kCacheInt8) {
      // The biased byte c + 128 in the low mantissa bits of 2^23 gives the
      // float 2^23 + 128 + c; subtracting 2^23 + 128 leaves the code exactly.
      const uint32_t v[4] = {w[pass].x ^ 0x80808080u, w[pass].y ^ 0x80808080u, w[pass].z ^ 0x80808080u,
                             w[pass].w ^ 0x80808080u};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float code = __fadd_rn(__uint_as_float(__byte_perm(v[e >> 2], 0x4B000000u, 0x7540u + (e & 3))),
                                     -8388736.0f);
        acc[e] = fmaf(code, sc[pass], acc[e]);
      }
    } else if constexpr (K == kCacheFp8) {
      const uint32_t v[4] = {w[pass].x, w[pass].y, w[pass].z, w[pass].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(
            static_cast<__nv_fp8x2_storage_t>((v[e >> 1] >> (16 * (e & 1))) & 0xFFFFu), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
        acc[2 * e] = fmaf(f.x, sc[pass], acc[2 * e]);
        acc[2 * e + 1] = fmaf(f.y, sc[pass], acc[2 * e + 1]);
      }
    } else {
      add_bf16x8(acc, w[pass]);
    }
  }
#pragma unroll
  for (int e = 0; e < kDims; ++e) part[rs][c * kDims + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < 128) {
    float s = 0.0f;
    for (int i = 0; i < kRowSlots; ++i) s += part[i][threadIdx.x];
    const long long idx = (static_cast<long long>(h) * p.n_tiles + t) * 128 + threadIdx.x;
    if (in_bounds(idx, 1, static_cast<long long>(p.heads) * p.n_tiles * 128, p.err)) p.kbar[idx] = s / static_cast<float>(n);
  }
}

// One CTA of 512 threads per (query group, head).
constexpr int kPickThreads = 512;
// Every global read of select_kernel goes through one per-thread ring of
// cp.async copies: thread i copies into slot i of a stage and reads back only
// that slot, so no barrier guards the ring.  Items 0 .. 7 are the group's
// query rows (rows rs + 64 i and rs + 64 i + 32, 16 bytes of each per
// thread), the items after them the mean keys of 32 tiles each (32 bytes per
// thread).  Items are requested kPickStages - 1 ahead: the slot refilled is
// the one the thread read in the step before, and the first mean keys are
// requested while the last query rows are still being summed.
constexpr int kPickStages = 4;
constexpr int kPickSlotBytes = 32;
constexpr int kPickQItems = 512 / 64;  // query items: two rows per thread each
constexpr int kPickStageBytes = kPickThreads * kPickSlotBytes;
constexpr int kPickRingBytes = kPickStages * kPickStageBytes;

__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// At most kPickStages - 1 copy groups pending: the current item has landed.
__device__ __forceinline__ void cp_async_wait_ring() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kPickStages - 1) : "memory");
}

__global__ void __launch_bounds__(kPickThreads, 2) select_kernel(const SparseSelectParams p) {
  // Dynamic shared memory: the copy ring, then the partial query sums
  // [32][129], later (after a barrier) the scores [n_tiles], turned into
  // selection keys in place.
  extern __shared__ __align__(16) uint8_t s_raw[];
  float(*part)[129] = reinterpret_cast<float(*)[129]>(s_raw + kPickRingBytes);
  float* s_scores = reinterpret_cast<float*>(s_raw + kPickRingBytes);
  __shared__ float s_q[128];
  __shared__ int s_warp[kPickThreads / 32];
  const int g = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t slot0 = static_cast<uint32_t>(__cvta_generic_to_shared(s_raw)) + kPickSlotBytes * threadIdx.x;
  const uint8_t* my_slot = s_raw + kPickSlotBytes * threadIdx.x;

  // Query rows: 16 lanes per 256-byte row slice (c), 64 rows per item (rs, rs + 32).
  // Mean keys: 16 lanes per tile (c: dims 8 c .. 8 c + 7), 32 tiles per item (rs).
  const int c = threadIdx.x & 15, rs = threadIdx.x >> 4;
  const int r0 = g * 512, n = min(512, p.nq - r0);
  const char* qrow = reinterpret_cast<const char*>(p.q) + ((static_cast<long long>(r0) * p.heads + h) * 128 + 8 * c) * 2;
  const long long q_row_bytes = static_cast<long long>(p.heads) * 256;
  const float* kb_lane = p.kbar + static_cast<size_t>(h) * p.n_tiles * 128 + 8 * c;
  const int n_items = kPickQItems + (p.n_tiles + 31) / 32;
  const auto issue = [&](int it) {
    const uint32_t dst = slot0 + (it % kPickStages) * kPickStageBytes;
    if (it < kPickQItems) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int r = rs + 64 * it + 32 * u;
        if (r < n && in_bounds((static_cast<long long>(r0 + r) * p.heads + h) * 128 + 8 * c, 8,
                               static_cast<long long>(p.nq) * p.heads * 128, p.err))
          cp_async16(dst + 16 * u, qrow + r * q_row_bytes);
      }
    } else if (it < n_items) {
      const int t = 32 * (it - kPickQItems) + rs;
      if (t < p.n_tiles && in_bounds((static_cast<long long>(h) * p.n_tiles + t) * 128 + 8 * c, 8,
                                     static_cast<long long>(p.heads) * p.n_tiles * 128, p.err)) {
        const float* src = kb_lane + static_cast<size_t>(t) * 128;
        cp_async16(dst, src);
        cp_async16(dst + 16, src + 4);
      }
    }
    cp_async_commit();  // one group per item, empty or not, so the group count stays uniform
  };
  for (int it = 0; it < kPickStages - 1; ++it) issue(it);

  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
  float qd[8];  // this lane's eight dims of the mean query
  for (int it = 0; it < n_items; ++it) {
    issue(it + kPickStages - 1);
    cp_async_wait_ring();  // this thread's copies of item `it` have landed
    const uint8_t* slot = my_slot + (it % kPickStages) * kPickStageBytes;
    if (it < kPickQItems) {
      // rows in increasing order, as one row per step would add them
      if (rs + 64 * it < n) add_bf16x8(acc, *reinterpret_cast<const uint4*>(slot));
      if (rs + 64 * it + 32 < n) add_bf16x8(acc, *reinterpret_cast<const uint4*>(slot + 16));
      if (it == kPickQItems - 1) {
        // Mean query of the group, partial sums added in a fixed order.
#pragma unroll
        for (int e = 0; e < 8; ++e) part[rs][c * 8 + e] = acc[e];
        __syncthreads();
        if (threadIdx.x < 128) {
          float sum = 0.0f;
          for (int i = 0; i < 32; ++i) sum += part[i][threadIdx.x];
          s_q[threadIdx.x] = sum / static_cast<float>(n);
        }
        __syncthreads();  // part is dead from here on: the scores reuse its memory
#pragma unroll
        for (int e = 0; e < 8; ++e) qd[e] = s_q[8 * c + e];
      }
      continue;
    }
    const int t = 32 * (it - kPickQItems) + rs;
    const float4 k0 = *reinterpret_cast<const float4*>(slot);
    const float4 k1 = *reinterpret_cast<const float4*>(slot + 16);
    float a = qd[0] * k0.x;
    a = fmaf(qd[1], k0.y, a);
    a = fmaf(qd[2], k0.z, a);
    a = fmaf(qd[3], k0.w, a);
    a = fmaf(qd[4], k1.x, a);
    a = fmaf(qd[5], k1.y, a);
    a = fmaf(qd[6], k1.z, a);
    a = fmaf(qd[7], k1.w, a);
    // the 16 lanes of a tile sit in one half of the warp
    a += __shfl_xor_sync(0xffffffffu, a, 8);
    a += __shfl_xor_sync(0xffffffffu, a, 4);
    a += __shfl_xor_sync(0xffffffffu, a, 2);
    a += __shfl_xor_sync(0xffffffffu, a, 1);
    if (t < p.n_tiles && c == 0) s_scores[t] = a;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // Top-k by radix selection.  Scores become order-preserving 32-bit keys
  // (-0 folded into +0 first, so equal scores give equal keys); four 8-bit
  // passes, most significant first, histogram the keys that match the prefix
  // found so far and pick the digit where the count of larger keys reaches
  // k.  That leaves the k-th largest key K and how many tiles equal to K are
  // kept (`need`): every key > K, and the first `need` keys == K in tile
  // order (ties to the lower tile).  Linear in the tile count.
  uint32_t* s_keys = reinterpret_cast<uint32_t*>(s_scores);
  for (int t = threadIdx.x; t < p.n_tiles; t += kPickThreads) {
    const uint32_t u = __float_as_uint(s_scores[t] + 0.0f);
    s_keys[t] = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  __shared__ uint32_t s_hist[256];
  __shared__ uint32_t s_sel[2];  // prefix of K found so far, tiles still to take among the matching ones
  uint32_t prefix = 0u, mask = 0u;
  int need = p.keep;
  const bool keep_all = p.keep >= p.n_tiles;
  if (!keep_all) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (threadIdx.x < 256) s_hist[threadIdx.x] = 0u;
      __syncthreads();
      for (int t = threadIdx.x; t < p.n_tiles; t += kPickThreads) {
        const uint32_t key = s_keys[t];
        if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // Lane l holds digits 255 - 8 l .. 248 - 8 l (descending).
        uint32_t c[8], lane_sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = s_hist[255 - 8 * lane - i];
          lane_sum += c[i];
        }
        uint32_t incl = lane_sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += y;
        }
        uint32_t above = incl - lane_sum;  // matching keys with a larger digit than this lane's
        if (above < static_cast<uint32_t>(need) && static_cast<uint32_t>(need) <= incl) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (above + c[i] >= static_cast<uint32_t>(need)) {
              s_sel[0] = prefix | (static_cast<uint32_t>(255 - 8 * lane - i) << shift);
              s_sel[1] = static_cast<uint32_t>(need) - above;
              break;
            }
            above += c[i];
          }
        }
      }
      __syncthreads();
      prefix = s_sel[0];
      need = static_cast<int>(s_sel[1]);
      mask |= 255u << shift;
    }
  }

  // Kept tiles in increasing order: a tile is kept if its key exceeds K, or
  // equals K and fewer than `need` tiles equal to K come before it; its
  // position is the number of kept tiles before it (two block-wide prefix
  // counts per pass of 512 tiles).
  const size_t hg = static_cast<size_t>(h) * p.n_groups + g;
  int* out = p.tiles + hg * p.max_keep;
  int base = 0, base_eq = 0;
  for (int t0 = 0; t0 < p.n_tiles; t0 += kPickThreads) {
    const int t = t0 + threadIdx.x;
    const bool live = t < p.n_tiles;
    const uint32_t key = live ? s_keys[t] : 0u;
    const bool eq = live && !keep_all && key == prefix;
    const unsigned bal_eq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) s_warp[warp] = __popc(bal_eq);
    __syncthreads();
    int eq_before = base_eq;
    for (int w = 0; w < warp; ++w) eq_before += s_warp[w];
    eq_before += __popc(bal_eq & ((1u << lane) - 1u));
    for (int w = 0; w < kPickThreads / 32; ++w) base_eq += s_warp[w];
    __syncthreads();
    const bool k = live && (keep_all || key > prefix || (eq && eq_before < need));
    const unsigned bal = __ballot_sync(0xffffffffu, k);
    if (lane == 0) s_warp[warp] = __popc(bal);
    __syncthreads();
    int before = base;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    before += __popc(bal & ((1u << lane) - 1u));
    if (k && before < p.keep && in_bounds(static_cast<long long>(hg) * p.max_keep + before, 1,
                                          static_cast<long long>(p.heads) * p.n_groups * p.max_keep, p.err))
      out[before] = t;
    for (int w = 0; w < kPickThreads / 32; ++w) base += s_warp[w];
    __syncthreads();
  }
  if (threadIdx.x == 0) p.counts[hg] = min(base, p.keep);
}

}  // namespace

size_t sparse_select_smem(int n_tiles) {
  const size_t need = static_cast<size_t>(n_tiles) * 4, part = 32 * 129 * sizeof(float);
  return kPickRingBytes + (((need > part ? need : part) + 15) & ~size_t(15));
}

cudaError_t launch_sparse_select(int kind, bool reuse_key_means, const SparseSelectParams& p,
                                 cudaStream_t stream) {
  if (p.n_tiles > 0 && !reuse_key_means) {
    const dim3 tg(p.n_tiles, p.heads);
    if (kind == kCacheInt8)
      tile_means_kernel<kCacheInt8><<<tg, kSelThreads, 0, stream>>>(p);
    else if (kind == kCacheFp8)
      tile_means_kernel<kCacheFp8><<<tg, kSelThreads, 0, stream>>>(p);
    else
      tile_means_kernel<kCacheBF16><<<tg, kSelThreads, 0, stream>>>(p);
  }
  // The shared-memory limit is raised once per device, to what the largest
  // tile count the entry point accepts (8192) needs.
  static int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(sparse_select_smem(8192)));
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  const size_t smem = sparse_select_smem(p.n_tiles);
  const dim3 gg(p.n_groups, p.heads);
  select_kernel<<<gg, kPickThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nomas
