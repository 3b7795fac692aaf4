// kvcache_append.cu - write a finished segment's K/V into the ring cache
// (INT8 with per-(block, head, token) absmax scales, or a BF16 copy), and the
// zero-fill kernel behind a memory-clearing reset.
//
// The low-memory preset stores the KV cache in INT8 and keeps a window of 18
// latent frames on the GPU (Hy-Nomas auf einer RTX 4090, section "Das
// Single-GPU-Preset"); after each segment its keys and values are written to
// the cache (the "Schreiben des KV-Cache" stage, section "Zeiten").
//
// One row = the head_dim = 128 values of one (tensor, block, head, token).
// Bf16 input (append8_kernel): 8 lanes own a row (16 values each, two 16-byte
// loads), reduce the absmax with three shuffles and write 16 code bytes each
// plus the row's scale; a CTA takes 64 consecutive (token, head) rows, one
// contiguous 16 KB range of the input.  Float32 input (append_kernel): 16
// lanes per row, a CTA per two tokens and 16 heads.  Large appends stream
// through shared memory instead (append_staged_kernel).  A row's token, head
// and frame come from multiply-shift division by run-time constants.
//
// Codec bits (identical to the reference definition): scale = fl32(m / 127),
// inv = fl32(127 / m) (IEEE round-to-nearest divisions), code =
// rint(fl32(x * inv)) (ties to even), which lies in [-127, 127].  The rounding
// adds 1.5 * 2^23 to the product and takes the code's byte from the sum's
// bits.  When inv overflows (absmax below 127 / FLT_MAX) the products are
// +-inf or NaN (0 * inf): that row takes a float->int conversion instead,
// with NaN -> 0 and +-inf clamped to +-127.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "checks.cuh"
#include "kernels.h"
#include "rope_math.cuh"
#include "sm100.cuh"

namespace nomas {
namespace {

template <bool kF32In>
__device__ __forceinline__ void load8(const void* base, long long off, float (&x)[8]) {
  if constexpr (kF32In) {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + off + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(u[e] << 16);
      x[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
    }
  }
}

// E4M3 codes of fl32(x[i] * inv), four per word with x[4q] in the low byte.
// The conversion rounds to nearest (ties to even) and saturates at +-448; when
// inv overflowed (finite_inv false) a NaN product (0 * inf) is coded 0.
template <int N>
__device__ __forceinline__ void fp8_encode(const float (&x)[N], float inv, bool finite_inv, uint32_t (&out)[N / 4]) {
#pragma unroll
  for (int q = 0; q < N / 4; ++q) {
    float y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = __fmul_rn(x[4 * q + e], inv);
    if (!finite_inv) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (isnan(y[e])) y[e] = 0.0f;
    }
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(y[0], y[1]), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(y[2], y[3]), __NV_SATFINITE, __NV_E4M3);
    out[q] = (lo & 0xFFFFu) | (hi << 16);
  }
}

// Quantise (or copy) one row from 8 values per lane of a 16-lane group and
// write it to its ring slot.  K: kCacheBF16, kCacheInt8 or kCacheFp8.
template <int K>
__device__ __forceinline__ void write_row(const AppendParams& p, int tensor, long long dst_row, const float (&x)[8],
                                          int g, unsigned gmask) {
  if (!in_bounds(dst_row, 1, p.cache_rows, p.err)) return;  // uniform over the lane group
  if constexpr (K != kCacheBF16) {
    constexpr float kQMax = K == kCacheInt8 ? 127.0f : 448.0f;
    float m = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(x[e]));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(gmask, m, off));
    const float scale = __fdiv_rn(m, kQMax);
    const float inv = __fdiv_rn(kQMax, m);
    uint32_t lo, hi;
    if constexpr (K == kCacheFp8) {
      uint32_t c[2];
      fp8_encode<8>(x, inv, inv <= 3.0e38f, c);
      lo = c[0];
      hi = c[1];
    } else if (inv <= 3.0e38f) {
      // |fl32(x * inv)| <= 127: adding 1.5 * 2^23 rounds it to an integer
      // (nearest, ties to even) held in the low mantissa bits, whose low byte
      // is the two's-complement code.
      uint32_t b[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) b[e] = __float_as_uint(__fadd_rn(__fmul_rn(x[e], inv), 12582912.0f));
      lo = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
      hi = __byte_perm(__byte_perm(b[4], b[5], 0x0040), __byte_perm(b[6], b[7], 0x0040), 0x5410);
    } else {
      // inv overflowed (absmax below 127 / FLT_MAX): +-inf products clamp to
      // +-127 and NaN (0 * inf) converts to 0.
      lo = hi = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int c = __float2int_rn(__fmul_rn(x[e], inv));
        c = max(-127, min(127, c));
        const uint32_t byte = static_cast<uint32_t>(c) & 0xFFu;
        if (e < 4)
          lo |= byte << (8 * e);
        else
          hi |= byte << (8 * (e - 4));
      }
    }

    int8_t* dst = static_cast<int8_t*>(tensor ? p.cv : p.ck) + dst_row * 128 + 8 * g;
    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
    if (g == 0) (tensor ? p.vs : p.ks)[dst_row] = scale;
  } else {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(tensor ? p.cv : p.ck) + dst_row * 128 + 8 * g;
    uint4 w;
    uint32_t* u = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 t = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
      u[e] = *reinterpret_cast<const uint32_t*>(&t);
    }
    *reinterpret_cast<uint4*>(dst) = w;
  }
}

// Quantise (or round to bf16) one row from 16 values per lane of an 8-lane
// group and write it to its ring slot.
template <int K>
__device__ __forceinline__ void store_row16(const AppendParams& p, int tensor, long long dst_row, const float (&x)[16],
                                            int g, unsigned gmask) {
  if (!in_bounds(dst_row, 1, p.cache_rows, p.err)) return;  // uniform over the lane group
  if constexpr (K != kCacheBF16) {
    constexpr float kQMax = K == kCacheInt8 ? 127.0f : 448.0f;
    float m0 = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    float m1 = fmaxf(fmaxf(fabsf(x[4]), fabsf(x[5])), fmaxf(fabsf(x[6]), fabsf(x[7])));
    float m2 = fmaxf(fmaxf(fabsf(x[8]), fabsf(x[9])), fmaxf(fabsf(x[10]), fabsf(x[11])));
    float m3 = fmaxf(fmaxf(fabsf(x[12]), fabsf(x[13])), fmaxf(fabsf(x[14]), fabsf(x[15])));
    float m = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(gmask, m, off));
    const float scale = __fdiv_rn(m, kQMax);
    const float inv = __fdiv_rn(kQMax, m);
    uint32_t c[4];
    if constexpr (K == kCacheFp8) {
      fp8_encode<16>(x, inv, inv <= 3.0e38f, c);
    } else if (inv <= 3.0e38f) {
      // rint(fl32(x * inv)) in [-127, 127]: adding 1.5 * 2^23 rounds to an
      // integer (ties to even) whose low byte is the two's-complement code.
      // The product is rounded on its own (the packed multiply) and the add
      // is a separate scalar __fadd_rn: a packed add right after the packed
      // multiply is contracted into a fused multiply-add, which skips the
      // product's rounding and can move a tie to the other code.
      const uint64_t inv2 = f2_pack(inv, inv);
      uint32_t bb[16];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float y0, y1;
        f2_unpack(f2_mul(f2_pack(x[2 * e], x[2 * e + 1]), inv2), y0, y1);
        bb[2 * e] = __float_as_uint(__fadd_rn(y0, 12582912.0f));
        bb[2 * e + 1] = __float_as_uint(__fadd_rn(y1, 12582912.0f));
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        c[q] = __byte_perm(__byte_perm(bb[4 * q], bb[4 * q + 1], 0x0040), __byte_perm(bb[4 * q + 2], bb[4 * q + 3], 0x0040),
                           0x5410);
    } else {
      // inv overflowed (absmax below 127 / FLT_MAX): +-inf products clamp to
      // +-127 and NaN (0 * inf) converts to 0.
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        c[q] = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          int ci = __float2int_rn(__fmul_rn(x[4 * q + e], inv));
          ci = max(-127, min(127, ci));
          c[q] |= (static_cast<uint32_t>(ci) & 0xFFu) << (8 * e);
        }
      }
    }
    int8_t* dst = static_cast<int8_t*>(tensor ? p.cv : p.ck) + dst_row * 128 + 16 * g;
    *reinterpret_cast<uint4*>(dst) = make_uint4(c[0], c[1], c[2], c[3]);
    if (g == 0) (tensor ? p.vs : p.ks)[dst_row] = scale;
  } else {
    uint4 o[2];
    uint32_t* u = reinterpret_cast<uint32_t*>(o);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      __nv_bfloat162 t = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
      u[e] = *reinterpret_cast<const uint32_t*>(&t);
    }
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(tensor ? p.cv : p.ck) + dst_row * 128 + 16 * g);
    dst[0] = o[0];
    dst[1] = o[1];
  }
}

constexpr int kAppendTokens = 2;  // tokens per block (and rows per 16-lane group)

// Grid: x = groups of kAppendTokens tokens, y = groups of 16 heads, z = (block,
// tensor).  16 lanes own one (token, head) row, 8 values each; the 16 row
// groups of a CTA are 16 consecutive heads, so a CTA reads whole token rows
// ([heads][128] contiguous in the input) and writes, per head, kAppendTokens
// consecutive ring slots.  Each lane group issues all its loads before any
// arithmetic.
// Many small CTAs (eight per SM for bf16 input) keep enough rows in flight.
template <bool kF32In, int K>
__global__ void __launch_bounds__(256, kF32In ? 4 : 8) append_kernel(const __grid_constant__ AppendParams p) {
  const int h = blockIdx.y * 16 + (threadIdx.x >> 4);
  if (h >= p.heads) return;  // whole 16-lane groups leave together
  const int g = threadIdx.x & 15;
  const unsigned gmask = 0xFFFFu << (threadIdx.x & 16);
  const int tensor = blockIdx.z & 1;
  const int b = blockIdx.z >> 1;
  const int n0 = blockIdx.x * kAppendTokens;
  const void* src = tensor ? p.v : p.k;
  const long long plane = static_cast<long long>(b) * p.heads + h;  // cache [block][head] plane
  float x[kAppendTokens][8];
#pragma unroll
  for (int r = 0; r < kAppendTokens; ++r) {
    const int n = n0 + r;
    if (n < p.n_tokens) {
      const long long src_tok = static_cast<long long>(p.first_frame) * p.tpf + n;
      const long long off = b * p.block_stride + (src_tok * p.heads + h) * 128 + 8 * g;
      if (in_bounds(off, 8, p.src_extent, p.err))
        load8<kF32In>(src, off, x[r]);
      else
#pragma unroll
        for (int e = 0; e < 8; ++e) x[r][e] = 0.0f;
    }
  }
#pragma unroll
  for (int r = 0; r < kAppendTokens; ++r) {
    const int n = n0 + r;
    if (n >= p.n_tokens) break;
    const int f = fast_div(n, p.tpf_div);  // written frames never exceed the ring, so one wrap at most
    int slot_frame = p.base_slot_frame + f;
    if (slot_frame >= p.capacity_frames) slot_frame -= p.capacity_frames;
    const long long dst_row = plane * p.cap_slots + static_cast<long long>(slot_frame) * p.tpf + (n - f * p.tpf);
    write_row<K>(p, tensor, dst_row, x[r], g, gmask);
  }
}

// Direct append for bf16 input: 8 lanes own a row (16 values each, two
// 16-byte loads), so the per-row reduction and the two divisions are shared by
// twice as many values.  A CTA takes 64 consecutive (token, head) rows of the
// input, one contiguous 16 KB range, two rows per 8-lane group (both loads of
// both rows issued first).  Grid: x = groups of 64 rows, z = (block, tensor).
// A BF16 cache takes the bf16 values unchanged (a copy).
constexpr int kAppend8Rows = 64;

template <int K>
__global__ void __launch_bounds__(256, K != kCacheBF16 ? 5 : 8) append8_kernel(const __grid_constant__ AppendParams p) {
  const int g = threadIdx.x & 7;
  const unsigned gmask = 0xFFu << (threadIdx.x & 24);
  const int tensor = blockIdx.z & 1;
  const int b = blockIdx.z >> 1;
  // rows = n_tokens * heads < 2^31 (checked by the launcher)
  const int rows = p.n_tokens * p.heads;
  const int r0 = static_cast<int>(blockIdx.x) * kAppend8Rows;
  const long long src0 = b * p.block_stride + static_cast<long long>(p.first_frame) * p.tpf * p.heads * 128;
  const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(tensor ? p.v : p.k);
  uint4 w[2][2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = r0 + (threadIdx.x >> 3) + 32 * r;
    if (row < rows) {
      const long long off = src0 + static_cast<long long>(row) * 128 + 16 * g;
      if (in_bounds(off, 16, p.src_extent, p.err)) {
        const uint4* q = reinterpret_cast<const uint4*>(src + off);
        w[r][0] = q[0];
        w[r][1] = q[1];
      } else {
        w[r][0] = w[r][1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = r0 + (threadIdx.x >> 3) + 32 * r;
    if (row >= rows) break;  // rows of one 8-lane group: uniform
    const int n = fast_div(row, p.heads_div);
    const int h = row - n * p.heads;
    const int f = fast_div(n, p.tpf_div);  // written frames never exceed the ring, so one wrap at most
    int slot_frame = p.base_slot_frame + f;
    if (slot_frame >= p.capacity_frames) slot_frame -= p.capacity_frames;
    const long long dst_row = (static_cast<long long>(b) * p.heads + h) * p.cap_slots +
                              static_cast<long long>(slot_frame) * p.tpf + (n - f * p.tpf);
    if constexpr (K != kCacheBF16) {
      const uint32_t u[8] = {w[r][0].x, w[r][0].y, w[r][0].z, w[r][0].w, w[r][1].x, w[r][1].y, w[r][1].z, w[r][1].w};
      float x[16];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        x[2 * e] = __uint_as_float(u[e] << 16);
        x[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
      }
      store_row16<K>(p, tensor, dst_row, x, g, gmask);
    } else if (in_bounds(dst_row, 1, p.cache_rows, p.err)) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(tensor ? p.cv : p.ck) + dst_row * 128 + 16 * g);
      dst[0] = w[r][0];
      dst[1] = w[r][1];
    }
  }
}

// Staged append: persistent CTAs stream the input through shared memory.
// The input of one (block, tensor) is [tokens][heads][128] with whole token
// rows contiguous, so a chunk of chunk_tokens tokens is one contiguous range;
// warp 8 bulk-loads chunks (copy engine) into a kStages-deep ring, warps 0-7
// (16 groups of 16 lanes, one row per group at a time) convert them from
// shared memory and write codes and scales.  Chunks go round-robin to CTAs.
constexpr int kStages = 3;
constexpr int kStagedThreads = 288;      // 8 consumer warps + 1 producer warp
constexpr int kStageBytes = 32 * 1024;   // largest chunk

template <bool kF32In, int K>
__global__ void __launch_bounds__(kStagedThreads, 2) append_staged_kernel(const __grid_constant__ AppendParams p) {
  extern __shared__ __align__(128) uint8_t stage_raw[];
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ AbortState ab;
  constexpr int esz = kF32In ? 4 : 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row_elems = static_cast<long long>(p.heads) * 128;
  const int T = p.chunk_tokens;
  const int per = (p.n_tokens + T - 1) / T;          // chunks per (block, tensor)
  const long long n_chunks = 2LL * p.blocks * per;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);  // one arrival per consumer warp
    }
    ab.flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (warp == 8) {
    if (lane == 0) {
      int i = 0;
      bool ok = true;
      for (long long q = blockIdx.x; q < n_chunks && ok; q += gridDim.x, ++i) {
        const int s = i % kStages, u = i / kStages;
        if (u > 0 && !lane_wait(&empty[s], (u - 1) & 1, &ab, p.err)) {
          ok = false;
          break;
        }
        const long long bt = q / per;
        const int ci = static_cast<int>(q - bt * per);
        const int b = static_cast<int>(bt >> 1), tensor = static_cast<int>(bt & 1);
        const int n0 = ci * T, nt = min(T, p.n_tokens - n0);
        const char* src = static_cast<const char*>(tensor ? p.v : p.k) +
                          (b * p.block_stride + (static_cast<long long>(p.first_frame) * p.tpf + n0) * row_elems) * esz;
        const uint32_t bytes = static_cast<uint32_t>(nt * row_elems * esz);
        if (in_bounds(b * p.block_stride + (static_cast<long long>(p.first_frame) * p.tpf + n0) * row_elems,
                      nt * row_elems, p.src_extent, p.err)) {
          mbar_arrive_expect_tx(&full[s], bytes);
          bulk_load(stage_raw + s * kStageBytes, src, bytes, &full[s]);
        } else {
          mbar_arrive(&full[s]);  // nothing loaded; the slot's rows are written from stale data
        }
      }
      if (!ok) {
        // Abort: give the loads already issued time to land.
        for (int j = i - 1; j >= 0 && j >= i - kStages; --j)
          lane_wait_teardown(&full[j % kStages], (j / kStages) & 1, 20000000ull);
      }
    }
  } else {
    const int grp = threadIdx.x >> 4;  // 0..15
    const int g = threadIdx.x & 15;
    const unsigned gmask = 0xFFFFu << (threadIdx.x & 16);
    int i = 0;
    bool ok = true;
    for (long long q = blockIdx.x; q < n_chunks && ok; q += gridDim.x, ++i) {
      const int s = i % kStages, u = i / kStages;
      if (!warp_wait(&full[s], u & 1, &ab, p.err)) {
        ok = false;
        break;
      }
      const long long bt = q / per;
      const int ci = static_cast<int>(q - bt * per);
      const int b = static_cast<int>(bt >> 1), tensor = static_cast<int>(bt & 1);
      const int n0 = ci * T, nt = min(T, p.n_tokens - n0);
      const int rows = nt * p.heads;
      const uint8_t* stage = stage_raw + s * kStageBytes;
      // Both 16-lane groups of a warp take the same number of rows.
      for (int r = grp; r < ((rows + 15) & ~15); r += 16) {
        if (r < rows) {
          const int tok = fast_div(r, p.heads_div), h = r - tok * p.heads;
          float x[8];
          const uint8_t* src = stage + (r * 128 + 8 * g) * esz;  // row r = tok * heads + h of the chunk
          if constexpr (kF32In) {
            const float4 a = *reinterpret_cast<const float4*>(src);
            const float4 c = *reinterpret_cast<const float4*>(src + 16);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
          } else {
            const uint4 w = *reinterpret_cast<const uint4*>(src);
            const uint32_t uu[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              x[2 * e] = __uint_as_float(uu[e] << 16);
              x[2 * e + 1] = __uint_as_float(uu[e] & 0xFFFF0000u);
            }
          }
          const int n = n0 + tok;
          const int f = fast_div(n, p.tpf_div);  // written frames never exceed the ring, so one wrap at most
          int slot_frame = p.base_slot_frame + f;
          if (slot_frame >= p.capacity_frames) slot_frame -= p.capacity_frames;
          const long long dst_row = (static_cast<long long>(b) * p.heads + h) * p.cap_slots +
                                    static_cast<long long>(slot_frame) * p.tpf + (n - f * p.tpf);
          write_row<K>(p, tensor, dst_row, x, g, gmask);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

// Fused 3D RoPE + append (the KV-write stage): K rows are rotated in float32
// at their absolute positions (latent frame t0 + f, h, w) and then quantised
// or copied like any other row; V rows are appended unchanged.  A CTA covers
// kRopeAppendTokens consecutive tokens of 16 heads: it issues all its loads,
// computes the cos/sin of its tokens' rotary pairs once into shared memory
// (shared by the 16 heads), then rotates, quantises and writes.  With float32
// input the rotation is the RoPE kernel's arithmetic, so the cache receives
// exactly what RoPE followed by append would write.
constexpr int kRopeAppendTokens = 8;

template <bool kF32In, int K>
__global__ void __launch_bounds__(256) append_rope_kernel(const __grid_constant__ AppendParams p,
                                                          const __grid_constant__ RopeParams rp, TwoPi tp) {
  __shared__ float2 cs[kRopeAppendTokens][kRopeMaxPairs];  // (cos, sin) per token and pair
  const int h = blockIdx.y * 16 + (threadIdx.x >> 4);
  const bool live = h < p.heads;
  const int g = threadIdx.x & 15;
  const unsigned gmask = 0xFFFFu << (threadIdx.x & 16);
  const int tensor = blockIdx.z & 1;
  const int b = blockIdx.z >> 1;
  const int n0 = blockIdx.x * kRopeAppendTokens;
  const void* src = tensor ? p.v : p.k;
  const long long plane = static_cast<long long>(b) * p.heads + h;
  float x[kRopeAppendTokens][8];
  if (live) {
#pragma unroll
    for (int r = 0; r < kRopeAppendTokens; ++r) {
      const int n = n0 + r;
      if (n < p.n_tokens) {
        const long long src_tok = static_cast<long long>(p.first_frame) * p.tpf + n;
        const long long off = b * p.block_stride + (src_tok * p.heads + h) * 128 + 8 * g;
        if (in_bounds(off, 8, p.src_extent, p.err))
          load8<kF32In>(src, off, x[r]);
        else
#pragma unroll
          for (int e = 0; e < 8; ++e) x[r][e] = 0.0f;
      }
    }
  }
  if (tensor == 0) {
    for (int i = threadIdx.x; i < kRopeAppendTokens * kRopeMaxPairs; i += blockDim.x) {
      const int r = i / kRopeMaxPairs, pair = i - r * kRopeMaxPairs;
      const int n = n0 + r;
      const int a = rp.axis[pair];
      float c = 1.0f, sn = 0.0f;
      if (n < p.n_tokens && a >= 0) {
        const int f = fast_div(n, p.tpf_div);
        const int within = n - f * p.tpf;
        const int row = fast_div(within, rp.gw_div);
        const float pos = static_cast<float>(a == 0 ? static_cast<int>(rp.t0) + f
                                                    : (a == 1 ? row : within - row * rp.grid_w));
        sincosf(rope_reduced_angle(pos, rp.f_hi[pair], rp.f_lo[pair], tp), &sn, &c);
      }
      cs[r][pair] = make_float2(c, sn);
    }
    __syncthreads();  // tensor is uniform over the CTA
  }
  if (!live) return;  // whole 16-lane groups leave together
#pragma unroll
  for (int r = 0; r < kRopeAppendTokens; ++r) {
    const int n = n0 + r;
    if (n >= p.n_tokens) break;
    if (tensor == 0) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 t = cs[r][4 * g + e];
        rope_rotate_pair(x[r][2 * e], x[r][2 * e + 1], t.x, t.y);
      }
    }
    const int f = fast_div(n, p.tpf_div);  // written frames never exceed the ring, so one wrap at most
    int slot_frame = p.base_slot_frame + f;
    if (slot_frame >= p.capacity_frames) slot_frame -= p.capacity_frames;
    const long long dst_row = plane * p.cap_slots + static_cast<long long>(slot_frame) * p.tpf + (n - f * p.tpf);
    write_row<K>(p, tensor, dst_row, x[r], g, gmask);
  }
}

// Fused RoPE + append for bf16 input, in the 8-lanes-per-row layout of
// append8_kernel (lane g holds values 16g .. 16g+15, i.e. rotary pairs
// 8g .. 8g+7).  A CTA takes 64 consecutive (token, head) rows of the input,
// which is one contiguous 16 KB range, two rows per 8-lane group; the cos/sin
// of the tokens those rows belong to are computed once into shared memory.
constexpr int kRope8Rows = 64;
constexpr int kRope8MaxTokens = kRope8Rows + 1;  // tokens a 64-row range can touch (heads = 1)

template <int K>
__global__ void __launch_bounds__(256, 4) append8_rope_kernel(const __grid_constant__ AppendParams p,
                                                              const __grid_constant__ RopeParams rp, TwoPi tp) {
  __shared__ __align__(16) float2 cs[kRope8MaxTokens][kRopeMaxPairs];
  const int g = threadIdx.x & 7;
  const unsigned gmask = 0xFFu << (threadIdx.x & 24);
  const int tensor = blockIdx.z & 1;
  const int b = blockIdx.z >> 1;
  // rows = n_tokens * heads < 2^31 (checked by the launcher)
  const int rows = p.n_tokens * p.heads;
  const int r0 = static_cast<int>(blockIdx.x) * kRope8Rows;
  const long long src0 = b * p.block_stride + static_cast<long long>(p.first_frame) * p.tpf * p.heads * 128;
  const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(tensor ? p.v : p.k) + src0;
  uint4 w[2][2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = r0 + (threadIdx.x >> 3) + 32 * r;
    if (row < rows) {
      const long long off = src0 + static_cast<long long>(row) * 128 + 16 * g;
      if (in_bounds(off, 16, p.src_extent, p.err)) {
        const uint4* q = reinterpret_cast<const uint4*>(src + static_cast<long long>(row) * 128 + 16 * g);
        w[r][0] = q[0];
        w[r][1] = q[1];
      } else {
        w[r][0] = w[r][1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  const int tok0 = fast_div(r0, p.heads_div);
  if (tensor == 0) {
    const int n_tok = fast_div(min(rows - 1, r0 + kRope8Rows - 1), p.heads_div) - tok0 + 1;
    for (int i = threadIdx.x; i < n_tok * kRopeMaxPairs; i += blockDim.x) {
      const int t = i / kRopeMaxPairs, pair = i - t * kRopeMaxPairs;
      const int n = tok0 + t;
      const int a = rp.axis[pair];
      float c = 1.0f, sn = 0.0f;
      if (a >= 0) {
        const int f = fast_div(n, p.tpf_div);
        const int within = n - f * p.tpf;
        const int hrow = fast_div(within, rp.gw_div);
        const float pos = static_cast<float>(a == 0 ? static_cast<int>(rp.t0) + f
                                                    : (a == 1 ? hrow : within - hrow * rp.grid_w));
        sincosf(rope_reduced_angle(pos, rp.f_hi[pair], rp.f_lo[pair], tp), &sn, &c);
      }
      // Lane g's pairs 8g .. 8g+7 as four 16-byte chunks, chunk i of all eight
      // lanes side by side: a group's table reads are contiguous 128 bytes.
      cs[t][((pair & 7) >> 1) * 16 + 2 * (pair >> 3) + (pair & 1)] = make_float2(c, sn);
    }
    __syncthreads();  // tensor is uniform over the CTA
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = r0 + (threadIdx.x >> 3) + 32 * r;
    if (row >= rows) break;  // rows of one 8-lane group: uniform
    const int n = fast_div(row, p.heads_div);
    const int h = row - n * p.heads;
    const uint32_t u[8] = {w[r][0].x, w[r][0].y, w[r][0].z, w[r][0].w, w[r][1].x, w[r][1].y, w[r][1].z, w[r][1].w};
    float x[16];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      x[2 * e] = __uint_as_float(u[e] << 16);
      x[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
    }
    if (tensor == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 t = *reinterpret_cast<const float4*>(&cs[n - tok0][16 * i + 2 * g]);
        rope_rotate_pair(x[4 * i], x[4 * i + 1], t.x, t.y);
        rope_rotate_pair(x[4 * i + 2], x[4 * i + 3], t.z, t.w);
      }
    }
    const int f = fast_div(n, p.tpf_div);  // written frames never exceed the ring, so one wrap at most
    int slot_frame = p.base_slot_frame + f;
    if (slot_frame >= p.capacity_frames) slot_frame -= p.capacity_frames;
    const long long dst_row = (static_cast<long long>(b) * p.heads + h) * p.cap_slots +
                              static_cast<long long>(slot_frame) * p.tpf + (n - f * p.tpf);
    store_row16<K>(p, tensor, dst_row, x, g, gmask);
  }
}

__global__ void __launch_bounds__(256) zero_fill_kernel(uint8_t* __restrict__ ptr, size_t bytes) {
  const size_t n16 = bytes / 16;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride)
    reinterpret_cast<uint4*>(ptr)[i] = make_uint4(0u, 0u, 0u, 0u);
  const size_t tail = n16 * 16 + static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tail < bytes) ptr[tail] = 0;
}

// BF16 copy of the resident window of a one-byte cache: x_hat = bf16(fl32(code
// * scale)), the same value the attention kernel's dequantising warps put in
// shared memory (the code converts exactly, one rounded multiply by the row
// scale, one rounding to bf16).  Eight lanes per 128-value row, 16 codes each:
// one 16-byte load, two 16-byte stores.  grid.y walks the (tensor, plane)
// pairs, grid.x and the loop the slots [0, n_slots) of a plane.
// Converts one 16-code chunk (codes of one row, its scale) to 16 bf16 values.
template <int K>
__device__ __forceinline__ void expand_chunk(const uint4& w, float sc, uint32_t (&o)[8]) {
  if constexpr (K == kCacheFp8) {
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wd[e] & 0xFFFFu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(wd[e] >> 16), __NV_E4M3);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      o[2 * e] = pack_bf16x2(__fmul_rn(a.x, sc), __fmul_rn(a.y, sc));
      o[2 * e + 1] = pack_bf16x2(__fmul_rn(b.x, sc), __fmul_rn(b.y, sc));
    }
  } else {
    // The biased byte c + 128 in the low mantissa bits of 2^23 gives the
    // float 2^23 + 128 + c; subtracting 2^23 + 128 leaves c exactly.
    const uint32_t wd[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float f[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        f[i] = __fmul_rn(__fadd_rn(__uint_as_float(__byte_perm(wd[e], 0x4B000000u, 0x7540u + i)), -8388736.0f), sc);
      o[2 * e] = pack_bf16x2(f[0], f[1]);
      o[2 * e + 1] = pack_bf16x2(f[2], f[3]);
    }
  }
}

// BF16 copy of the resident window of a one-byte cache: x_hat = bf16(fl32(code
// * scale)), the same value the attention kernel's dequantising warps put in
// shared memory (the code converts exactly, one rounded multiply by the row
// scale, one rounding to bf16).  Eight lanes per 128-value row, 16 codes each:
// one 16-byte load, two 16-byte stores; a lane group has the loads of eight
// rows in flight before it converts any.  grid.y walks the (tensor, plane)
// pairs, grid.x and the loop the slots [0, n_slots) of a plane.
constexpr int kExpandRows = 8;  // rows in flight per 8-lane group

template <int K>
__global__ void __launch_bounds__(256) expand_kernel(const __grid_constant__ ExpandParams p) {
  const int c = threadIdx.x & 7;  // 16-code chunk of the row
  const long long total_rows = static_cast<long long>(p.planes) * p.cap_slots;
  for (long long tp = blockIdx.y; tp < 2LL * p.planes; tp += gridDim.y) {
    const int tensor = tp >= p.planes ? 1 : 0;
    const long long plane = tp - static_cast<long long>(tensor) * p.planes;
    const uint8_t* codes = static_cast<const uint8_t*>(tensor ? p.vc : p.kc);
    const float* scales = tensor ? p.vs : p.ks;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(tensor ? p.vo : p.ko);
    for (long long slot0 = (static_cast<long long>(blockIdx.x) * 32 + (threadIdx.x >> 3)) * kExpandRows;
         slot0 < p.n_slots; slot0 += static_cast<long long>(gridDim.x) * 32 * kExpandRows) {
      uint4 w[kExpandRows];
      float sc[kExpandRows];
#pragma unroll
      for (int r = 0; r < kExpandRows; ++r) {
        const long long slot_row = plane * p.cap_slots + slot0 + r;  // row of the cache arrays
        const bool live = slot0 + r < p.n_slots && in_bounds(slot_row, 1, total_rows, p.err);
        w[r] = live ? *reinterpret_cast<const uint4*>(codes + slot_row * 128 + 16 * c) : make_uint4(0u, 0u, 0u, 0u);
        sc[r] = live ? scales[slot_row] : 0.0f;
      }
#pragma unroll
      for (int r = 0; r < kExpandRows; ++r) {
        const long long slot_row = plane * p.cap_slots + slot0 + r;
        if (slot0 + r >= p.n_slots || !in_bounds(slot_row, 1, total_rows, p.err)) continue;
        uint32_t o[8];
        expand_chunk<K>(w[r], sc[r], o);
        uint4* dst = reinterpret_cast<uint4*>(out + slot_row * 128 + 16 * c);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_expand(int kind, const ExpandParams& p, cudaStream_t stream) {
  if (p.planes <= 0 || p.n_slots <= 0) return cudaSuccess;
  if (kind != kCacheInt8 && kind != kCacheFp8) return cudaErrorInvalidValue;
  const long long xs = (p.n_slots + 32 * kExpandRows - 1) / (32 * kExpandRows);  // 32 lane groups per CTA
  const long long tps = 2LL * p.planes;
  const dim3 grid(static_cast<unsigned>(xs < 64 ? xs : 64), static_cast<unsigned>(tps < 65535 ? tps : 65535));
  if (kind == kCacheInt8)
    expand_kernel<kCacheInt8><<<grid, 256, 0, stream>>>(p);
  else
    expand_kernel<kCacheFp8><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append_rope(bool f32_in, int kind, const AppendParams& p, const RopeParams& rp,
                               cudaStream_t stream) {
  if (p.n_tokens <= 0 || p.blocks <= 0 || p.heads <= 0) return cudaSuccess;
  if (kind != kCacheBF16 && kind != kCacheInt8 && kind != kCacheFp8) return cudaErrorInvalidValue;
  const TwoPi tp = rope_two_pi();
  const long long rows = static_cast<long long>(p.n_tokens) * p.heads;
  if (f32_in || rows >= 0x7FFFFFFFLL - kRope8Rows) {
    // Float32 input, or more rows than 32-bit row indices cover: 16 lanes per
    // row, a CTA per 8 tokens and 16 heads.
    const dim3 grid(static_cast<unsigned>((p.n_tokens + kRopeAppendTokens - 1) / kRopeAppendTokens),
                    static_cast<unsigned>((p.heads + 15) / 16), static_cast<unsigned>(2 * p.blocks));
    if (grid.y > 65535 || grid.z > 65535) return cudaErrorInvalidValue;
    if (f32_in) {
      if (kind == kCacheInt8)
        append_rope_kernel<true, kCacheInt8><<<grid, 256, 0, stream>>>(p, rp, tp);
      else if (kind == kCacheFp8)
        append_rope_kernel<true, kCacheFp8><<<grid, 256, 0, stream>>>(p, rp, tp);
      else
        append_rope_kernel<true, kCacheBF16><<<grid, 256, 0, stream>>>(p, rp, tp);
    } else {
      if (kind == kCacheInt8)
        append_rope_kernel<false, kCacheInt8><<<grid, 256, 0, stream>>>(p, rp, tp);
      else if (kind == kCacheFp8)
        append_rope_kernel<false, kCacheFp8><<<grid, 256, 0, stream>>>(p, rp, tp);
      else
        append_rope_kernel<false, kCacheBF16><<<grid, 256, 0, stream>>>(p, rp, tp);
    }
  } else {
    const long long cta = (rows + kRope8Rows - 1) / kRope8Rows;
    if (2LL * p.blocks > 65535) return cudaErrorInvalidValue;
    const dim3 grid8(static_cast<unsigned>(cta), 1, static_cast<unsigned>(2 * p.blocks));
    if (kind == kCacheInt8)
      append8_rope_kernel<kCacheInt8><<<grid8, 256, 0, stream>>>(p, rp, tp);
    else if (kind == kCacheFp8)
      append8_rope_kernel<kCacheFp8><<<grid8, 256, 0, stream>>>(p, rp, tp);
    else
      append8_rope_kernel<kCacheBF16><<<grid8, 256, 0, stream>>>(p, rp, tp);
  }
  return cudaGetLastError();
}

namespace {
template <bool kF32In, int K>
cudaError_t launch_staged(const AppendParams& p, unsigned grid, cudaStream_t stream) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t smem = kStages * kStageBytes;
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(append_staged_kernel<kF32In, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  append_staged_kernel<kF32In, K><<<grid, kStagedThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int K>
cudaError_t launch_direct(bool f32_in, const AppendParams& p, cudaStream_t stream) {
  if (!f32_in) {
    const long long rows = static_cast<long long>(p.n_tokens) * p.heads;
    const long long cta = (rows + kAppend8Rows - 1) / kAppend8Rows;
    if (rows >= 0x7FFFFFFFLL - kAppend8Rows || 2LL * p.blocks > 65535) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(cta), 1, static_cast<unsigned>(2 * p.blocks));
    append8_kernel<K><<<grid, 256, 0, stream>>>(p);
  } else {
    const dim3 grid(static_cast<unsigned>((p.n_tokens + kAppendTokens - 1) / kAppendTokens),
                    static_cast<unsigned>((p.heads + 15) / 16), static_cast<unsigned>(2 * p.blocks));
    if (grid.y > 65535 || grid.z > 65535) return cudaErrorInvalidValue;
    append_kernel<true, K><<<grid, 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_append(bool f32_in, int kind, const AppendParams& p_in, int sms, cudaStream_t stream) {
  if (p_in.n_tokens <= 0 || p_in.blocks <= 0 || p_in.heads <= 0) return cudaSuccess;
  if (kind != kCacheBF16 && kind != kCacheInt8 && kind != kCacheFp8) return cudaErrorInvalidValue;
  AppendParams p = p_in;
  const long long token_bytes = static_cast<long long>(p.heads) * 128 * (f32_in ? 4 : 2);
  const long long in_bytes = 2LL * p.blocks * p.n_tokens * token_bytes;
  // Large appends (a whole session's worth of blocks) stream through shared
  // memory; small ones finish sooner with the direct kernel's many small CTAs.
  if (sms > 0 && p.err != nullptr && token_bytes <= kStageBytes && in_bytes >= (256LL << 20)) {
    // Staged path: chunks of up to 32 KB of whole token rows.
    p.chunk_tokens = static_cast<int>(kStageBytes / token_bytes);
    const long long chunks = 2LL * p.blocks * ((p.n_tokens + p.chunk_tokens - 1) / p.chunk_tokens);
    const unsigned grid = static_cast<unsigned>(chunks < 2LL * sms ? chunks : 2LL * sms);
    if (f32_in) {
      if (kind == kCacheInt8) return launch_staged<true, kCacheInt8>(p, grid, stream);
      if (kind == kCacheFp8) return launch_staged<true, kCacheFp8>(p, grid, stream);
      return launch_staged<true, kCacheBF16>(p, grid, stream);
    }
    if (kind == kCacheInt8) return launch_staged<false, kCacheInt8>(p, grid, stream);
    if (kind == kCacheFp8) return launch_staged<false, kCacheFp8>(p, grid, stream);
    return launch_staged<false, kCacheBF16>(p, grid, stream);
  }
  if (kind == kCacheInt8) return launch_direct<kCacheInt8>(f32_in, p, stream);
  if (kind == kCacheFp8) return launch_direct<kCacheFp8>(f32_in, p, stream);
  return launch_direct<kCacheBF16>(f32_in, p, stream);
}

cudaError_t launch_zero_fill(void* ptr, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  size_t blocks = (bytes / 16 + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 148 * 16) blocks = 148 * 16;
  zero_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<uint8_t*>(ptr), bytes);
  return cudaGetLastError();
}

}  // namespace nomas
