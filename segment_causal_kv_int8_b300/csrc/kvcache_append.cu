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
// 16 threads own a row (8 values each: a 16-byte bf16 or 32-byte f32 load),
// reduce the absmax with four shuffles and write 8 code bytes each plus the
// row's scale.  A CTA covers a few consecutive tokens of 16 heads, so it reads
// whole token rows and writes runs of consecutive ring slots per head.
//
// Codec bits (identical to the reference definition): scale = fl32(m / 127),
// inv = fl32(127 / m) (IEEE round-to-nearest divisions), code =
// clamp(cvt.rni(fl32(x * inv)), -127, 127); the float->int conversion maps NaN
// (0 * inf on an all-zero row) to 0 and saturates +-inf.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

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

constexpr int kAppendTokens = 2;  // tokens per block (and rows per 16-lane group)

// Grid: x = groups of kAppendTokens tokens, y = groups of 16 heads, z = (block,
// tensor).  16 lanes own one (token, head) row, 8 values each; the 16 row
// groups of a CTA are 16 consecutive heads, so a CTA reads whole token rows
// ([heads][128] contiguous in the input) and writes, per head, kAppendTokens
// consecutive ring slots.  Each lane group issues all its loads before any
// arithmetic.
// Many small CTAs (eight per SM for bf16 input) keep enough rows in flight.
template <bool kF32In, bool kInt8>
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
      load8<kF32In>(src, b * p.block_stride + (src_tok * p.heads + h) * 128 + 8 * g, x[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < kAppendTokens; ++r) {
    const int n = n0 + r;
    if (n >= p.n_tokens) break;
    const int f = n / p.tpf;  // written frames never exceed the ring, so one wrap at most
    int slot_frame = p.base_slot_frame + f;
    if (slot_frame >= p.capacity_frames) slot_frame -= p.capacity_frames;
    const long long dst_row = plane * p.cap_slots + static_cast<long long>(slot_frame) * p.tpf + (n - f * p.tpf);
    if constexpr (kInt8) {
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(x[r][e]));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(gmask, m, off));
      const float scale = __fdiv_rn(m, 127.0f);
      const float inv = __fdiv_rn(127.0f, m);
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int c = __float2int_rn(__fmul_rn(x[r][e], inv));
        c = max(-127, min(127, c));
        const uint32_t byte = static_cast<uint32_t>(c) & 0xFFu;
        if (e < 4)
          lo |= byte << (8 * e);
        else
          hi |= byte << (8 * (e - 4));
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
        __nv_bfloat162 t = __floats2bfloat162_rn(x[r][2 * e], x[r][2 * e + 1]);
        u[e] = *reinterpret_cast<const uint32_t*>(&t);
      }
      *reinterpret_cast<uint4*>(dst) = w;
    }
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

}  // namespace

cudaError_t launch_append(bool f32_in, bool int8_cache, const AppendParams& p, cudaStream_t stream) {
  if (p.n_tokens <= 0 || p.blocks <= 0 || p.heads <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((p.n_tokens + kAppendTokens - 1) / kAppendTokens),
                  static_cast<unsigned>((p.heads + 15) / 16), static_cast<unsigned>(2 * p.blocks));
  if (grid.y > 65535 || grid.z > 65535) return cudaErrorInvalidValue;
  if (f32_in) {
    if (int8_cache)
      append_kernel<true, true><<<grid, 256, 0, stream>>>(p);
    else
      append_kernel<true, false><<<grid, 256, 0, stream>>>(p);
  } else {
    if (int8_cache)
      append_kernel<false, true><<<grid, 256, 0, stream>>>(p);
    else
      append_kernel<false, false><<<grid, 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
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
