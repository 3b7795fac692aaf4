// camera_attn.cu - cross-attention of the video tokens to the camera tokens
// of their latent frame.
//
// Camera control enters as 4x4 extrinsic matrices grouped over four frames
// and fed through cross-attention in every block (the blog.authon.dev guide
// to running Hy-Nomas on an RTX 4090, section "What Hy-Nomas is", model-card
// specs; the orcarouter.ai explainer, section "Zwei Lenkräder, und nur eines
// davon ist ein Prompt", on steering by a trajectory of camera extrinsics).
// One latent frame covers four video frames (the same spec list: 4x temporal
// compression), so the reading here: the camera
// encoder turns each latent frame's group into n_cam key/value tokens per
// head, and every video token of that latent frame attends to exactly those
// tokens: O = softmax(s q K_f^T) V_f.  The encoder needs trained weights and
// lies upstream; this kernel takes its K/V.
//
// HBM-bound: each query row is read once and its output written once.  Both
// products run on the tensor cores, so the CUDA cores only do the softmax and
// the output conversion.  A CTA takes one tile of 128 query rows of one head
// and one latent frame:
//   - warp 4 TMA-loads the Q tile (two 64-column panels, 128-byte swizzle)
//     and the frame's camera K and V of the head (16 rows; rows past n_cam
//     lie outside the tensor map's camera-token extent and arrive as zeros),
//     then issues S = Q K^T (M 128, N 16, K 128) into tensor memory;
//   - warps 0-3 (one query row per thread, the row's tensor-memory lane) read
//     S, mask the columns past n_cam, take the softmax in float32 (log2
//     domain) and write P as bf16 over the first 32 bytes of each row of the
//     spent Q panel;
//   - warp 4 issues O = P V (M 128, N 128, K 16) over S's columns;
//   - warps 0-3 scale O by 1 / row sum, convert it to bf16 into the Q tile's
//     shared memory, and one thread TMA-stores it.  The tensor maps bound the
//     token coordinate by the frame's token count, so the last tile's rows past
//     the frame load as zeros and are not stored.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "checks.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace nomas {
namespace {

constexpr int kCamThreads = 160;                        // warps 0-3: rows; warp 4: TMA and MMA
constexpr uint32_t kCamPanel = 128 * 128;              // one 64-column bf16 panel of 128 rows
constexpr uint32_t kCamQBytes = 2 * kCamPanel;         // Q tile, later P, later O
constexpr uint32_t kCamKVPanel = 16 * 128;             // one 64-column panel of 16 camera rows
constexpr uint32_t kCamKVBytes = 2 * kCamKVPanel;
// 48 KB of dynamic shared memory caps residency at four CTAs per SM, which is
// what the 4 x 128 tensor-memory columns allow.
constexpr uint32_t kCamSmem = 48 * 1024;
static_assert(1024 + kCamQBytes + 2 * kCamKVBytes <= kCamSmem, "camera tile exceeds its shared memory");
constexpr uint32_t kIdescCamS = idesc_bf16_f32(128, 16, false);  // S = Q K^T, both K-major
constexpr uint32_t kIdescCamO = idesc_bf16_f32(128, 128, true);  // O = P V, V N-major

__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Tensor store of a box from shared memory; elements outside the tensor are
// not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* smem_src, int c0, int c1, int c2,
                                             int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until the committed tensor stores have read their shared-memory source.
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// 16-byte chunk `c` (0..7) of row `r` of a 128-byte-swizzled panel.
__device__ __forceinline__ uint4* sw128_chunk(uint8_t* panel, int r, int c) {
  return reinterpret_cast<uint4*>(panel + r * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kCamThreads, 4)
    camera_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CameraAttnParams p) {
  extern __shared__ uint8_t cam_raw[];
  uint8_t* sQ = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(cam_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sQ + kCamQBytes;
  uint8_t* sV = sK + kCamKVBytes;
  // 0: loads landed, 1: S ready, 2: P written (one arrival per row), 3: O ready
  __shared__ uint64_t bars[4];
  __shared__ uint32_t tmem_base;
  __shared__ AbortState ab;
  const int warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * 128, h = blockIdx.y, f = blockIdx.z;
  if (threadIdx.x == 0) {
    ab.flag = 0;
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 128);
    mbar_init(&bars[3], 1);
    fence_mbarrier_init();
  }
  if (warp == 4) {
    tmem_alloc(&tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA and MMA
    if (elect_one()) {
      // The grid covers exactly the tiles, heads and frames (recorded, never false, in the checked build).
      (void)(in_bounds(t0, 1, p.tpf, p.err) && in_bounds(h, 1, p.heads, p.err) && in_bounds(f, 1, p.frames, p.err));
      tma_prefetch_desc(&tm_q);
      mbar_arrive_expect_tx(&bars[0], kCamQBytes + 2 * kCamKVBytes);
      for (int pn = 0; pn < 2; ++pn) {
        tma_load_4d(sQ + pn * kCamPanel, &tm_q, &bars[0], 64 * pn, h, t0, f);
        tma_load_4d(sK + pn * kCamKVPanel, &tm_k, &bars[0], 64 * pn, h, 0, f);
        tma_load_4d(sV + pn * kCamKVPanel, &tm_v, &bars[0], 64 * pn, h, 0, f);
      }
    }
    __syncwarp();
    int issued = 0;  // MMA groups committed (S, then O)
    bool ok = warp_wait(&bars[0], 0, &ab, p.err);
    if (ok) {
      tc_fence_after();
      const uint64_t q_desc = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t k_desc = smem_desc_sw128(smem_u32(sK), 16, 1024);
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t a = q_desc + (((k >> 2) * kCamPanel + (k & 3) * 32) >> 4);
          const uint64_t b = k_desc + (((k >> 2) * kCamKVPanel + (k & 3) * 32) >> 4);
          mma_ss(tmem, a, b, kIdescCamS, k > 0 ? 1u : 0u);
        }
        mma_commit(&bars[1]);
      }
      __syncwarp();
      issued = 1;
      ok = warp_wait(&bars[2], 0, &ab, p.err);
    }
    if (ok) {
      tc_fence_after();
      // P: the first 16 columns (32 bytes) of each row of Q's first panel.
      // V: 16 camera rows, N-major, its two 64-column panels kCamKVPanel apart.
      const uint64_t p_desc = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t v_desc = smem_desc_sw128(smem_u32(sV), kCamKVPanel, 1024);
      if (elect_one()) {
        mma_ss(tmem, p_desc, v_desc, kIdescCamO, 0u);
        mma_commit(&bars[3]);
      }
      __syncwarp();
      issued = 2;
    }
    // Teardown: the loads and every MMA group this warp issued have landed
    // before the CTA's shared and tensor memory go away (immediate when the
    // other warps already waited for them).
    warp_wait_teardown(&bars[0], 0, 20000000ull);
    if (issued >= 1) warp_wait_teardown(&bars[1], 0, 20000000ull);
    if (issued >= 2) warp_wait_teardown(&bars[3], 0, 20000000ull);
  } else {
    // ------------------------------------------------------------ softmax and output (row r)
    const int r = threadIdx.x;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
    float inv_l = 0.0f;
    bool ok = warp_wait(&bars[1], 0, &ab, p.err);
    if (ok) {
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld_x32(taddr, sr);  // columns 0..15 hold S; the rest are unused
      float s[16];
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        s[j] = j < p.n_cam ? __uint_as_float(sr[j]) * p.scale_log2 : -INFINITY;
        m = fmaxf(m, s[j]);
      }
      float l = 0.0f;
      uint32_t pk[8];
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const float p0 = fast_exp2(s[j] - m), p1 = fast_exp2(s[j + 1] - m);
        l += p0 + p1;
        pk[j >> 1] = pack_bf16x2(p0, p1);
      }
      inv_l = 1.0f / l;
      *sw128_chunk(sQ, r, 0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *sw128_chunk(sQ, r, 1) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[2]);
      ok = warp_wait(&bars[3], 0, &ab, p.err);
    }
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {  // output columns 32 c4 .. 32 c4 + 31
        uint32_t o[32];
        tmem_ld_x32(taddr + 32 * c4, o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        uint8_t* panel = sQ + (c4 >> 1) * kCamPanel;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *sw128_chunk(panel, r, 4 * (c4 & 1) + q) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    named_bar_sync(1, 128);  // every row is staged (or the CTA gave up)
    if (r == 0 && !ab.flag) {
      for (int pn = 0; pn < 2; ++pn) tma_store_4d(&tm_o, sQ + pn * kCamPanel, 64 * pn, h, t0, f);
      tma_store_wait_read();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

}  // namespace

cudaError_t launch_camera_attn(const CameraTensorMaps& tm, const CameraAttnParams& p, cudaStream_t stream) {
  if (p.frames <= 0 || p.tpf <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((p.tpf + 127) / 128), static_cast<unsigned>(p.heads),
                  static_cast<unsigned>(p.frames));
  if (grid.y > 65535 || grid.z > 65535) return cudaErrorInvalidValue;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(camera_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCamSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  camera_attn_kernel<<<grid, kCamThreads, kCamSmem, stream>>>(tm.q, tm.k, tm.v, tm.o, p);
  return cudaGetLastError();
}

}  // namespace nomas
