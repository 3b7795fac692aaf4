// rope3d.cu - in-place 3D rotary position embedding of the video rows of Q and K.
//
// "3D RoPE" over (latent frame, h, w) is part of the model card (Hy-Nomas auf
// einer RTX 4090, section "Modell und Dateien").  The head dimension splits
// into contiguous chunks per axis; pair (x[o+2i], x[o+2i+1]) of the chunk of
// axis a rotates by pos_a * f_{a,i}, f_{a,i} = theta^(-2i/d_a).
//
// HBM-bound elementwise kernel: 16 threads own one token, each thread four
// consecutive pairs (one 16-byte bf16 vector or two float4 of a head row) of a
// group of heads.  The cos/sin of a (token, pair) is computed once per head
// group and applied to those heads of Q and K (angle arithmetic in
// rope_math.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "kernels.h"
#include "rope_math.cuh"

namespace nomas {
namespace {

constexpr int kRopeHeadsPerThread = 4;

// Rotate one 8-value group (4 pairs) held as floats.
__device__ __forceinline__ void rotate8(float (&x)[8], const float (&cs)[4], const float (&sn)[4]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) rope_rotate_pair(x[2 * e], x[2 * e + 1], cs[e], sn[e]);
}

// Block: 16 tokens x 16 lanes (a lane owns 4 consecutive rotary pairs, i.e. 8
// values, of every head row); blockIdx.y picks a group of kRopeHeadsPerThread
// heads.  All loads of a thread (its heads of Q and K) are issued before any
// arithmetic so enough bytes are in flight to keep HBM busy.
template <bool kBF16>
__global__ void __launch_bounds__(256) rope3d_kernel(void* __restrict__ q, void* __restrict__ k,
                                                     const __grid_constant__ RopeParams p, TwoPi tp) {
  constexpr int HT = kRopeHeadsPerThread;
  const int g = threadIdx.x & 15;
  const int tok = blockIdx.x * 16 + (threadIdx.x >> 4);
  if (tok >= p.n_video) return;
  const int h0 = blockIdx.y * HT;
  const int nh = min(HT, p.heads - h0);
  bool any = false;
#pragma unroll
  for (int e = 0; e < 4; ++e) any |= p.axis[4 * g + e] >= 0;
  if (!any) return;
  const int nt = (k != nullptr) ? 2 : 1;
  using Vec = typename std::conditional<kBF16, uint4, float4>::type;
  constexpr int kVecs = kBF16 ? 1 : 2;  // 16-byte vectors per 8-value group
  Vec w[2][HT][kVecs];
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    if (which >= nt) break;
    const Vec* row = reinterpret_cast<const Vec*>(static_cast<const char*>(which ? k : q) +
                                                  (static_cast<long long>(tok) * p.row_stride + h0 * 128 + 8 * g) * (kBF16 ? 2 : 4));
#pragma unroll
    for (int u = 0; u < HT; ++u)
      if (u < nh)
#pragma unroll
        for (int c = 0; c < kVecs; ++c) w[which][u][c] = row[u * (128 * (kBF16 ? 2 : 4) / 16) + c];
  }
  const int frame = tok / p.tpf;
  const int within = tok - frame * p.tpf;
  const int row = within / p.grid_w;
  const float pos[3] = {static_cast<float>(p.t0 + frame), static_cast<float>(row),
                        static_cast<float>(within - row * p.grid_w)};
  float cs[4], sn[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int pair = 4 * g + e;
    const int a = p.axis[pair];
    if (a < 0) {
      cs[e] = 1.0f;
      sn[e] = 0.0f;
    } else {
      sincosf(rope_reduced_angle(pos[a], p.f_hi[pair], p.f_lo[pair], tp), &sn[e], &cs[e]);
    }
  }
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    if (which >= nt) break;
    Vec* row = reinterpret_cast<Vec*>(static_cast<char*>(which ? k : q) +
                                      (static_cast<long long>(tok) * p.row_stride + h0 * 128 + 8 * g) * (kBF16 ? 2 : 4));
#pragma unroll
    for (int u = 0; u < HT; ++u) {
      if (u >= nh) continue;
      float x[8];
      if constexpr (kBF16) {
        const uint32_t* v = reinterpret_cast<const uint32_t*>(&w[which][u][0]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[2 * e] = __uint_as_float(v[e] << 16);
          x[2 * e + 1] = __uint_as_float(v[e] & 0xFFFF0000u);
        }
      } else {
        const float* v = reinterpret_cast<const float*>(&w[which][u][0]);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = v[e];
      }
      rotate8(x, cs, sn);
      if constexpr (kBF16) {
        uint4 o;
        uint32_t* ov = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat162 t2 = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
          ov[e] = *reinterpret_cast<const uint32_t*>(&t2);
        }
        row[u * 16] = o;
      } else {
        row[u * 32] = make_float4(x[0], x[1], x[2], x[3]);
        row[u * 32 + 1] = make_float4(x[4], x[5], x[6], x[7]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_rope3d(bool bf16_io, void* q, void* k, const RopeParams& p, cudaStream_t stream) {
  if (p.n_video <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((p.n_video + 15) / 16),
                  static_cast<unsigned>((p.heads + kRopeHeadsPerThread - 1) / kRopeHeadsPerThread));
  if (grid.y > 65535) return cudaErrorInvalidValue;
  const TwoPi tp = rope_two_pi();
  if (bf16_io)
    rope3d_kernel<true><<<grid, 256, 0, stream>>>(q, k, p, tp);
  else
    rope3d_kernel<false><<<grid, 256, 0, stream>>>(q, k, p, tp);
  return cudaGetLastError();
}

}  // namespace nomas
