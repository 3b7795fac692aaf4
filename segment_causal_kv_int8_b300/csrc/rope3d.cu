// rope3d.cu - in-place 3D rotary position embedding of the video rows of Q and K.
//
// "3D RoPE" over (latent frame, h, w) is part of the model card (Hy-Nomas auf
// einer RTX 4090, section "Modell und Dateien").  The head dimension splits
// into contiguous chunks per axis; pair (x[o+2i], x[o+2i+1]) of the chunk of
// axis a rotates by pos_a * f_{a,i}, f_{a,i} = theta^(-2i/d_a).
//
// HBM-bound elementwise kernel: 16 threads own one token, each thread four
// consecutive pairs (one 16-byte bf16 vector or two float4 of every head row).
// The cos/sin of a (token, pair) is computed once and applied to all heads of
// Q and K.  The angle pos * f is formed as a two-float product (f = f_hi +
// f_lo, exact product error by fma) and reduced by the nearest multiple of
// 2*pi with a three-float 2*pi (Cody-Waite reduction with fma), so the angle
// error stays ~1e-7 rad at any frame index below 2^24; sincosf then sees |r|
// <= pi.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace nomas {
namespace {

struct TwoPi {
  float a, b, c;  // 2*pi = a + b + c (each the float nearest the remainder)
};

__device__ __forceinline__ float reduced_angle(float pos, float f_hi, float f_lo, const TwoPi& tp) {
  const float a = pos * f_hi;
  const float a_err = fmaf(pos, f_hi, -a);
  const float a_lo = fmaf(pos, f_lo, a_err);
  const float kq = rintf(a * 0.159154943091895336f);
  float r = fmaf(-kq, tp.a, a);
  r = fmaf(-kq, tp.b, r);
  r = fmaf(-kq, tp.c, r);
  return r + a_lo;
}

template <bool kBF16>
__global__ void __launch_bounds__(256) rope3d_kernel(void* __restrict__ q, void* __restrict__ k,
                                                     const __grid_constant__ RopeParams p, TwoPi tp) {
  const int g = threadIdx.x & 15;
  const long long tok = static_cast<long long>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  if (tok >= p.n_video) return;
  const int within = static_cast<int>(tok % p.tpf);
  const float pos[3] = {static_cast<float>(p.t0 + tok / p.tpf), static_cast<float>(within / p.grid_w),
                        static_cast<float>(within % p.grid_w)};
  float cs[4], sn[4];
  bool any = false;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int pair = 4 * g + e;
    const int a = p.axis[pair];
    if (a < 0) {
      cs[e] = 1.0f;
      sn[e] = 0.0f;
    } else {
      any = true;
      sincosf(reduced_angle(pos[a], p.f_hi[pair], p.f_lo[pair], tp), &sn[e], &cs[e]);
    }
  }
  if (!any) return;
  for (int which = 0; which < 2; ++which) {
    void* base = which ? k : q;
    if (base == nullptr) continue;
    if constexpr (kBF16) {
      __nv_bfloat16* row = static_cast<__nv_bfloat16*>(base) + tok * p.row_stride + 8 * g;
      for (int h0 = 0; h0 < p.heads; h0 += 4) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (h0 + u < p.heads) w[u] = *reinterpret_cast<const uint4*>(row + (h0 + u) * 128);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (h0 + u >= p.heads) continue;
          uint32_t* x = reinterpret_cast<uint32_t*>(&w[u]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&x[e]);
            const float x0 = __bfloat162float(v2.x), x1 = __bfloat162float(v2.y);
            const float y0 = fmaf(x0, cs[e], -x1 * sn[e]);
            const float y1 = fmaf(x0, sn[e], x1 * cs[e]);
            __nv_bfloat162 o2 = __floats2bfloat162_rn(y0, y1);
            x[e] = *reinterpret_cast<const uint32_t*>(&o2);
          }
          *reinterpret_cast<uint4*>(row + (h0 + u) * 128) = w[u];
        }
      }
    } else {
      float* row = static_cast<float*>(base) + tok * p.row_stride + 8 * g;
      for (int h0 = 0; h0 < p.heads; h0 += 2) {
        float4 w[2][2];
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if (h0 + u < p.heads) {
            w[u][0] = *reinterpret_cast<const float4*>(row + (h0 + u) * 128);
            w[u][1] = *reinterpret_cast<const float4*>(row + (h0 + u) * 128 + 4);
          }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (h0 + u >= p.heads) continue;
          float* x = reinterpret_cast<float*>(&w[u][0]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = x[2 * e], x1 = x[2 * e + 1];
            x[2 * e] = fmaf(x0, cs[e], -x1 * sn[e]);
            x[2 * e + 1] = fmaf(x0, sn[e], x1 * cs[e]);
          }
          *reinterpret_cast<float4*>(row + (h0 + u) * 128) = w[u][0];
          *reinterpret_cast<float4*>(row + (h0 + u) * 128 + 4) = w[u][1];
        }
      }
    }
  }
}

TwoPi two_pi_split() {
  // 2*pi to 64-bit long double precision, split into three floats.
  const long double tp = 6.283185307179586476925286766559005768L;
  TwoPi r;
  r.a = static_cast<float>(tp);
  r.b = static_cast<float>(tp - static_cast<long double>(r.a));
  r.c = static_cast<float>(tp - static_cast<long double>(r.a) - static_cast<long double>(r.b));
  return r;
}

}  // namespace

cudaError_t launch_rope3d(bool bf16_io, void* q, void* k, const RopeParams& p, cudaStream_t stream) {
  if (p.n_video <= 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((p.n_video + 15) / 16);
  const TwoPi tp = two_pi_split();
  if (bf16_io)
    rope3d_kernel<true><<<blocks, 256, 0, stream>>>(q, k, p, tp);
  else
    rope3d_kernel<false><<<blocks, 256, 0, stream>>>(q, k, p, tp);
  return cudaGetLastError();
}

}  // namespace nomas
