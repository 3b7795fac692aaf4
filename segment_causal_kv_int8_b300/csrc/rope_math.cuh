// rope_math.cuh - angle arithmetic shared by the RoPE kernel and the fused
// RoPE + append kernel.
//
// Pair i of axis a rotates by pos_a * f_{a,i}, f_{a,i} = theta^(-2i/d_a)
// (3D RoPE over latent frame, h and w; Hy-Nomas auf einer RTX 4090, section
// "Modell und Dateien").  The angle is formed as a two-float product (f =
// f_hi + f_lo, the product's rounding error recovered by fma) and reduced by
// the nearest multiple of 2*pi held as three floats (Cody-Waite reduction with
// fma), so its error stays ~1e-7 rad at any frame index below 2^24 and
// sincosf sees |r| <= pi.
#pragma once

#include <cuda_runtime.h>

namespace nomas {

struct TwoPi {
  float a, b, c;  // 2*pi = a + b + c (each the float nearest the remainder)
};

__device__ __forceinline__ float rope_reduced_angle(float pos, float f_hi, float f_lo, const TwoPi& tp) {
  const float a = pos * f_hi;
  const float a_err = fmaf(pos, f_hi, -a);
  const float a_lo = fmaf(pos, f_lo, a_err);
  const float kq = rintf(a * 0.159154943091895336f);
  float r = fmaf(-kq, tp.a, a);
  r = fmaf(-kq, tp.b, r);
  r = fmaf(-kq, tp.c, r);
  return r + a_lo;
}

// (x0, x1) -> (x0 c - x1 s, x0 s + x1 c)
__device__ __forceinline__ void rope_rotate_pair(float& x0, float& x1, float c, float s) {
  const float y0 = fmaf(x0, c, -x1 * s);
  const float y1 = fmaf(x0, s, x1 * c);
  x0 = y0;
  x1 = y1;
}

inline TwoPi rope_two_pi() {
  // 2*pi to 64-bit long double precision, split into three floats.
  const long double tp = 6.283185307179586476925286766559005768L;
  TwoPi r;
  r.a = static_cast<float>(tp);
  r.b = static_cast<float>(tp - static_cast<long double>(r.a));
  r.c = static_cast<float>(tp - static_cast<long double>(r.a) - static_cast<long double>(r.b));
  return r;
}

}  // namespace nomas
