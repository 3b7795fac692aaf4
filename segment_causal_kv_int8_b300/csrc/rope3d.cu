// rope3d.cu - in-place 3D rotary position embedding of the video rows of Q and K.
//
// "3D RoPE" over (latent frame, h, w) is part of the model card (Hy-Nomas auf
// einer RTX 4090, section "Modell und Dateien").  The head dimension splits
// into contiguous chunks per axis; pair (x[o+2i], x[o+2i+1]) of the chunk of
// axis a rotates by pos_a * f_{a,i}, f_{a,i} = theta^(-2i/d_a).
//
// HBM-bound elementwise kernel: one warp per (tensor, token).  A token's video
// row of Q (or K) is heads head rows of 128 elements, back to back, so a warp
// streams it as 16-byte vectors with 512-byte coalesced accesses, and every
// vector of a lane holds the same rotary pairs.  A CTA computes the cos/sin of
// its tokens' pairs into shared memory (angle arithmetic in rope_math.cuh;
// one value per (token, pair), shared by every head and by Q and K) while its
// first loads are in flight; each lane then reads its pairs' values once.  The
// cos/sin of a pair depend only on its position and frequency, so the rotation
// is bit for bit what per-element evaluation gives.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "checks.cuh"
#include "kernels.h"
#include "rope_math.cuh"

namespace nomas {
namespace {

// Rotates the pairs of one 16-byte vector by the (cos, sin) in cc/ss.
template <bool kBF16, typename Vec>
__device__ __forceinline__ void rotate_vec(Vec& v, const float (&cc)[kBF16 ? 4 : 2], const float (&ss)[kBF16 ? 4 : 2]) {
  if constexpr (kBF16) {
    uint32_t* u = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float x0 = __uint_as_float(u[e] << 16);
      float x1 = __uint_as_float(u[e] & 0xFFFF0000u);
      rope_rotate_pair(x0, x1, cc[e], ss[e]);
      __nv_bfloat162 t2 = __floats2bfloat162_rn(x0, x1);
      u[e] = *reinterpret_cast<const uint32_t*>(&t2);
    }
  } else {
    rope_rotate_pair(v.x, v.y, cc[0], ss[0]);
    rope_rotate_pair(v.z, v.w, cc[1], ss[1]);
  }
}

// One warp per (tensor, token).  A token's video row of Q (or K) is heads
// head rows of 128 elements, back to back: V = heads * VPR 16-byte vectors.
// Lane l takes vectors l, l + 32, l + 64, ..., so each warp access moves 512
// contiguous bytes, and since 32 is a multiple of VPR every vector of a lane
// holds the same rotary pairs: the lane reads its cos/sin once per token and
// keeps them in registers.  Up to kTokBatch vectors per lane are loaded before
// any is rotated; the CTA's first loads go out before it computes the cos/sin
// table of its tokens.  With two tensors, warps 2t and 2t + 1 take Q and K of
// token t of the CTA, so both use one table row.  CTAs are four warps, so a
// barrier couples few warps and a finished CTA is replaced quickly.
constexpr int kTokBatch = 8;     // vectors per lane in flight
constexpr int kTokThreads = 128;  // four warps per CTA

template <bool kBF16, bool kTwo>
__global__ void __launch_bounds__(kTokThreads, 8) rope3d_token_kernel(char* __restrict__ q, char* __restrict__ k,
                                                              const __grid_constant__ RopeParams p, TwoPi tp) {
  constexpr int VPR = kBF16 ? 16 : 32;  // vectors per head row
  constexpr int PPV = kBF16 ? 4 : 2;    // rotary pairs per vector
  constexpr int ESZ = kBF16 ? 2 : 4;
  constexpr int TPC = kTwo ? 2 : 4;     // tokens per CTA
  using Vec = typename std::conditional<kBF16, uint4, float4>::type;
  __shared__ __align__(16) float2 cs[TPC * 64];  // (cos, sin) of [token of the CTA][pair], interleaved
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tl = kTwo ? (warp >> 1) : warp;
  const int tok0 = blockIdx.x * TPC;
  const int tok = tok0 + tl;
  const int g = lane & (VPR - 1);  // the lane's pair group
  bool rotated = false;
#pragma unroll
  for (int e = 0; e < PPV; ++e) rotated |= p.axis[g * PPV + e] >= 0;
  const bool active = tok < p.n_video && rotated;
  const int V = p.heads * VPR;
  const long long row_elem = static_cast<long long>(tok) * p.row_stride;
  char* const row = ((kTwo && (warp & 1)) ? k : q) + row_elem * ESZ;
  Vec w[kTokBatch];
  const auto live = [&](int j) { return j < V && in_bounds(row_elem + j * (16 / ESZ), 16 / ESZ, p.extent, p.err); };
  const auto load = [&](int j0) {
#pragma unroll
    for (int u = 0; u < kTokBatch; ++u) {
      const int j = j0 + lane + 32 * u;
      if (live(j)) w[u] = *reinterpret_cast<const Vec*>(row + 16LL * j);
    }
  };
  if (active) load(0);
  for (int e = tid; e < TPC * 64; e += kTokThreads) {
    const int t = e >> 6, pair = e & 63;
    const int a = p.axis[pair];
    const int tk = tok0 + t;
    float c = 1.0f, sn = 0.0f;
    if (a >= 0 && tk < p.n_video) {
      const int frame = fast_div(tk, p.tpf_div);
      const int within = tk - frame * p.tpf;
      const int hrow = fast_div(within, p.gw_div);
      // positions stay below 2^24 (checked by the caller): 32-bit integer to float is exact
      const float pos = static_cast<float>(a == 0 ? static_cast<int>(p.t0) + frame
                                                  : (a == 1 ? hrow : within - hrow * p.grid_w));
      sincosf(rope_reduced_angle(pos, p.f_hi[pair], p.f_lo[pair], tp), &sn, &c);
    }
    // pair group g's chunks h2 = 0, 1 sit in rows of 16 consecutive groups
    cs[t * 64 + ((pair % PPV) >> 1) * 32 + 2 * (pair / PPV) + (pair & 1)] = make_float2(c, sn);
  }
  __syncthreads();
  if (!active) return;
  float cc[PPV], ss[PPV];
#pragma unroll
  for (int h2 = 0; h2 < PPV / 2; ++h2) {
    const float4 t4 = *reinterpret_cast<const float4*>(&cs[tl * 64 + h2 * 32 + 2 * g]);
    cc[2 * h2] = t4.x;
    ss[2 * h2] = t4.y;
    cc[2 * h2 + 1] = t4.z;
    ss[2 * h2 + 1] = t4.w;
  }
  for (int j0 = 0; j0 < V; j0 += 32 * kTokBatch) {
    if (j0 > 0) load(j0);
#pragma unroll
    for (int u = 0; u < kTokBatch; ++u) {
      const int j = j0 + lane + 32 * u;
      if (!live(j)) continue;
      rotate_vec<kBF16>(w[u], cc, ss);
      *reinterpret_cast<Vec*>(row + 16LL * j) = w[u];
    }
  }
}

}  // namespace

cudaError_t launch_rope3d(bool bf16_io, void* q, void* k, const RopeParams& p, cudaStream_t stream) {
  if (p.n_video <= 0) return cudaSuccess;
  // vector indices of a token row and token indices of a CTA stay in int
  if (p.heads <= 0 || p.heads > kRopeMaxHeads || p.n_video > kRopeMaxVideoRows) return cudaErrorInvalidValue;
  const TwoPi tp = rope_two_pi();
  const int tpc = k ? 2 : 4;  // tokens per CTA: Q and K of 2, or Q of 4
  const unsigned grid = static_cast<unsigned>((p.n_video + tpc - 1) / tpc);
  char* qc = static_cast<char*>(q);
  char* kc = static_cast<char*>(k);
  if (bf16_io) {
    if (k)
      rope3d_token_kernel<true, true><<<grid, kTokThreads, 0, stream>>>(qc, kc, p, tp);
    else
      rope3d_token_kernel<true, false><<<grid, kTokThreads, 0, stream>>>(qc, kc, p, tp);
  } else {
    if (k)
      rope3d_token_kernel<false, true><<<grid, kTokThreads, 0, stream>>>(qc, kc, p, tp);
    else
      rope3d_token_kernel<false, false><<<grid, kTokThreads, 0, stream>>>(qc, kc, p, tp);
  }
  return cudaGetLastError();
}

}  // namespace nomas
