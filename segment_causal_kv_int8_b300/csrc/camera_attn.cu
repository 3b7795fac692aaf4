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
// HBM-bound: each query row is read once and its output written once; the
// frame's camera K/V (n_cam x 4 heads x 512 B per CTA) sit in shared memory.
// 16 lanes own a row (8 values each); a CTA covers 16 tokens of one latent
// frame and 4 heads, i.e. 64 rows, four per 16-lane group (one head, four
// tokens), whose loads are all issued before any arithmetic.  Scores are
// reduced over the 16 lanes with four shuffles, the four rows' reductions
// interleaved; the softmax over the n_cam scores runs online in float32 (log2
// domain, ex2.approx), with packed f32x2 arithmetic for the dot products and
// the output update.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "checks.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace nomas {
namespace {

constexpr int kCamTokens = 16;      // tokens per CTA
constexpr int kCamHeads = 4;        // heads per CTA
constexpr int kCamRowsPerGroup = kCamTokens * kCamHeads / 16;

__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(u[e] << 16);
    x[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(256) camera_attn_kernel(const __grid_constant__ CameraAttnParams p) {
  extern __shared__ uint4 s_cam[];  // [2][n_cam][kCamHeads][16] uint4: K then V
  const int f = blockIdx.y;
  const int h0 = blockIdx.z * kCamHeads;
  const int nh = min(kCamHeads, p.heads - h0);
  const int cam_vecs = p.n_cam * kCamHeads * 16;
  const int g = threadIdx.x & 15;
  const int grp = threadIdx.x >> 4;  // 0..15
  const unsigned gmask = 0xFFFFu << (threadIdx.x & 16);
  // Rows of this 16-lane group: one head (h0 + grp % kCamHeads) and tokens
  // t0 + grp / kCamHeads + 4 r; their query loads go out first.
  const int hh = grp % kCamHeads;
  const int tok0 = blockIdx.x * kCamTokens + grp / kCamHeads;
  uint4 qw[kCamRowsPerGroup];
#pragma unroll
  for (int r = 0; r < kCamRowsPerGroup; ++r) {
    const int tok = tok0 + 4 * r;
    qw[r] = make_uint4(0u, 0u, 0u, 0u);
    if (tok < p.tpf && hh < nh &&
        in_bounds(((static_cast<long long>(f) * p.tpf + tok) * p.heads + h0 + hh) * 128 + 8 * g, 8,
                  static_cast<long long>(p.frames) * p.tpf * p.heads * 128, p.err))
      qw[r] = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                             ((static_cast<size_t>(f) * p.tpf + tok) * p.heads + h0 + hh) * 128)[g];
  }
  // Stage the frame's camera K and V for this CTA's heads.
  for (int i = threadIdx.x; i < 2 * cam_vecs; i += blockDim.x) {
    const int kv = i / cam_vecs, r = i - kv * cam_vecs;
    const int j = r / (kCamHeads * 16), ch = (r / 16) % kCamHeads, c = r % 16;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (ch < nh && in_bounds(((static_cast<long long>(f) * p.n_cam + j) * p.heads + h0 + ch) * 128 + 8 * c, 8,
                             static_cast<long long>(p.frames) * p.n_cam * p.heads * 128, p.err)) {
      const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(kv ? p.v_cam : p.k_cam);
      w = reinterpret_cast<const uint4*>(src + ((static_cast<size_t>(f) * p.n_cam + j) * p.heads + h0 + ch) * 128)[c];
    }
    s_cam[i] = w;
  }
  __syncthreads();
  float q[kCamRowsPerGroup][8], o[kCamRowsPerGroup][8], m[kCamRowsPerGroup], l[kCamRowsPerGroup];
#pragma unroll
  for (int r = 0; r < kCamRowsPerGroup; ++r) {
    unpack8(qw[r], q[r]);
    m[r] = -INFINITY;
    l[r] = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[r][e] = 0.0f;
  }
  // The group's rows share a head, so each camera token's K and V slice is
  // read once for all of them, and their score reductions interleave.
  for (int j = 0; j < p.n_cam; ++j) {
    float k[8], v[8];
    unpack8(s_cam[(j * kCamHeads + hh) * 16 + g], k);
    unpack8(s_cam[cam_vecs + (j * kCamHeads + hh) * 16 + g], v);
    float sc[kCamRowsPerGroup];
#pragma unroll
    for (int r = 0; r < kCamRowsPerGroup; ++r) {
      // two interleaved partial sums in one packed f32x2 accumulator
      uint64_t acc = f2_mul(f2_pack(q[r][0], q[r][1]), f2_pack(k[0], k[1]));
#pragma unroll
      for (int e = 2; e < 8; e += 2) acc = f2_fma(f2_pack(q[r][e], q[r][e + 1]), f2_pack(k[e], k[e + 1]), acc);
      float a0, a1;
      f2_unpack(acc, a0, a1);
      sc[r] = a0 + a1;
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1)
#pragma unroll
      for (int r = 0; r < kCamRowsPerGroup; ++r) sc[r] += __shfl_xor_sync(gmask, sc[r], off);
#pragma unroll
    for (int r = 0; r < kCamRowsPerGroup; ++r) {
      const float s = sc[r] * p.scale_log2;
      const float m_new = fmaxf(m[r], s);
      const float alpha = fast_exp2(m[r] - m_new);  // 0 on the first camera token (m = -inf)
      const float pj = fast_exp2(s - m_new);
      l[r] = fmaf(l[r], alpha, pj);
      const uint64_t a2 = f2_pack(alpha, alpha), p2 = f2_pack(pj, pj);
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const uint64_t o2 = f2_fma(f2_pack(o[r][e], o[r][e + 1]), a2, f2_mul(p2, f2_pack(v[e], v[e + 1])));
        f2_unpack(o2, o[r][e], o[r][e + 1]);
      }
      m[r] = m_new;
    }
  }
#pragma unroll
  for (int r = 0; r < kCamRowsPerGroup; ++r) {
    const int tok = tok0 + 4 * r;
    if (tok < p.tpf && hh < nh &&
        in_bounds(((static_cast<long long>(f) * p.tpf + tok) * p.heads + h0 + hh) * 128 + 8 * g, 8,
                  static_cast<long long>(p.frames) * p.tpf * p.heads * 128, p.err)) {
      const float inv = 1.0f / l[r];
      uint4 w;
      uint32_t* u = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 t = __floats2bfloat162_rn(o[r][2 * e] * inv, o[r][2 * e + 1] * inv);
        u[e] = *reinterpret_cast<const uint32_t*>(&t);
      }
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                               ((static_cast<size_t>(f) * p.tpf + tok) * p.heads + h0 + hh) * 128)[g] = w;
    }
  }
}

}  // namespace

cudaError_t launch_camera_attn(const CameraAttnParams& p, cudaStream_t stream) {
  if (p.frames <= 0 || p.tpf <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((p.tpf + kCamTokens - 1) / kCamTokens), static_cast<unsigned>(p.frames),
                  static_cast<unsigned>((p.heads + kCamHeads - 1) / kCamHeads));
  if (grid.y > 65535 || grid.z > 65535) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(2) * p.n_cam * kCamHeads * 16 * sizeof(uint4);
  camera_attn_kernel<<<grid, 256, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nomas
