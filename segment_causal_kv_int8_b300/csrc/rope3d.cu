// rope3d.cu - in-place 3D rotary position embedding of the video rows of Q and K.
//
// "3D RoPE" over (latent frame, h, w) is part of the model card (Hy-Nomas auf
// einer RTX 4090, section "Modell und Dateien").  The head dimension splits
// into contiguous chunks per axis; pair (x[o+2i], x[o+2i+1]) of the chunk of
// axis a rotates by pos_a * f_{a,i}, f_{a,i} = theta^(-2i/d_a).
//
// HBM-bound elementwise kernel.  The grid is one resident wave of CTAs, each
// taking an equal run of consecutive tokens (no partial last wave).  A CTA
// first computes the cos/sin of every (token, pair) of its run into shared
// memory (angle arithmetic in rope_math.cuh; shared by every head and by Q
// and K), then streams the rows of Q and K as 16-byte vectors.  A thread's
// vectors always hold the same rotary pairs of some head, so its table reads
// are one or two 16-byte loads.  The cos/sin of a pair depend only on its
// position and frequency, so the rotation is bit for bit what per-element
// evaluation gives.
//
// Two forms: rope3d_async_kernel (token rows of up to 1024 vectors) copies
// each thread's vectors through a cp.async ring in shared memory;
// rope3d_run_kernel (wider rows) double-buffers items of two tokens' vectors
// in registers, the first item's loads issued before the table is computed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "checks.cuh"
#include "kernels.h"
#include "rope_math.cuh"

namespace nomas {
namespace {

constexpr int kRunMax = 32;  // tokens of one table fill (32 x 64 pairs x 8 B = 16 KB of shared memory)

// Streams the video rows of Q and K (row_stride elements apart) as 16-byte
// vectors: V = heads * VPR vectors per token, VPR = 16 (bf16) or 32 (f32).
template <bool kBF16>
__global__ void __launch_bounds__(256) rope3d_run_kernel(void* __restrict__ q, void* __restrict__ k,
                                                         const __grid_constant__ RopeParams p, TwoPi tp,
                                                         int run_tokens) {
  constexpr int VPR = kBF16 ? 16 : 32;  // vectors per head row
  constexpr int PPV = kBF16 ? 4 : 2;    // rotary pairs per vector
  constexpr int ESZ = kBF16 ? 2 : 4;
  using Vec = typename std::conditional<kBF16, uint4, float4>::type;
  __shared__ __align__(16) float2 cs[kRunMax * 64];   // (cos, sin) of [token of the fill][pair]
  __shared__ int8_t axis_s[64];
  const int tid = threadIdx.x;
  if (tid < 64) axis_s[tid] = p.axis[tid];
  const int tok_begin = blockIdx.x * run_tokens;
  const int tok_end = min(p.n_video, tok_begin + run_tokens);
  const int V = p.heads * VPR;
  // Fixed per thread: which tokens of a fill (t_off, t_off + tpi, ...) and
  // which vectors of a token row (rem, rem + 256, ...) it handles.
  const int tpi = V >= 256 ? 1 : 256 / V;   // tokens per pass of the CTA
  const int t_off = V >= 256 ? 0 : tid / V;
  const int rem0 = V >= 256 ? tid : tid - t_off * V;
  const bool active = t_off < tpi;
  const int g = rem0 & (VPR - 1);           // the thread's pair group
  __syncthreads();
  bool rotated = false;
#pragma unroll
  for (int e = 0; e < PPV; ++e) rotated |= axis_s[g * PPV + e] >= 0;
  const int nt = (k != nullptr) ? 2 : 1;
  constexpr int U = 2;  // tokens of one item: U vectors of Q and U of K per thread
  const int nrem = active ? (V - rem0 + 255) / 256 : 0;  // vectors of a token row this thread visits
  // Item i of a fill: tokens t_off + (i / nrem) * U * tpi + u * tpi (u < U),
  // vector rem0 + 256 * (i % nrem) of each token row.
  auto locate = [&](int f0, int nf, int i, int u, int& tl, long long& off) {
    const int a = i / nrem, b = i - (i / nrem) * nrem;
    tl = t_off + a * U * tpi + u * tpi;
    off = static_cast<long long>(f0 + tl) * p.row_stride + ((rem0 + 256 * b) / VPR) * 128 + g * (16 / ESZ);
    return tl < nf && in_bounds(off, 16 / ESZ, p.extent, p.err);
  };
  auto load = [&](int f0, int nf, int i, Vec (&w)[2][U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      int tl;
      long long off;
      if (!locate(f0, nf, i, u, tl, off)) continue;
#pragma unroll
      for (int which = 0; which < 2; ++which)
        if (which < nt) w[which][u] = reinterpret_cast<const Vec*>(static_cast<const char*>(which ? k : q))[off * ESZ / 16];
    }
  };
  auto rotate_store = [&](int f0, int nf, int i, const Vec (&w)[2][U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      int tl;
      long long off;
      if (!locate(f0, nf, i, u, tl, off)) continue;
      const float4* tab = reinterpret_cast<const float4*>(&cs[tl * 64 + g * PPV]);
      float cc[PPV], ss[PPV];
#pragma unroll
      for (int h2 = 0; h2 < PPV / 2; ++h2) {
        const float4 t4 = tab[h2];
        cc[2 * h2] = t4.x;
        ss[2 * h2] = t4.y;
        cc[2 * h2 + 1] = t4.z;
        ss[2 * h2 + 1] = t4.w;
      }
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        if (which >= nt) break;
        Vec o;
        if constexpr (kBF16) {
          const uint32_t* v = reinterpret_cast<const uint32_t*>(&w[which][u]);
          uint32_t* ov = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x0 = __uint_as_float(v[e] << 16);
            float x1 = __uint_as_float(v[e] & 0xFFFF0000u);
            rope_rotate_pair(x0, x1, cc[e], ss[e]);
            __nv_bfloat162 t2 = __floats2bfloat162_rn(x0, x1);
            ov[e] = *reinterpret_cast<const uint32_t*>(&t2);
          }
        } else {
          const float* v = reinterpret_cast<const float*>(&w[which][u]);
          float x[4] = {v[0], v[1], v[2], v[3]};
          rope_rotate_pair(x[0], x[1], cc[0], ss[0]);
          rope_rotate_pair(x[2], x[3], cc[1], ss[1]);
          o = make_float4(x[0], x[1], x[2], x[3]);
        }
        reinterpret_cast<Vec*>(static_cast<char*>(which ? k : q))[off * ESZ / 16] = o;
      }
    }
  };
  for (int f0 = tok_begin; f0 < tok_end; f0 += kRunMax) {
    const int nf = min(kRunMax, tok_end - f0);
    const int n_items = (active && rotated && nf > t_off) ? ((nf - t_off + U * tpi - 1) / (U * tpi)) * nrem : 0;
    Vec wa[2][U], wb[2][U];
    // The first item's loads go out before the table is computed.
    if (n_items > 0) load(f0, nf, 0, wa);
    // cos/sin of the fill's tokens: entry (t, pair) at t * 64 + pair
    for (int e = tid; e < nf * 64; e += 256) {
      const int t = e >> 6, pair = e & 63;
      const int a = axis_s[pair];
      float c = 1.0f, sn = 0.0f;
      if (a >= 0) {
        const int tok = f0 + t;
        const int frame = fast_div(tok, p.tpf_div);
        const int within = tok - frame * p.tpf;
        const int row = fast_div(within, p.gw_div);
        // positions stay below 2^24 (checked by the caller): 32-bit integer to float is exact
        const float pos = static_cast<float>(a == 0 ? static_cast<int>(p.t0) + frame
                                                    : (a == 1 ? row : within - row * p.grid_w));
        sincosf(rope_reduced_angle(pos, p.f_hi[pair], p.f_lo[pair], tp), &sn, &c);
      }
      cs[e] = make_float2(c, sn);
    }
    __syncthreads();
    // Two buffers: the next item's loads are in flight while this one rotates.
    for (int i = 0; i < n_items; i += 2) {
      if (i + 1 < n_items) load(f0, nf, i + 1, wb);
      rotate_store(f0, nf, i, wa);
      if (i + 2 < n_items) load(f0, nf, i + 2, wa);
      if (i + 1 < n_items) rotate_store(f0, nf, i + 1, wb);
    }
    __syncthreads();  // the table's readers are done before the next fill rewrites it
  }
}

// ---------------------------------------------------------------- async-copy form
// Each CTA takes an equal run of tokens and streams it in items of T tokens
// (T * heads * 16 vectors of each of Q and K, at most 4 vectors per thread per
// tensor).  Every thread fetches its own vectors of an item with 16-byte
// cp.async copies into a 3-stage shared-memory ring, so up to 3 items (24
// copies, 384 bytes per thread) are in flight without holding registers, and
// reads them back itself once its copy group has landed (no barrier): rotate,
// then store to global memory.  The item layout is the same for every item,
// so a thread's (token, head, pair group) of each vector, and its byte offset
// within an item, are computed once; an item adds one 32-bit offset.  Q and K
// are separate template cases, so no pointer is chosen at run time.
constexpr int kAsyncStages = 3;
constexpr int kAsyncVecs = 1024;  // vectors per tensor per item (16 KB)

__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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

template <bool kBF16, bool kTwo>
__global__ void __launch_bounds__(256) rope3d_async_kernel(char* __restrict__ q, char* __restrict__ k,
                                                           const __grid_constant__ RopeParams p, TwoPi tp,
                                                           int run_tokens, int item_tokens) {
  constexpr int VPR = kBF16 ? 16 : 32;  // vectors per head row
  constexpr int PPV = kBF16 ? 4 : 2;    // rotary pairs per vector
  constexpr int ESZ = kBF16 ? 2 : 4;
  constexpr int M = kAsyncVecs / 256;   // vectors per thread per tensor per item
  using Vec = typename std::conditional<kBF16, uint4, float4>::type;
  extern __shared__ __align__(16) uint8_t asm_raw[];
  const Vec* ring = reinterpret_cast<const Vec*>(asm_raw);                            // [stage][tensor][kAsyncVecs]
  float2* cs = reinterpret_cast<float2*>(asm_raw + kAsyncStages * 2 * kAsyncVecs * 16);  // [kRunMax][64]
  __shared__ int8_t axis_s[64];
  const int tid = threadIdx.x;
  if (tid < 64) axis_s[tid] = p.axis[tid];
  const int tok_begin = blockIdx.x * run_tokens;
  const int tok_end = min(p.n_video, tok_begin + run_tokens);
  const int V = p.heads * VPR;
  const int T = item_tokens;                           // T * V <= kAsyncVecs
  const int g = tid & (VPR - 1);                       // the thread's pair group (fixed: 256 % VPR == 0)
  const uint32_t row_bytes = static_cast<uint32_t>(p.row_stride) * ESZ;  // kRunMax rows stay below 2^31 bytes
  const uint32_t item_bytes = static_cast<uint32_t>(T) * row_bytes;
  int tl_m[M];          // token within the item (T: this slot is unused)
  uint32_t boff_m[M];   // byte offset within the item
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int j = tid + 256 * m;
    const int tl = j / V;
    tl_m[m] = j < T * V ? tl : T;
    boff_m[m] = static_cast<uint32_t>(tl) * row_bytes + static_cast<uint32_t>(((j - tl * V) / VPR) * 128 * ESZ + g * 16);
  }
  const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(asm_raw)) + 16u * tid;
  __syncthreads();
  bool rotated = false;
#pragma unroll
  for (int e = 0; e < PPV; ++e) rotated |= axis_s[g * PPV + e] >= 0;
  for (int f0 = tok_begin; f0 < tok_end; f0 += kRunMax) {
    const int nf = min(kRunMax, tok_end - f0);
    const int n_items = (nf + T - 1) / T;
    const long long fill_elem = static_cast<long long>(f0) * p.row_stride;
    char* const qf = q + fill_elem * ESZ;
    char* const kf = kTwo ? k + fill_elem * ESZ : nullptr;
    // The element offset a slot's vector starts at (bounds-checked build only).
    const auto elem_of = [&](int tl, int m) {
      return static_cast<long long>(f0 + tl) * p.row_stride + (boff_m[m] - tl_m[m] * row_bytes) / ESZ;
    };
    int stage_w = 0, stage_r = 0;
    // Item i uses every slot of every thread when the items tile the ring
    // exactly and i is not the fill's partial last item: such items take a
    // path without per-slot checks.
    const bool dense = T * V == kAsyncVecs;
    const auto fetch = [&](int i) {
      if (rotated && i < n_items) {
        const uint32_t st = ring_s + stage_w * (2 * kAsyncVecs * 16);
        const uint32_t ib = static_cast<uint32_t>(i) * item_bytes;
        const char* qb = qf + ib;
        const char* kb = kTwo ? kf + ib : nullptr;
        const auto copy_slot = [&](int m) {
          cp_async16(st + m * 256 * 16, qb + boff_m[m]);
          if constexpr (kTwo) cp_async16(st + (kAsyncVecs + m * 256) * 16, kb + boff_m[m]);
        };
        if (dense && (i + 1) * T <= nf) {
#pragma unroll
          for (int m = 0; m < M; ++m) {
            if (!in_bounds(elem_of(i * T + tl_m[m], m), 16 / ESZ, p.extent, p.err)) continue;
            copy_slot(m);
          }
        } else {
#pragma unroll
          for (int m = 0; m < M; ++m) {
            const int tl = i * T + tl_m[m];
            if (tl_m[m] >= T || tl >= nf) continue;
            if (!in_bounds(elem_of(tl, m), 16 / ESZ, p.extent, p.err)) continue;
            copy_slot(m);
          }
        }
      }
      cp_async_commit();  // one group per item, empty or not, so the group count stays uniform
      stage_w = stage_w == kAsyncStages - 1 ? 0 : stage_w + 1;
    };
    for (int i = 0; i < kAsyncStages - 1; ++i) fetch(i);
    // cos/sin of the fill's tokens while the first items are in flight
    for (int e = tid; e < nf * 64; e += 256) {
      const int t = e >> 6, pair = e & 63;
      const int a = axis_s[pair];
      float c = 1.0f, sn = 0.0f;
      if (a >= 0) {
        const int tok = f0 + t;
        const int frame = fast_div(tok, p.tpf_div);
        const int within = tok - frame * p.tpf;
        const int row = fast_div(within, p.gw_div);
        // positions stay below 2^24 (checked by the caller): 32-bit integer to float is exact
        const float pos = static_cast<float>(a == 0 ? static_cast<int>(p.t0) + frame
                                                    : (a == 1 ? row : within - row * p.grid_w));
        sincosf(rope_reduced_angle(pos, p.f_hi[pair], p.f_lo[pair], tp), &sn, &c);
      }
      // Stored so that each pair group's 16-byte table chunks h2 = 0, 1 sit in
      // rows of 16 consecutive groups: a warp's table reads are contiguous
      // 256-byte spans, free of bank conflicts.
      cs[t * 64 + ((pair % PPV) >> 1) * 32 + 2 * (pair / PPV) + (pair & 1)] = make_float2(c, sn);
    }
    __syncthreads();
    for (int i = 0; i < n_items; ++i) {
      fetch(i + kAsyncStages - 1);
      cp_async_wait<kAsyncStages - 1>();  // this thread's copies of item i have landed
      const Vec* st = ring + stage_r * 2 * kAsyncVecs + tid;
      stage_r = stage_r == kAsyncStages - 1 ? 0 : stage_r + 1;
      if (!rotated) continue;
      const uint32_t ib = static_cast<uint32_t>(i) * item_bytes;
      char* qb = qf + ib;
      char* kb = kTwo ? kf + ib : nullptr;
      const auto rotate_slot = [&](int m, int tl) {
        float cc[PPV], ss[PPV];
#pragma unroll
        for (int h2 = 0; h2 < PPV / 2; ++h2) {
          const float4 t4 = *reinterpret_cast<const float4*>(&cs[tl * 64 + h2 * 32 + 2 * g]);
          cc[2 * h2] = t4.x;
          ss[2 * h2] = t4.y;
          cc[2 * h2 + 1] = t4.z;
          ss[2 * h2 + 1] = t4.w;
        }
        Vec vq = st[256 * m];
        rotate_vec<kBF16>(vq, cc, ss);
        *reinterpret_cast<Vec*>(qb + boff_m[m]) = vq;
        if constexpr (kTwo) {
          Vec vk = st[kAsyncVecs + 256 * m];
          rotate_vec<kBF16>(vk, cc, ss);
          *reinterpret_cast<Vec*>(kb + boff_m[m]) = vk;
        }
      };
      if (dense && (i + 1) * T <= nf) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const int tl = i * T + tl_m[m];
          if (!in_bounds(elem_of(tl, m), 16 / ESZ, p.extent, p.err)) continue;
          rotate_slot(m, tl);
        }
      } else {
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const int tl = i * T + tl_m[m];
          if (tl_m[m] >= T || tl >= nf) continue;
          if (!in_bounds(elem_of(tl, m), 16 / ESZ, p.extent, p.err)) continue;
          rotate_slot(m, tl);
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // the table's readers are done before the next fill rewrites it
  }
}

constexpr int kAsyncSmem = kAsyncStages * 2 * kAsyncVecs * 16 + kRunMax * 64 * 8;

template <bool kBF16, bool kTwo>
cudaError_t launch_async(void* q, void* k, const RopeParams& p, const TwoPi& tp, int sms, int dev,
                         cudaStream_t stream) {
  static int configured[64] = {0};
  if (!configured[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(rope3d_async_kernel<kBF16, kTwo>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAsyncSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rope3d_async_kernel<kBF16, kTwo>, 256, kAsyncSmem) !=
          cudaSuccess ||
      per_sm <= 0) {
    (void)cudaGetLastError();
    per_sm = 1;
  }
  const long long slots = static_cast<long long>(sms) * per_sm;
  const int run = static_cast<int>((p.n_video + slots - 1) / slots);
  const unsigned grid = static_cast<unsigned>((p.n_video + run - 1) / run);
  const int item = kAsyncVecs / (p.heads * (kBF16 ? 16 : 32));
  rope3d_async_kernel<kBF16, kTwo><<<grid, 256, kAsyncSmem, stream>>>(static_cast<char*>(q), static_cast<char*>(k), p,
                                                                     tp, run, item);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope3d(bool bf16_io, void* q, void* k, const RopeParams& p, cudaStream_t stream) {
  if (p.n_video <= 0) return cudaSuccess;
  const TwoPi tp = rope_two_pi();
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  const int V = p.heads * (bf16_io ? 16 : 32);  // 16-byte vectors per token row
  const int esz = bf16_io ? 2 : 4;
  if (V <= kAsyncVecs && dev >= 0 && dev < 64 && p.row_stride * esz * kRunMax < (1ll << 31)) {
    // Async-copy form: one resident wave of CTAs (two per SM) with equal runs.
    return bf16_io ? (k ? launch_async<true, true>(q, k, p, tp, sms, dev, stream)
                        : launch_async<true, false>(q, k, p, tp, sms, dev, stream))
                   : (k ? launch_async<false, true>(q, k, p, tp, sms, dev, stream)
                        : launch_async<false, false>(q, k, p, tp, sms, dev, stream));
  }
  // Rows wider than one item (or a token stride too large for 32-bit offsets
  // within a fill): the register-streaming form.
  int per_sm = 0;
  const cudaError_t e = bf16_io ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rope3d_run_kernel<true>, 256, 0)
                                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rope3d_run_kernel<false>, 256, 0);
  if (e != cudaSuccess || per_sm <= 0) {
    (void)cudaGetLastError();
    per_sm = 3;
  }
  const long long slots = static_cast<long long>(sms) * per_sm;
  const int run = static_cast<int>((p.n_video + slots - 1) / slots);
  const unsigned grid = static_cast<unsigned>((p.n_video + run - 1) / run);
  if (bf16_io)
    rope3d_run_kernel<true><<<grid, 256, 0, stream>>>(q, k, p, tp, run);
  else
    rope3d_run_kernel<false><<<grid, 256, 0, stream>>>(q, k, p, tp, run);
  return cudaGetLastError();
}

}  // namespace nomas
