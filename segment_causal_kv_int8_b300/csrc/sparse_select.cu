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
// Three small kernels: mean key per (head, tile) of the resident cache
// (dequantised for INT8), mean query per (head, group), and the ranking.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace nomas {
namespace {

// One CTA per (tile, head); thread d sums dimension d over the tile's rows.
template <bool kInt8>
__global__ void __launch_bounds__(128) tile_means_kernel(const SparseSelectParams p) {
  const int t = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const long long plane = static_cast<long long>(p.block_head_base + h) * p.cap_slots;
  const int r0 = t * 128, r1 = min(p.nc, r0 + 128);
  float acc = 0.0f;
  for (int r = r0; r < r1; ++r) {
    float x;
    if constexpr (kInt8) {
      x = static_cast<float>(static_cast<const int8_t*>(p.kcache)[(plane + r) * 128 + d]) * p.kscale[plane + r];
    } else {
      x = __bfloat162float(static_cast<const __nv_bfloat16*>(p.kcache)[(plane + r) * 128 + d]);
    }
    acc += x;
  }
  p.kbar[(static_cast<size_t>(h) * p.n_tiles + t) * 128 + d] = acc / static_cast<float>(r1 - r0);
}

// One CTA per (group, head): mean of the group's query rows.
__global__ void __launch_bounds__(128) group_means_kernel(const SparseSelectParams p) {
  const int g = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const int r0 = g * 512, r1 = min(p.nq, r0 + 512);
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
  float acc = 0.0f;
  for (int r = r0; r < r1; ++r) acc += __bfloat162float(q[(static_cast<size_t>(r) * p.heads + h) * 128 + d]);
  p.qbar[(static_cast<size_t>(h) * p.n_groups + g) * 128 + d] = acc / static_cast<float>(r1 - r0);
}

// One CTA per (group, head): scores of every tile, rank (score descending,
// index ascending), keep ranks below k, write them in increasing order.
__global__ void __launch_bounds__(256) rank_kernel(const SparseSelectParams p) {
  extern __shared__ float s_scores[];  // [n_tiles]
  __shared__ float s_q[128];
  const int g = blockIdx.x, h = blockIdx.y;
  if (threadIdx.x < 128) s_q[threadIdx.x] = p.qbar[(static_cast<size_t>(h) * p.n_groups + g) * 128 + threadIdx.x];
  __syncthreads();
  for (int t = threadIdx.x; t < p.n_tiles; t += blockDim.x) {
    const float* kb = p.kbar + (static_cast<size_t>(h) * p.n_tiles + t) * 128;
    float acc = 0.0f;
    for (int d = 0; d < 128; ++d) acc = fmaf(s_q[d], kb[d], acc);
    s_scores[t] = acc;
  }
  __syncthreads();
  unsigned char* keep = reinterpret_cast<unsigned char*>(s_scores + p.n_tiles);
  for (int t = threadIdx.x; t < p.n_tiles; t += blockDim.x) {
    const float st = s_scores[t];
    int rank = 0;
    for (int u = 0; u < p.n_tiles; ++u) {
      const float su = s_scores[u];
      rank += (su > st || (su == st && u < t)) ? 1 : 0;
    }
    keep[t] = rank < p.keep ? 1 : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const size_t hg = static_cast<size_t>(h) * p.n_groups + g;
    int* out = p.tiles + hg * p.max_keep;
    int c = 0;
    for (int t = 0; t < p.n_tiles && c < p.keep; ++t)
      if (keep[t]) out[c++] = t;
    p.counts[hg] = c;
  }
}

}  // namespace

size_t sparse_select_smem(int n_tiles) { return static_cast<size_t>(n_tiles) * 5; }

cudaError_t launch_sparse_select(bool int8_cache, const SparseSelectParams& p, cudaStream_t stream) {
  if (p.n_tiles > 0) {
    const dim3 tg(p.n_tiles, p.heads);
    if (int8_cache)
      tile_means_kernel<true><<<tg, 128, 0, stream>>>(p);
    else
      tile_means_kernel<false><<<tg, 128, 0, stream>>>(p);
  }
  const dim3 gg(p.n_groups, p.heads);
  group_means_kernel<<<gg, 128, 0, stream>>>(p);
  if (p.n_tiles > 0) rank_kernel<<<gg, 256, sparse_select_smem(p.n_tiles), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nomas
