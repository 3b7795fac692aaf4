// kernels.h - internal interface between the C ABI shim and the CUDA kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nomas {

// ------------------------------------------------------------------ RoPE-3D
// Cache storage kinds: bf16 values, or one-byte codes (INT8 or FP8 E4M3)
// with one float32 scale per (block, head, token).
constexpr int kCacheBF16 = 0;
constexpr int kCacheInt8 = 1;
constexpr int kCacheFp8 = 2;

constexpr int kRopeMaxPairs = 64;  // head_dim 128 -> 64 rotary pairs
constexpr int kRopeMaxHeads = 1 << 19;            // heads * 32 vectors per token row stay in int
constexpr int kRopeMaxVideoRows = 0x7FFFFFFF - 8;  // token index of a CTA's last warp stays in int

// Division by a run-time constant d >= 1 as one multiply and one shift
// (division by invariant integers, Granlund and Montgomery, PLDI 1994): with
// 2^L >= d > 2^(L-1) and mul = ceil(2^(31+L) / d), which fits 32 bits,
// (n * mul) >> (31 + L) == n / d for every 0 <= n < 2^31.
struct FastDiv {
  uint32_t mul;
  uint32_t shift;
};
inline FastDiv make_fast_div(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  const uint64_t two = uint64_t(1) << (31 + l);
  return FastDiv{static_cast<uint32_t>((two + d - 1) / d), 31 + l};
}
#ifdef __CUDACC__
__device__ __forceinline__ int fast_div(int n, FastDiv f) {
  return static_cast<int>((static_cast<uint64_t>(static_cast<uint32_t>(n)) * f.mul) >> f.shift);
}
#endif

struct RopeParams {
  float f_hi[kRopeMaxPairs];     // frequency of each pair, high float
  float f_lo[kRopeMaxPairs];     // fl32(f - f_hi): low float of a two-float frequency
  int8_t axis[kRopeMaxPairs];    // 0 = t, 1 = h, 2 = w, -1 = not rotated
  int n_video;
  int heads;
  long long row_stride;          // elements between tokens
  int tpf;                       // grid_h * grid_w
  int grid_w;
  long long t0;
  long long extent;              // elements of Q (and K) the call may touch (checked build)
  uint32_t* err;                 // device error word (checked build)
  FastDiv tpf_div;               // n / tpf
  FastDiv gw_div;                // n / grid_w
};

cudaError_t launch_rope3d(bool bf16_io, void* q, void* k, const RopeParams& p, cudaStream_t stream);

// ------------------------------------------------------------------ append
struct AppendParams {
  const void* k;
  const void* v;
  long long block_stride;        // elements between blocks of the input
  int blocks;
  int heads;
  int tpf;
  int first_frame;               // first segment frame written
  int n_tokens;                  // tokens written = (n_frames - first_frame) * tpf
  int base_slot_frame;           // ring frame-slot of the first written frame
  int capacity_frames;
  long long cap_slots;           // capacity_frames * tpf
  void* ck;                      // cache K (int8 or bf16)
  void* cv;
  float* ks;                     // scales (int8 only)
  float* vs;
  int chunk_tokens;              // staged kernel: tokens per bulk-loaded chunk
  uint32_t* err;                 // device error word (staged kernel's bounded waits; checked build)
  long long src_extent;          // elements of each input tensor (checked build)
  long long cache_rows;          // blocks * heads * cap_slots rows of each cache tensor (checked build)
  FastDiv heads_div;             // n / heads
  FastDiv tpf_div;               // n / tpf
};

cudaError_t launch_append(bool f32_in, int kind, const AppendParams& p, int sms, cudaStream_t stream);
// Append with 3D RoPE of the K rows (rp.t0 = absolute frame of the first
// written frame; rp.tpf, rp.grid_w and the pair tables set).
cudaError_t launch_append_rope(bool f32_in, int kind, const AppendParams& p, const RopeParams& rp,
                               cudaStream_t stream);

// ------------------------------------------------------------------ BF16 expansion
// The resident window of a one-byte cache as BF16 values (slots [0, n_slots)
// of every (block, head) plane).
struct ExpandParams {
  const void* kc;                // codes [planes][cap_slots][128]
  const void* vc;
  const float* ks;               // scales [planes][cap_slots]
  const float* vs;
  void* ko;                      // bf16 [planes][cap_slots][128]
  void* vo;
  int planes;                    // blocks * heads
  long long cap_slots;
  long long n_slots;             // valid_frames * tpf
  uint32_t* err;                 // device error word (checked build)
};

cudaError_t launch_expand(int kind, const ExpandParams& p, cudaStream_t stream);

// ------------------------------------------------------------------ reset
cudaError_t launch_zero_fill(void* ptr, size_t bytes, cudaStream_t stream);

// ------------------------------------------------------------------ self-test
cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t stream);
bool bounds_checked_build();
cudaError_t launch_bounds_check_selftest(uint32_t* err, cudaStream_t stream);

// ------------------------------------------------------------------ sparse selection
struct SparseSelectParams {
  const void* kcache;            // cache K (int8 or bf16), [blocks*heads][cap_slots][128]
  const float* kscale;           // int8 only
  long long cap_slots;
  int block_head_base;
  int nc;                        // resident cache tokens
  int n_tiles;                   // ceil(nc / 128)
  const void* q;                 // bf16 [nq][heads][128]
  int nq;
  int heads;
  int n_groups;                  // ceil(nq / 512)
  int keep;                      // tiles kept per (head, group)
  int max_keep;                  // row length of tiles
  float* kbar;                   // workspace [heads][n_tiles][128]
  int* tiles;                    // [heads][n_groups][max_keep]
  int* counts;                   // [heads][n_groups]
  long long cache_rows;          // blocks * heads * cap_slots (checked build)
  uint32_t* err;                 // device error word (checked build)
};

size_t sparse_select_smem(int n_tiles);
cudaError_t launch_sparse_select(int kind, bool reuse_key_means, const SparseSelectParams& p,
                                 cudaStream_t stream);

// ------------------------------------------------------------------ camera cross-attention
struct CameraAttnParams {
  const void* q;                 // bf16 [frames * tpf][heads][128] (video rows)
  const void* k_cam;             // bf16 [frames][n_cam][heads][128]
  const void* v_cam;
  void* out;                     // bf16 [frames * tpf][heads][128]
  int frames;
  int tpf;
  int heads;
  int n_cam;                     // camera tokens per latent frame, 1 .. 16
  float scale_log2;              // softmax scale * log2(e)
  uint32_t* err;                 // device error word (checked build)
};

// TMA maps (128 dims, heads, tokens, frames) of the query rows and the output
// (tokens = tpf), and of the camera K and V (tokens = n_cam); boxes of 64
// dims x 1 head x 128 (16 for camera) tokens x 1 frame, 128-byte swizzle.
struct CameraTensorMaps {
  CUtensorMap q, k, v, o;
};

cudaError_t launch_camera_attn(const CameraTensorMaps& tm, const CameraAttnParams& p, cudaStream_t stream);

// ------------------------------------------------------------------ attention
struct AttnTensorMaps {
  CUtensorMap q, kcur, vcur, kc, vc;
};

// Work plan of one attention call.  A unit is one head x one block of 256
// query rows (BF16 cache) or one head x two adjacent such blocks (one-byte
// caches, whose CTA pairs share every dequantised tile), units ordered head
// by head.  Work items 0 .. n_full-1 are whole units (item i = unit i); every
// later unit is cut into tail_splits pieces of its key-tile range, whose
// partial outputs a combine pass merges in piece order.  With n_full = all
// units nothing is split; with n_full = 0 every unit is split evenly.
struct AttnParams {
  int nq;                        // current-segment tokens (queries and current keys)
  int nc;                        // resident cache tokens
  int heads;
  int n_cache_tiles;             // ceil(nc / 128)
  int n_cur_tiles;               // ceil(nq / 128)
  int units_per_head;            // query units per head
  int n_full;                    // whole-unit work items
  int tail_splits;               // pieces per unit after the whole ones (1 = none)
  int block_head_base;           // block * heads: row of the cache's [blocks*heads] axis
  float scale_log2;              // softmax scale * log2(e)
  __nv_bfloat16* out;
  float* lse;                    // nullable
  float* ws_o;                   // [pieces][ctas per unit][256][128] f32 partial outputs (tail_splits > 1)
  float* ws_lse;                 // [pieces][ctas per unit][256] partial log-sum-exps (natural log)
  const float* k_scale;          // int8 cache scales, [blocks*heads][scale_stride]
  const float* v_scale;
  long long scale_stride;        // cache slots per (block, head)
  uint32_t* err;                 // device error word
  const int* sparse_tiles;       // nullable: [heads][groups][max_keep] kept cache tiles, increasing
  const int* sparse_counts;      // [heads][groups]
  int max_keep;
  int n_groups;                  // 512-query groups (two 256-query blocks each)
  int block_heads;               // blocks * heads: planes of the cache (checked build)
  long long ws_rows;             // partial-output rows the workspace holds (checked build)
};

// n_items = n_full + (units - n_full) * tail_splits work items.
cudaError_t launch_segment_attn(int kind, const AttnTensorMaps& tm, const AttnParams& p, int n_items,
                                cudaStream_t stream);
// Merges the pieces of units n_full .. units-1 (tail_splits > 1 only).
cudaError_t launch_attn_combine(const AttnParams& p, int units, int ctas_per_unit, cudaStream_t stream);
// Work items of the attention kernel that run at once on the current device:
// SMs for a BF16 cache (one CTA per SM), co-resident CTA pairs for one-byte
// caches.  0 if the device cannot be queried.
int attn_concurrent_items(int kind);
int attn_smem_bytes(bool int8_cache);

}  // namespace nomas
