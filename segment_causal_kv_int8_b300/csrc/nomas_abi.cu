// nomas_abi.cu - the C ABI (include/nomas.h): argument validation, cache
// metadata, TMA descriptor encoding and kernel launches.  Host code only; no
// allocation, no synchronisation (except nomas_device_error, documented as
// synchronous).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/nomas.h"
#include "kernels.h"

#define NOMAS_API extern "C" __attribute__((visibility("default")))

namespace nomas {
namespace {

// Device-side error word: kernels that give up waiting store a status here.
__device__ uint32_t g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_err_ptr[kMaxDevices] = {nullptr};
int g_sm_count[kMaxDevices] = {0};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

nomas_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NOMAS_OK : NOMAS_ERR_CUDA; }

// Per-device state (error word address, SM count), set up on first use.
nomas_status device_state(uint32_t** err, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NOMAS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NOMAS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return NOMAS_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return NOMAS_ERR_CUDA;
    g_sm_count[dev] = n;
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  if (err) *err = g_err_ptr[dev];
  if (sms) *sms = g_sm_count[dev];
  return NOMAS_OK;
}

nomas_status encoder(EncodeTiledFn* fn) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || f == nullptr)
      return NOMAS_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(f);
  }
  *fn = g_encode;
  return NOMAS_OK;
}

// One-byte codes with per-row scales (INT8 or FP8) rather than bf16 values.
bool quantised(const nomas_kvcache* c) { return c->dtype == NOMAS_INT8 || c->dtype == NOMAS_FP8; }

int cache_kind(const nomas_kvcache* c) {
  return c->dtype == NOMAS_INT8 ? kCacheInt8 : (c->dtype == NOMAS_FP8 ? kCacheFp8 : kCacheBF16);
}

int64_t window_of(const nomas_kvcache* c) { return c->past_frames > 0 ? c->past_frames : c->capacity_frames; }

nomas_status validate_cache(const nomas_kvcache* c) {
  if (c == nullptr) return NOMAS_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->heads <= 0 || c->grid_h <= 0 || c->grid_w <= 0 || c->capacity_frames <= 0 ||
      c->past_frames < 0 || c->reserved != 0)
    return NOMAS_ERR_INVALID_ARG;
  if (c->head_dim <= 0) return NOMAS_ERR_INVALID_ARG;
  if (c->head_dim != 128) return NOMAS_ERR_UNSUPPORTED;
  if (c->past_frames > 0 && c->capacity_frames != c->past_frames) return NOMAS_ERR_INVALID_ARG;
  if (c->dtype != NOMAS_INT8 && c->dtype != NOMAS_BF16 && c->dtype != NOMAS_FP8) return NOMAS_ERR_INVALID_ARG;
  const int64_t tpf = static_cast<int64_t>(c->grid_h) * c->grid_w;
  const int64_t slots = tpf * c->capacity_frames;
  if (slots > (int64_t(1) << 30) || static_cast<int64_t>(c->num_blocks) * c->heads > (int64_t(1) << 24))
    return NOMAS_ERR_UNSUPPORTED;
  if (c->k == nullptr || c->v == nullptr || !aligned16(c->k) || !aligned16(c->v)) return NOMAS_ERR_INVALID_ARG;
  if (quantised(c)) {
    if (c->k_scale == nullptr || c->v_scale == nullptr) return NOMAS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(c->k_scale) & 3u) || (reinterpret_cast<uintptr_t>(c->v_scale) & 3u))
      return NOMAS_ERR_INVALID_ARG;
  }
  if (c->total_frames < 0 || c->valid_frames < 0) return NOMAS_ERR_INVALID_ARG;
  if (c->valid_frames != std::min<int64_t>(c->total_frames, window_of(c))) return NOMAS_ERR_INVALID_ARG;
  return NOMAS_OK;
}

nomas_status plan(const nomas_kvcache* c, int32_t n_frames, int32_t* first, int32_t* slot_frame,
                  int64_t* new_total, int32_t* new_valid) {
  if (n_frames < 0) return NOMAS_ERR_INVALID_ARG;
  const int64_t t = c->total_frames, w = window_of(c);
  if (c->past_frames == 0 && t + n_frames > c->capacity_frames) return NOMAS_ERR_CAPACITY;
  const int64_t f0 = std::max<int64_t>(0, n_frames - w);
  if (first) *first = static_cast<int32_t>(f0);
  if (slot_frame) *slot_frame = static_cast<int32_t>((t + f0) % c->capacity_frames);
  if (new_total) *new_total = t + n_frames;
  if (new_valid) *new_valid = static_cast<int32_t>(std::min<int64_t>(t + n_frames, w));
  return NOMAS_OK;
}

// Encode a 3D tiled TMA descriptor (dims/strides innermost first, strides in bytes).
nomas_status encode3d(CUtensorMap* m, CUtensorMapDataType dt, void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  EncodeTiledFn fn = nullptr;
  nomas_status st = encoder(&fn);
  if (st != NOMAS_OK) return st;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NOMAS_OK : NOMAS_ERR_CUDA;
}

// Encode a 4D tiled TMA descriptor (dims/strides innermost first, strides in bytes).
nomas_status encode4d(CUtensorMap* m, void* base, const uint64_t (&d)[4], const uint64_t (&s)[3],
                      const uint32_t (&b)[4]) {
  EncodeTiledFn fn = nullptr;
  nomas_status st = encoder(&fn);
  if (st != NOMAS_OK) return st;
  const cuuint64_t dims[4] = {d[0], d[1], d[2], d[3]};
  const cuuint64_t strides[3] = {s[0], s[1], s[2]};
  const cuuint32_t box[4] = {b[0], b[1], b[2], b[3]};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NOMAS_OK : NOMAS_ERR_CUDA;
}

// Work plan of one attention call (see AttnParams): units of one head x 256
// query rows (BF16 cache) or x 512 rows in a CTA pair (one-byte caches);
// units 0 .. n_full-1 run whole, every later unit in `splits` pieces of its
// key-tile range.
struct AttnPlan {
  int nq, nc, n_cache_tiles, n_cur_tiles;
  int ctas;            // CTAs per unit
  int units_per_head;
  int units;
  int n_full;
  int splits;          // pieces per split unit (1 = nothing split)
  int n_items;         // work items launched
  size_t ws_o_bytes, ws_lse_bytes;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

void plan_workspace(AttnPlan* pl) {
  const size_t rows = pl->splits > 1 ? static_cast<size_t>(pl->units - pl->n_full) * pl->splits * pl->ctas * 256 : 0;
  pl->ws_o_bytes = round256(rows * 128 * 4);
  pl->ws_lse_bytes = round256(rows * 4);
  pl->n_items = pl->n_full + (pl->units - pl->n_full) * pl->splits;
}

// Modelled time of a plan, in key-tile iterations of one CTA: waves of work
// items on `slots` concurrent items, a fixed cost per item (Q load, pipeline
// fill, epilogue), and for split units the combine pass (partials written by
// the kernel and read back, about 6.5 TB/s, plus one launch).  Whole units
// are dispatched first; the pieces fill the waves after them.
double plan_cost(int units, int n_full, int splits, int n_tiles, int slots, int ctas, double tile_us) {
  constexpr double kFixed = 2.5;
  const int per_piece = (n_tiles + splits - 1) / splits;
  double t = std::ceil(static_cast<double>(n_full) / slots) * (n_tiles + kFixed);
  const int rest = units - n_full;
  if (rest > 0) {
    t += std::ceil(static_cast<double>(rest) * splits / slots) * (per_piece + kFixed);
    if (splits > 1) {
      const double bytes = static_cast<double>(rest) * ctas * 256 * (2.0 * splits * 516 + 256);
      t += (bytes / 6.5e12 * 1e6 + 3.0) / tile_us;
    }
  }
  return t;
}

// The plan nomas_segment_attn chooses for num_splits = 0: no split; or the
// units of the last, partial wave each cut into s pieces (the whole units fill
// the full waves); or every unit cut into s pieces.  Cheapest modelled time,
// ties to fewer pieces.
void auto_plan(AttnPlan* pl, int n_tiles, int slots, bool one_byte) {
  const double tile_us = one_byte ? 2.0 : 1.6;
  const int U = pl->units;
  double best = plan_cost(U, U, 1, n_tiles, slots, pl->ctas, tile_us);
  int best_full = U, best_s = 1;
  const int s_max = std::min(8, std::max(1, n_tiles / 4));
  const int tail_full = (U / slots) * slots;
  for (int s = 2; s <= s_max; ++s) {
    for (int full : {tail_full, 0}) {
      if (full >= U) continue;
      const double c = plan_cost(U, full, s, n_tiles, slots, pl->ctas, tile_us);
      if (c < best * 0.98) {
        best = c;
        best_full = full;
        best_s = s;
      }
    }
  }
  pl->n_full = best_full;
  pl->splits = best_s;
}

// num_splits: 0 = automatic, 1 = no split, s > 1 = every unit in s pieces.
// n_tiles_eff (> 0) replaces the dense key-tile count in the automatic choice
// (block-sparse attention).
AttnPlan attn_plan(const nomas_kvcache* c, int32_t n_video, int32_t n_text, int32_t num_splits, int slots,
                   int n_tiles_eff = 0) {
  AttnPlan pl;
  pl.nq = n_video + n_text;
  pl.nc = static_cast<int>(static_cast<int64_t>(c->valid_frames) * c->grid_h * c->grid_w);
  pl.n_cache_tiles = (pl.nc + 127) / 128;
  pl.n_cur_tiles = (pl.nq + 127) / 128;
  const bool one_byte = quantised(c);
  pl.ctas = one_byte ? 2 : 1;
  const int n_qblocks = (pl.nq + 255) / 256;
  pl.units_per_head = one_byte ? (n_qblocks + 1) / 2 : n_qblocks;
  pl.units = pl.units_per_head * c->heads;
  const int n_tiles = pl.n_cache_tiles + pl.n_cur_tiles;
  if (num_splits == 0) {
    auto_plan(&pl, n_tiles_eff > 0 ? n_tiles_eff : n_tiles,
              slots > 0 ? slots : (one_byte ? 74 : 148), one_byte);
  } else {
    const int s = std::max(1, std::min(num_splits, std::min(n_tiles, 64)));
    pl.splits = s;
    pl.n_full = s > 1 ? 0 : pl.units;
  }
  plan_workspace(&pl);
  return pl;
}

// Concurrent work items of the attention kernel on the current device.
int attn_slots(const nomas_kvcache* c) {
  return attn_concurrent_items(cache_kind(c));
}
}  // namespace
}  // namespace nomas

using namespace nomas;

NOMAS_API int32_t nomas_version(void) { return 100; }

NOMAS_API const char* nomas_status_string(nomas_status s) {
  switch (s) {
    case NOMAS_OK: return "NOMAS_OK";
    case NOMAS_ERR_INVALID_ARG: return "NOMAS_ERR_INVALID_ARG";
    case NOMAS_ERR_UNSUPPORTED: return "NOMAS_ERR_UNSUPPORTED";
    case NOMAS_ERR_CAPACITY: return "NOMAS_ERR_CAPACITY";
    case NOMAS_ERR_CUDA: return "NOMAS_ERR_CUDA";
    case NOMAS_ERR_DEVICE_TIMEOUT: return "NOMAS_ERR_DEVICE_TIMEOUT";
  }
  return "NOMAS_UNKNOWN_STATUS";
}

NOMAS_API nomas_status nomas_kvcache_validate(const nomas_kvcache* cache) { return validate_cache(cache); }

NOMAS_API size_t nomas_kvcache_bytes(const nomas_kvcache* c) {
  if (c == nullptr || c->num_blocks <= 0 || c->heads <= 0 || c->head_dim <= 0 || c->grid_h <= 0 || c->grid_w <= 0 ||
      c->capacity_frames <= 0)
    return 0;
  const size_t rows = static_cast<size_t>(c->num_blocks) * c->heads * c->grid_h * c->grid_w * c->capacity_frames;
  if (quantised(c)) return 2 * rows * (static_cast<size_t>(c->head_dim) + 4);
  if (c->dtype == NOMAS_BF16) return 2 * rows * static_cast<size_t>(c->head_dim) * 2;
  return 0;
}

NOMAS_API nomas_status nomas_kvcache_plan_append(const nomas_kvcache* cache, int32_t n_frames, int32_t* first_frame,
                                                 int32_t* slot_frame, int64_t* new_total, int32_t* new_valid) {
  const nomas_status st = validate_cache(cache);
  if (st != NOMAS_OK) return st;
  return plan(cache, n_frames, first_frame, slot_frame, new_total, new_valid);
}

namespace {
// Pair tables of 3D RoPE: axis chunks of d_t, d_h, d_w dims in that order,
// pair i of a chunk of d_a dims at frequency theta^(-2i/d_a) (two floats).
void rope_tables(RopeParams* p, float theta, int32_t d_t, int32_t d_h, int32_t d_w) {
  memset(p, 0, sizeof(*p));
  const int dims[3] = {d_t, d_h, d_w};
  int pair = 0;
  for (int a = 0; a < 3; ++a) {
    for (int i = 0; i < dims[a] / 2; ++i, ++pair) {
      const double f = pow(static_cast<double>(theta), -2.0 * i / dims[a]);
      p->f_hi[pair] = static_cast<float>(f);
      p->f_lo[pair] = static_cast<float>(f - static_cast<double>(p->f_hi[pair]));
      p->axis[pair] = static_cast<int8_t>(a);
    }
  }
  for (; pair < kRopeMaxPairs; ++pair) p->axis[pair] = -1;
}

bool rope_split_ok(float theta, int32_t d_t, int32_t d_h, int32_t d_w) {
  if (d_t < 0 || d_h < 0 || d_w < 0 || ((d_t | d_h | d_w) & 1) != 0 || d_t + d_h + d_w > 128) return false;
  return theta > 0.0f && isfinite(theta);
}
}  // namespace

NOMAS_API nomas_status nomas_rope3d_apply(void* q, void* k, nomas_dtype io_dt, int32_t n_video, int32_t heads,
                                          int32_t head_dim, int64_t row_stride_elems, int32_t frames, int32_t grid_h,
                                          int32_t grid_w, int64_t t0, float theta, int32_t d_t, int32_t d_h,
                                          int32_t d_w, cudaStream_t stream) {
  if (io_dt != NOMAS_F32 && io_dt != NOMAS_BF16) return NOMAS_ERR_INVALID_ARG;
  if (q == nullptr || heads <= 0 || head_dim <= 0 || frames < 0 || grid_h <= 0 || grid_w <= 0 || n_video < 0)
    return NOMAS_ERR_INVALID_ARG;
  if (head_dim != 128) return NOMAS_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(frames) * grid_h * grid_w != n_video) return NOMAS_ERR_INVALID_ARG;
  if (!rope_split_ok(theta, d_t, d_h, d_w)) return NOMAS_ERR_INVALID_ARG;
  if (t0 < 0 || t0 + frames >= (int64_t(1) << 24) || grid_h >= (1 << 24) || grid_w >= (1 << 24))
    return NOMAS_ERR_UNSUPPORTED;
  if (heads > kRopeMaxHeads || n_video > kRopeMaxVideoRows) return NOMAS_ERR_UNSUPPORTED;
  const int64_t esz = io_dt == NOMAS_BF16 ? 2 : 4;
  if (row_stride_elems < static_cast<int64_t>(heads) * head_dim || (row_stride_elems * esz) % 16 != 0)
    return NOMAS_ERR_INVALID_ARG;
  if (!aligned16(q) || (k != nullptr && !aligned16(k))) return NOMAS_ERR_INVALID_ARG;
  if (n_video == 0) return NOMAS_OK;
  RopeParams p;
  rope_tables(&p, theta, d_t, d_h, d_w);
  p.n_video = n_video;
  p.heads = heads;
  p.row_stride = row_stride_elems;
  p.tpf = grid_h * grid_w;
  p.grid_w = grid_w;
  p.tpf_div = make_fast_div(static_cast<uint32_t>(p.tpf));
  p.gw_div = make_fast_div(static_cast<uint32_t>(grid_w));
  p.t0 = t0;
  p.extent = (static_cast<long long>(n_video) - 1) * row_stride_elems + static_cast<long long>(heads) * head_dim;
  p.err = nullptr;
  if (device_state(&p.err, nullptr) != NOMAS_OK) p.err = nullptr;
  return from_cuda(launch_rope3d(io_dt == NOMAS_BF16, q, k, p, stream));
}

namespace {
// Append, optionally with 3D RoPE of the K rows (rope != nullptr: the pair
// tables; positions are filled in here).
nomas_status append_impl(nomas_kvcache* cache, const void* k, const void* v, nomas_dtype in_dt, int32_t n_frames,
                         int64_t block_stride_elems, const RopeParams* rope, cudaStream_t stream) {
  nomas_status st = validate_cache(cache);
  if (st != NOMAS_OK) return st;
  if (in_dt != NOMAS_F32 && in_dt != NOMAS_BF16) return NOMAS_ERR_INVALID_ARG;
  if (n_frames < 0) return NOMAS_ERR_INVALID_ARG;
  const int64_t tpf = static_cast<int64_t>(cache->grid_h) * cache->grid_w;
  const int64_t seg_elems = n_frames * tpf * cache->heads * cache->head_dim;
  if (n_frames > 0) {
    if (k == nullptr || v == nullptr || !aligned16(k) || !aligned16(v)) return NOMAS_ERR_INVALID_ARG;
    if (cache->num_blocks > 1 && block_stride_elems < seg_elems) return NOMAS_ERR_INVALID_ARG;
    if (block_stride_elems < 0 || (block_stride_elems * (in_dt == NOMAS_F32 ? 4 : 2)) % 16 != 0)
      return NOMAS_ERR_INVALID_ARG;
  }
  int32_t first = 0, slot_frame = 0, new_valid = 0;
  int64_t new_total = 0;
  st = plan(cache, n_frames, &first, &slot_frame, &new_total, &new_valid);
  if (st != NOMAS_OK) return st;
  const int64_t n_tokens = (n_frames - first) * tpf;
  if (n_tokens > 0) {
    if (n_tokens > (int64_t(1) << 30)) return NOMAS_ERR_UNSUPPORTED;
    AppendParams p;
    p.k = k;
    p.v = v;
    p.block_stride = block_stride_elems;
    p.blocks = cache->num_blocks;
    p.heads = cache->heads;
    p.tpf = static_cast<int>(tpf);
    p.first_frame = first;
    p.n_tokens = static_cast<int>(n_tokens);
    p.base_slot_frame = slot_frame;
    p.capacity_frames = cache->capacity_frames;
    p.cap_slots = tpf * cache->capacity_frames;
    p.ck = cache->k;
    p.cv = cache->v;
    p.ks = cache->k_scale;
    p.vs = cache->v_scale;
    p.chunk_tokens = 0;
    p.err = nullptr;
    p.src_extent = static_cast<long long>(cache->num_blocks - 1) * block_stride_elems + seg_elems;
    p.cache_rows = static_cast<long long>(cache->num_blocks) * cache->heads * p.cap_slots;
    p.heads_div = make_fast_div(static_cast<uint32_t>(p.heads));
    p.tpf_div = make_fast_div(static_cast<uint32_t>(p.tpf));
    int sms = 0;
    if (device_state(&p.err, &sms) != NOMAS_OK) {
      p.err = nullptr;
      sms = 0;
    }
    if (rope != nullptr) {
      RopeParams rp = *rope;
      rp.t0 = cache->total_frames + first;  // absolute latent frame of the first written frame
      rp.tpf = p.tpf;
      rp.grid_w = cache->grid_w;
      rp.tpf_div = p.tpf_div;
      rp.gw_div = make_fast_div(static_cast<uint32_t>(cache->grid_w));
      rp.heads = cache->heads;
      rp.n_video = p.n_tokens;
      rp.row_stride = static_cast<long long>(cache->heads) * cache->head_dim;
      st = from_cuda(launch_append_rope(in_dt == NOMAS_F32, cache_kind(cache), p, rp, stream));
    } else {
      st = from_cuda(launch_append(in_dt == NOMAS_F32, cache_kind(cache), p, sms, stream));
    }
    if (st != NOMAS_OK) return st;
  }
  cache->total_frames = new_total;
  cache->valid_frames = new_valid;
  return NOMAS_OK;
}
}  // namespace

NOMAS_API nomas_status nomas_kvcache_append(nomas_kvcache* cache, const void* k, const void* v, nomas_dtype in_dt,
                                            int32_t n_frames, int64_t block_stride_elems, cudaStream_t stream) {
  return append_impl(cache, k, v, in_dt, n_frames, block_stride_elems, nullptr, stream);
}

NOMAS_API nomas_status nomas_kvcache_append_rope(nomas_kvcache* cache, const void* k, const void* v,
                                                 nomas_dtype in_dt, int32_t n_frames, int64_t block_stride_elems,
                                                 float theta, int32_t d_t, int32_t d_h, int32_t d_w,
                                                 cudaStream_t stream) {
  nomas_status st = validate_cache(cache);
  if (st != NOMAS_OK) return st;
  if (!rope_split_ok(theta, d_t, d_h, d_w) || n_frames < 0) return NOMAS_ERR_INVALID_ARG;
  if (cache->total_frames + n_frames >= (int64_t(1) << 24) || cache->grid_h >= (1 << 24) ||
      cache->grid_w >= (1 << 24))
    return NOMAS_ERR_UNSUPPORTED;
  RopeParams rp;
  rope_tables(&rp, theta, d_t, d_h, d_w);
  return append_impl(cache, k, v, in_dt, n_frames, block_stride_elems, &rp, stream);
}

NOMAS_API size_t nomas_kvcache_archive_frame_bytes(const nomas_kvcache* c) {
  if (validate_cache(c) != NOMAS_OK || !quantised(c)) return 0;
  const size_t rows = static_cast<size_t>(c->num_blocks) * c->heads * c->grid_h * c->grid_w;
  return 2 * rows * (static_cast<size_t>(c->head_dim) + 4);
}

NOMAS_API nomas_status nomas_kvcache_append_archive(nomas_kvcache* cache, const void* k, const void* v,
                                                    nomas_dtype in_dt, int32_t n_frames, int64_t block_stride_elems,
                                                    void* archive, size_t archive_bytes, size_t* archive_used,
                                                    cudaStream_t stream) {
  nomas_status st = validate_cache(cache);
  if (st != NOMAS_OK) return st;
  if (!quantised(cache)) return NOMAS_ERR_UNSUPPORTED;
  if (archive == nullptr || archive_used == nullptr || n_frames < 0) return NOMAS_ERR_INVALID_ARG;
  if (in_dt != NOMAS_F32 && in_dt != NOMAS_BF16) return NOMAS_ERR_INVALID_ARG;
  st = plan(cache, n_frames, nullptr, nullptr, nullptr, nullptr);
  if (st != NOMAS_OK) return st;
  const size_t frame_bytes = nomas_kvcache_archive_frame_bytes(cache);
  if (*archive_used > archive_bytes || static_cast<size_t>(n_frames) * frame_bytes > archive_bytes - *archive_used)
    return NOMAS_ERR_CAPACITY;
  const int64_t tpf = static_cast<int64_t>(cache->grid_h) * cache->grid_w;
  const int64_t planes = static_cast<int64_t>(cache->num_blocks) * cache->heads;
  const int64_t cap_slots = tpf * cache->capacity_frames;
  const int64_t esz = in_dt == NOMAS_F32 ? 4 : 2;
  const int64_t frame_elems = tpf * cache->heads * cache->head_dim;  // per block of the input
  const int64_t window = window_of(cache);
  const size_t code_bytes = static_cast<size_t>(planes * tpf * cache->head_dim);
  const size_t scale_bytes = static_cast<size_t>(planes * tpf * 4);
  uint8_t* dst = static_cast<uint8_t*>(archive) + *archive_used;
  // Chunks of at most one window: every frame of the segment passes through
  // the ring (so it is quantised there) and is copied out before a later
  // chunk of the same segment could overwrite its slot.
  for (int32_t done = 0; done < n_frames;) {
    const int32_t chunk = static_cast<int32_t>(std::min<int64_t>(window, n_frames - done));
    const char* kc = static_cast<const char*>(k) + static_cast<int64_t>(done) * frame_elems * esz;
    const char* vc = static_cast<const char*>(v) + static_cast<int64_t>(done) * frame_elems * esz;
    st = nomas_kvcache_append(cache, kc, vc, in_dt, chunk, block_stride_elems, stream);
    if (st != NOMAS_OK) return st;
    for (int32_t i = 0; i < chunk; ++i) {
      const int64_t slot = (cache->total_frames - chunk + i) % cache->capacity_frames;
      // Per frame: K codes, V codes [planes][tpf][head_dim], then K scales, V
      // scales [planes][tpf]; each a strided 2-D copy out of the ring.
      const void* src[4] = {static_cast<const int8_t*>(cache->k) + slot * tpf * cache->head_dim,
                            static_cast<const int8_t*>(cache->v) + slot * tpf * cache->head_dim,
                            cache->k_scale + slot * tpf, cache->v_scale + slot * tpf};
      const size_t width[4] = {static_cast<size_t>(tpf * cache->head_dim), static_cast<size_t>(tpf * cache->head_dim),
                               static_cast<size_t>(tpf * 4), static_cast<size_t>(tpf * 4)};
      const size_t pitch[4] = {static_cast<size_t>(cap_slots * cache->head_dim),
                               static_cast<size_t>(cap_slots * cache->head_dim), static_cast<size_t>(cap_slots * 4),
                               static_cast<size_t>(cap_slots * 4)};
      for (int j = 0; j < 4; ++j) {
        if (cudaMemcpy2DAsync(dst, width[j], src[j], pitch[j], width[j], static_cast<size_t>(planes),
                              cudaMemcpyDeviceToHost, stream) != cudaSuccess)
          return NOMAS_ERR_CUDA;
        dst += j < 2 ? code_bytes : scale_bytes;
      }
      *archive_used += frame_bytes;
    }
    done += chunk;
  }
  return NOMAS_OK;
}

NOMAS_API nomas_status nomas_camera_cross_attn(const void* q, const void* k_cam, const void* v_cam, int32_t frames,
                                               int32_t grid_h, int32_t grid_w, int32_t heads, int32_t n_cam,
                                               float softmax_scale, void* out, cudaStream_t stream) {
  if (frames < 0 || grid_h <= 0 || grid_w <= 0 || heads <= 0 || n_cam <= 0) return NOMAS_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || !isfinite(softmax_scale)) return NOMAS_ERR_INVALID_ARG;
  if (n_cam > 16 || heads > 65535 || frames > 65535) return NOMAS_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(grid_h) * grid_w > (int64_t(1) << 30)) return NOMAS_ERR_UNSUPPORTED;
  if (frames == 0) return NOMAS_OK;
  if (q == nullptr || k_cam == nullptr || v_cam == nullptr || out == nullptr) return NOMAS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cam) || !aligned16(v_cam) || !aligned16(out)) return NOMAS_ERR_INVALID_ARG;
  CameraAttnParams p;
  p.q = q;
  p.k_cam = k_cam;
  p.v_cam = v_cam;
  p.out = out;
  p.frames = frames;
  p.tpf = grid_h * grid_w;
  p.heads = heads;
  p.n_cam = n_cam;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.err = nullptr;
  if (device_state(&p.err, nullptr) != NOMAS_OK) p.err = nullptr;
  // Rows [frame][token][head][128]: the token extent of the query and output
  // maps is one frame's tpf, of the camera maps n_cam, so a box never reaches
  // into the next frame.
  const uint64_t H = static_cast<uint64_t>(heads), T = static_cast<uint64_t>(p.tpf), C = static_cast<uint64_t>(n_cam);
  CameraTensorMaps tm;
  nomas_status st = encode4d(&tm.q, const_cast<void*>(q), {128, H, T, static_cast<uint64_t>(frames)},
                             {256, H * 256, T * H * 256}, {64, 1, 128, 1});
  if (st == NOMAS_OK)
    st = encode4d(&tm.o, out, {128, H, T, static_cast<uint64_t>(frames)}, {256, H * 256, T * H * 256}, {64, 1, 128, 1});
  if (st == NOMAS_OK)
    st = encode4d(&tm.k, const_cast<void*>(k_cam), {128, H, C, static_cast<uint64_t>(frames)},
                  {256, H * 256, C * H * 256}, {64, 1, 16, 1});
  if (st == NOMAS_OK)
    st = encode4d(&tm.v, const_cast<void*>(v_cam), {128, H, C, static_cast<uint64_t>(frames)},
                  {256, H * 256, C * H * 256}, {64, 1, 16, 1});
  if (st != NOMAS_OK) return st;
  return from_cuda(launch_camera_attn(tm, p, stream));
}

NOMAS_API nomas_status nomas_kvcache_expand(const nomas_kvcache* src, nomas_kvcache* dst, cudaStream_t stream) {
  nomas_status st = validate_cache(src);
  if (st != NOMAS_OK) return st;
  if (dst == nullptr) return NOMAS_ERR_INVALID_ARG;
  st = validate_cache(dst);
  if (st != NOMAS_OK) return st;
  if (!quantised(src) || dst->dtype != NOMAS_BF16) return NOMAS_ERR_INVALID_ARG;
  if (src->num_blocks != dst->num_blocks || src->heads != dst->heads || src->head_dim != dst->head_dim ||
      src->grid_h != dst->grid_h || src->grid_w != dst->grid_w || src->capacity_frames != dst->capacity_frames ||
      src->past_frames != dst->past_frames)
    return NOMAS_ERR_INVALID_ARG;
  if (dst->k == src->k || dst->v == src->v || dst->k == dst->v) return NOMAS_ERR_INVALID_ARG;
  const int64_t tpf = static_cast<int64_t>(src->grid_h) * src->grid_w;
  ExpandParams p;
  p.kc = src->k;
  p.vc = src->v;
  p.ks = src->k_scale;
  p.vs = src->v_scale;
  p.ko = dst->k;
  p.vo = dst->v;
  p.planes = src->num_blocks * src->heads;
  p.cap_slots = tpf * src->capacity_frames;
  p.n_slots = tpf * src->valid_frames;
  p.err = nullptr;
  if (device_state(&p.err, nullptr) != NOMAS_OK) p.err = nullptr;
  st = from_cuda(launch_expand(cache_kind(src), p, stream));
  if (st != NOMAS_OK) return st;
  dst->total_frames = src->total_frames;
  dst->valid_frames = src->valid_frames;
  return NOMAS_OK;
}

NOMAS_API nomas_status nomas_kvcache_reset(nomas_kvcache* cache, int zero_memory, cudaStream_t stream) {
  nomas_status st = validate_cache(cache);
  if (st != NOMAS_OK) return st;
  if (zero_memory) {
    const size_t rows = static_cast<size_t>(cache->num_blocks) * cache->heads * cache->grid_h * cache->grid_w *
                        cache->capacity_frames;
    const size_t kv_bytes = rows * cache->head_dim * (quantised(cache) ? 1 : 2);
    st = from_cuda(launch_zero_fill(cache->k, kv_bytes, stream));
    if (st == NOMAS_OK) st = from_cuda(launch_zero_fill(cache->v, kv_bytes, stream));
    if (st == NOMAS_OK && quantised(cache)) {
      st = from_cuda(launch_zero_fill(cache->k_scale, rows * 4, stream));
      if (st == NOMAS_OK) st = from_cuda(launch_zero_fill(cache->v_scale, rows * 4, stream));
    }
    if (st != NOMAS_OK) return st;
  }
  cache->total_frames = 0;
  cache->valid_frames = 0;
  return NOMAS_OK;
}

namespace {
// The plan a call with these arguments runs (host only; the automatic choice
// depends on the current device's SM count).
nomas_status query_plan(const nomas_kvcache* cache, int32_t n_video, int32_t n_text, int32_t num_splits,
                        AttnPlan* pl) {
  nomas_status st = validate_cache(cache);
  if (st != NOMAS_OK) return st;
  if (n_video < 0 || n_text < 0 || num_splits < 0) return NOMAS_ERR_INVALID_ARG;
  *pl = attn_plan(cache, n_video, n_text, num_splits, num_splits == 0 ? attn_slots(cache) : 0);
  return NOMAS_OK;
}
}  // namespace

NOMAS_API nomas_status nomas_segment_attn_workspace_bytes(const nomas_kvcache* cache, int32_t n_video, int32_t n_text,
                                                          int32_t num_splits, size_t* bytes) {
  if (bytes == nullptr) return NOMAS_ERR_INVALID_ARG;
  AttnPlan pl;
  const nomas_status st = query_plan(cache, n_video, n_text, num_splits, &pl);
  if (st != NOMAS_OK) return st;
  *bytes = pl.ws_o_bytes + pl.ws_lse_bytes;
  return NOMAS_OK;
}

NOMAS_API nomas_status nomas_segment_attn_plan(const nomas_kvcache* cache, int32_t n_video, int32_t n_text,
                                               int32_t num_splits, nomas_attn_plan* out) {
  if (out == nullptr) return NOMAS_ERR_INVALID_ARG;
  AttnPlan pl;
  const nomas_status st = query_plan(cache, n_video, n_text, num_splits, &pl);
  if (st != NOMAS_OK) return st;
  out->units = pl.units;
  out->whole_units = pl.n_full;
  out->pieces_per_split_unit = pl.splits;
  out->ctas_per_unit = pl.ctas;
  out->work_items = pl.n_items;
  out->reserved = 0;
  out->workspace_bytes = pl.ws_o_bytes + pl.ws_lse_bytes;
  return NOMAS_OK;
}

namespace {
// Dense attention (tiles == nullptr) or block-sparse attention over kept
// cache-tile lists.  The workspace nomas_segment_attn_workspace_bytes reports
// for the same num_splits suffices for both.  `forced` (nullable) replaces
// the plan num_splits would give.
nomas_status segment_attn_impl(const nomas_kvcache* cache, int32_t block, const void* q, const void* k_cur,
                               const void* v_cur, int32_t n_video, int32_t n_text, float softmax_scale, void* out,
                               float* lse, void* workspace, size_t workspace_bytes, int32_t num_splits,
                               const int32_t* tiles, const int32_t* counts, int32_t max_keep,
                               const AttnPlan* forced, cudaStream_t stream) {
  nomas_status st = validate_cache(cache);
  if (st != NOMAS_OK) return st;
  if (block < 0 || block >= cache->num_blocks || n_video < 0 || n_text < 0 || num_splits < 0)
    return NOMAS_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || !isfinite(softmax_scale)) return NOMAS_ERR_INVALID_ARG;
  if (q == nullptr || k_cur == nullptr || v_cur == nullptr || out == nullptr) return NOMAS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cur) || !aligned16(v_cur) || !aligned16(out)) return NOMAS_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return NOMAS_ERR_INVALID_ARG;
  if (cache->heads > 65535) return NOMAS_ERR_UNSUPPORTED;
  const int64_t nq64 = static_cast<int64_t>(n_video) + n_text;
  if (nq64 == 0) return NOMAS_OK;
  if (nq64 > (int64_t(1) << 28)) return NOMAS_ERR_UNSUPPORTED;
  uint32_t* err = nullptr;
  st = device_state(&err, nullptr);
  if (st != NOMAS_OK) return st;
  const int slots = num_splits == 0 ? attn_slots(cache) : 0;
  AttnPlan pl = forced ? *forced : attn_plan(cache, n_video, n_text, num_splits, slots);
  if (!forced && tiles != nullptr && num_splits == 0) {
    // Block-sparse: plan for at most max_keep cache tiles per unit; keep the
    // dense plan (whose workspace the caller sized) if the sparse one needs more.
    const AttnPlan dense = pl;
    const int eff = std::min(max_keep, pl.n_cache_tiles) + pl.n_cur_tiles;
    pl = attn_plan(cache, n_video, n_text, 0, slots, std::max(1, eff));
    if (pl.ws_o_bytes + pl.ws_lse_bytes > dense.ws_o_bytes + dense.ws_lse_bytes) pl = dense;
  }
  if (pl.splits > 1 && (workspace == nullptr || workspace_bytes < pl.ws_o_bytes + pl.ws_lse_bytes ||
                        (reinterpret_cast<uintptr_t>(workspace) & 255u))) {
    if (num_splits > 1 || forced) return NOMAS_ERR_INVALID_ARG;  // an explicit split count needs its workspace
    pl = attn_plan(cache, n_video, n_text, 1, 0);
  }
  if (pl.n_items <= 0 || static_cast<int64_t>(pl.n_items) * pl.ctas > 0x7FFFFFFF) return NOMAS_ERR_UNSUPPORTED;
  const bool int8 = quantised(cache);  // one-byte codes (INT8 or FP8): staged and dequantised in the kernel
  AttnTensorMaps tm;
  memset(&tm, 0, sizeof(tm));
  const uint64_t H = cache->heads;
  const uint64_t tok_stride = H * 128 * 2;
  st = encode3d(&tm.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(q), 128, H, pl.nq, 256, tok_stride, 64, 1,
                128);
  if (st == NOMAS_OK)
    st = encode3d(&tm.kcur, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(k_cur), 128, H, pl.nq, 256,
                  tok_stride, 64, 1, 128);
  if (st == NOMAS_OK)
    st = encode3d(&tm.vcur, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(v_cur), 128, H, pl.nq, 256,
                  tok_stride, 64, 1, 128);
  const uint64_t cap_slots = static_cast<uint64_t>(cache->grid_h) * cache->grid_w * cache->capacity_frames;
  const uint64_t bh_rows = static_cast<uint64_t>(cache->num_blocks) * H;
  if (st == NOMAS_OK && pl.nc > 0) {
    if (int8) {
      // Each CTA of an INT8 pair stages half a tile: boxes of 64 rows.
      st = encode3d(&tm.kc, CU_TENSOR_MAP_DATA_TYPE_UINT8, cache->k, 128, pl.nc, bh_rows, 128, cap_slots * 128, 128,
                    64, 1);
      if (st == NOMAS_OK)
        st = encode3d(&tm.vc, CU_TENSOR_MAP_DATA_TYPE_UINT8, cache->v, 128, pl.nc, bh_rows, 128, cap_slots * 128, 128,
                      64, 1);
    } else {
      st = encode3d(&tm.kc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cache->k, 128, pl.nc, bh_rows, 256, cap_slots * 256, 64,
                    128, 1);
      if (st == NOMAS_OK)
        st = encode3d(&tm.vc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cache->v, 128, pl.nc, bh_rows, 256, cap_slots * 256,
                      64, 128, 1);
    }
  }
  if (st != NOMAS_OK) return st;
  AttnParams p;
  p.nq = pl.nq;
  p.nc = pl.nc;
  p.heads = cache->heads;
  p.n_cache_tiles = pl.n_cache_tiles;
  p.n_cur_tiles = pl.n_cur_tiles;
  p.units_per_head = pl.units_per_head;
  p.n_full = pl.n_full;
  p.tail_splits = pl.splits;
  p.block_head_base = block * cache->heads;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.ws_o = pl.splits > 1 ? static_cast<float*>(workspace) : nullptr;
  p.ws_lse = pl.splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.ws_o_bytes) : nullptr;
  p.k_scale = cache->k_scale;
  p.v_scale = cache->v_scale;
  p.scale_stride = static_cast<long long>(cap_slots);
  p.err = err;
  p.sparse_tiles = tiles;
  p.sparse_counts = counts;
  p.max_keep = max_keep;
  p.n_groups = (pl.nq + 511) / 512;
  p.block_heads = cache->num_blocks * cache->heads;
  p.ws_rows = pl.splits > 1 ? static_cast<long long>(pl.units - pl.n_full) * pl.splits * pl.ctas * 256 : 0;
  st = from_cuda(launch_segment_attn(cache_kind(cache), tm, p, pl.n_items, stream));
  if (st == NOMAS_OK && pl.splits > 1) st = from_cuda(launch_attn_combine(p, pl.units, pl.ctas, stream));
  return st;
}

int32_t sparse_keep_count(int32_t n_tiles, float keep_fraction) {
  const double k = std::ceil(static_cast<double>(keep_fraction) * n_tiles - 1e-9);
  return static_cast<int32_t>(std::min<double>(n_tiles, std::max(0.0, k)));
}
}  // namespace

NOMAS_API nomas_status nomas_segment_attn(const nomas_kvcache* cache, int32_t block, const void* q, const void* k_cur,
                                          const void* v_cur, int32_t n_video, int32_t n_text, float softmax_scale,
                                          void* out, float* lse, void* workspace, size_t workspace_bytes,
                                          int32_t num_splits, cudaStream_t stream) {
  return segment_attn_impl(cache, block, q, k_cur, v_cur, n_video, n_text, softmax_scale, out, lse, workspace,
                           workspace_bytes, num_splits, nullptr, nullptr, 0, nullptr, stream);
}

NOMAS_API nomas_status nomas_segment_attn_planned(const nomas_kvcache* cache, int32_t block, const void* q,
                                                  const void* k_cur, const void* v_cur, int32_t n_video,
                                                  int32_t n_text, float softmax_scale, void* out, float* lse,
                                                  void* workspace, size_t workspace_bytes,
                                                  const nomas_attn_plan* plan, cudaStream_t stream) {
  if (plan == nullptr) return NOMAS_ERR_INVALID_ARG;
  AttnPlan pl;
  nomas_status st = query_plan(cache, n_video, n_text, 1, &pl);
  if (st != NOMAS_OK) return st;
  const int n_tiles = pl.n_cache_tiles + pl.n_cur_tiles;
  if (plan->units != pl.units || plan->ctas_per_unit != pl.ctas || plan->whole_units < 0 ||
      plan->whole_units > pl.units || plan->pieces_per_split_unit < 1 ||
      plan->pieces_per_split_unit > std::max(1, std::min(n_tiles, 64)))
    return NOMAS_ERR_INVALID_ARG;
  pl.n_full = plan->whole_units;
  pl.splits = plan->whole_units == pl.units ? 1 : plan->pieces_per_split_unit;
  if (pl.splits == 1) pl.n_full = pl.units;
  plan_workspace(&pl);
  return segment_attn_impl(cache, block, q, k_cur, v_cur, n_video, n_text, softmax_scale, out, lse, workspace,
                           workspace_bytes, 0, nullptr, nullptr, 0, &pl, stream);
}

NOMAS_API nomas_status nomas_sparse_select_workspace_bytes(const nomas_kvcache* cache, int32_t n_video, int32_t n_text,
                                                           size_t* bytes) {
  nomas_status st = validate_cache(cache);
  if (st != NOMAS_OK) return st;
  if (bytes == nullptr || n_video < 0 || n_text < 0) return NOMAS_ERR_INVALID_ARG;
  // The mean key of every resident tile: [heads][T][128] float32.
  const int64_t nc = static_cast<int64_t>(cache->valid_frames) * cache->grid_h * cache->grid_w;
  const int64_t n_tiles = (nc + 127) / 128;
  *bytes = round256(static_cast<size_t>(cache->heads) * n_tiles * 128 * 4);
  return NOMAS_OK;
}

NOMAS_API nomas_status nomas_sparse_select(const nomas_kvcache* cache, int32_t block, const void* q, int32_t n_video,
                                           int32_t n_text, float keep_fraction, int32_t* tiles, int32_t* counts,
                                           int32_t max_keep, int32_t reuse_key_means, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream) {
  nomas_status st = validate_cache(cache);
  if (st != NOMAS_OK) return st;
  if (block < 0 || block >= cache->num_blocks || n_video < 0 || n_text < 0) return NOMAS_ERR_INVALID_ARG;
  if (q == nullptr || tiles == nullptr || counts == nullptr || !aligned16(q)) return NOMAS_ERR_INVALID_ARG;
  if (!(keep_fraction > 0.0f) || !(keep_fraction <= 1.0f)) return NOMAS_ERR_INVALID_ARG;
  const int64_t nq = static_cast<int64_t>(n_video) + n_text;
  const int64_t nc = static_cast<int64_t>(cache->valid_frames) * cache->grid_h * cache->grid_w;
  const int64_t n_tiles = (nc + 127) / 128, n_groups = (nq + 511) / 512;
  if (n_tiles > 8192 || nq > (int64_t(1) << 28) || cache->heads > 65535) return NOMAS_ERR_UNSUPPORTED;
  const int32_t keep = sparse_keep_count(static_cast<int32_t>(n_tiles), keep_fraction);
  if (max_keep < keep) return NOMAS_ERR_INVALID_ARG;
  size_t need = 0;
  nomas_sparse_select_workspace_bytes(cache, n_video, n_text, &need);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return NOMAS_ERR_INVALID_ARG;
  if (nq == 0) return NOMAS_OK;
  SparseSelectParams p;
  p.kcache = cache->k;
  p.kscale = cache->k_scale;
  p.cap_slots = static_cast<long long>(cache->grid_h) * cache->grid_w * cache->capacity_frames;
  p.block_head_base = block * cache->heads;
  p.nc = static_cast<int>(nc);
  p.n_tiles = static_cast<int>(n_tiles);
  p.q = q;
  p.nq = static_cast<int>(nq);
  p.heads = cache->heads;
  p.n_groups = static_cast<int>(n_groups);
  p.keep = keep;
  p.max_keep = max_keep;
  p.kbar = static_cast<float*>(workspace);
  p.tiles = tiles;
  p.counts = counts;
  p.cache_rows = static_cast<long long>(cache->num_blocks) * cache->heads * p.cap_slots;
  p.err = nullptr;
  if (device_state(&p.err, nullptr) != NOMAS_OK) p.err = nullptr;
  if (n_tiles == 0) {
    // Nothing resident: every list is empty.
    return from_cuda(cudaMemsetAsync(counts, 0, static_cast<size_t>(cache->heads) * n_groups * 4, stream));
  }
  return from_cuda(launch_sparse_select(cache_kind(cache), reuse_key_means != 0, p, stream));
}

NOMAS_API nomas_status nomas_segment_attn_sparse(const nomas_kvcache* cache, int32_t block, const void* q,
                                                 const void* k_cur, const void* v_cur, int32_t n_video, int32_t n_text,
                                                 float softmax_scale, const int32_t* tiles, const int32_t* counts,
                                                 int32_t max_keep, void* out, float* lse, void* workspace,
                                                 size_t workspace_bytes, int32_t num_splits, cudaStream_t stream) {
  if (tiles == nullptr || counts == nullptr || max_keep <= 0) return NOMAS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(tiles) & 3u) || (reinterpret_cast<uintptr_t>(counts) & 3u))
    return NOMAS_ERR_INVALID_ARG;
  return segment_attn_impl(cache, block, q, k_cur, v_cur, n_video, n_text, softmax_scale, out, lse, workspace,
                           workspace_bytes, num_splits, tiles, counts, max_keep, nullptr, stream);
}

NOMAS_API nomas_status nomas_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream) {
  if (limit_us == 0 || limit_us > 2000000u) return NOMAS_ERR_INVALID_ARG;
  uint32_t* err = nullptr;
  nomas_status st = device_state(&err, nullptr);
  if (st != NOMAS_OK) return st;
  return from_cuda(launch_wait_timeout_selftest(err, static_cast<uint64_t>(limit_us) * 1000ull, stream));
}

NOMAS_API int32_t nomas_bounds_checked(void) { return bounds_checked_build() ? 1 : 0; }

NOMAS_API nomas_status nomas_selftest_bounds_check(cudaStream_t stream) {
  if (!bounds_checked_build()) return NOMAS_ERR_UNSUPPORTED;
  uint32_t* err = nullptr;
  nomas_status st = device_state(&err, nullptr);
  if (st != NOMAS_OK) return st;
  return from_cuda(launch_bounds_check_selftest(err, stream));
}

NOMAS_API nomas_status nomas_device_error(nomas_status* status, int clear) {
  if (status == nullptr) return NOMAS_ERR_INVALID_ARG;
  uint32_t* err = nullptr;
  nomas_status st = device_state(&err, nullptr);
  if (st != NOMAS_OK) return st;
  uint32_t v = 0;
  if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return NOMAS_ERR_CUDA;
  if (clear && v != 0) {
    const uint32_t z = 0;
    if (cudaMemcpy(err, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return NOMAS_ERR_CUDA;
  }
  *status = static_cast<nomas_status>(v);
  return NOMAS_OK;
}

// ---------------------------------------------------------------------------
// nomas_segment_attn_noalloc: the same attention, with its split-KV scratch
// in a fixed device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory on this path: a serving engine
// that reserves nearly all of HBM for its own pools at start-up (a cudaMalloc
// here would fail or fragment that reservation), or a latency-bound loop where
// an allocation's implicit device synchronisation is not acceptable.  They call
// this entry point and pass only inputs and outputs.
//
// The scratch is one array per device, kNoAllocScratchBytes long, held by every
// device that loads this library for as long as the process lives.  All calls
// share it and it keeps whatever the last call left there; nothing in it needs
// to start at zero (every split writes each partial row before the combine
// reads it).  Two calls whose kernels overlap on the GPU (different streams,
// or different host threads without ordering) race on it.  The first call on
// a device looks up the array's device address (cudaGetSymbolAddress) with
// that device current; make that first call before any stream capture.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOMAS_NOALLOC_SCRATCH_BYTES];

namespace nomas {
namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once per device.
nomas_status noalloc_scratch(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NOMAS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NOMAS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return NOMAS_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return NOMAS_OK;
}
}  // namespace
}  // namespace nomas

NOMAS_API nomas_status nomas_segment_attn_noalloc(const nomas_kvcache* cache, int32_t block, const void* q,
                                                  const void* k_cur, const void* v_cur, int32_t n_video,
                                                  int32_t n_text, float softmax_scale, void* out, float* lse,
                                                  int32_t num_splits, cudaStream_t stream) {
  AttnPlan pl;
  nomas_status st = query_plan(cache, n_video, n_text, num_splits, &pl);
  if (st != NOMAS_OK) return st;
  constexpr size_t kCap = static_cast<size_t>(NOMAS_NOALLOC_SCRATCH_BYTES);
  if (pl.ws_o_bytes + pl.ws_lse_bytes > kCap) {
    // An explicit piece count that does not fit is refused.  The automatic
    // plan instead keeps its whole units and cuts the rest into fewer pieces,
    // down to none, until the scratch fits.
    if (num_splits != 0) return NOMAS_ERR_CAPACITY;
    while (pl.splits > 1 && pl.ws_o_bytes + pl.ws_lse_bytes > kCap) {
      --pl.splits;
      if (pl.splits == 1) pl.n_full = pl.units;
      plan_workspace(&pl);
    }
  }
  const size_t need = pl.ws_o_bytes + pl.ws_lse_bytes;
  void* scratch = nullptr;
  if (need > 0) {
    st = noalloc_scratch(&scratch);
    if (st != NOMAS_OK) return st;
  }
  return segment_attn_impl(cache, block, q, k_cur, v_cur, n_video, n_text, softmax_scale, out, lse, scratch, need,
                           num_splits, nullptr, nullptr, 0, &pl, stream);
}
