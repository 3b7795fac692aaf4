/*
 * nomas.h - C ABI of the segment-causal KV-cache attention library (B300, sm_103a).
 *
 * The library implements the per-block hot path of a segment-autoregressive
 * video diffusion transformer of the Hy-Nomas kind: each segment's video and
 * text queries attend over a persistent KV cache of earlier latent frames plus
 * the segment's own keys and values ("segment-wise causal joint attention", the
 * madebyagents.com model page; the lifelong KV cache of the orcarouter.ai
 * explainer, section "Die Schleife"), with 3D rotary positions and an optional
 * INT8, sliding-window cache (the low-memory preset of "Hy-Nomas auf einer RTX
 * 4090", section "Das Single-GPU-Preset": kv_cache_quantization int8,
 * past_frames 18).
 *
 * Conventions (all entry points):
 *  - Every device pointer is caller-owned device memory; the library never
 *    allocates, frees or synchronises.  Work is enqueued on the given stream
 *    and runs asynchronously; host-side metadata is updated at enqueue time.
 *  - Arguments are validated on the host before anything is launched; a
 *    failed validation returns a status and launches nothing.  A CUDA launch
 *    error returns NOMAS_ERR_CUDA.
 *  - Shapes: head_dim must be 128.  Activations are token-major
 *    [tokens][heads][head_dim] with the heads of a token contiguous.  Video
 *    tokens come first, in (latent frame, h, w) row-major order, then text
 *    tokens.
 *  - Device pointers must be 16-byte aligned.
 *  - Calls on distinct cache descriptors are thread-safe.
 *  - Kernels that wait on on-chip barriers give up after about one second,
 *    record NOMAS_ERR_DEVICE_TIMEOUT in a device-side error word and return;
 *    nomas_device_error() reads and optionally clears that word.
 */
#ifndef NOMAS_H_
#define NOMAS_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NOMAS_OK = 0,
  NOMAS_ERR_INVALID_ARG = 1,    /* bad pointer, shape, dtype, alignment or scale   */
  NOMAS_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. head_dim != 128) */
  NOMAS_ERR_CAPACITY = 3,       /* append beyond the capacity of a cache w/o window */
  NOMAS_ERR_CUDA = 4,           /* a CUDA runtime / launch error                    */
  NOMAS_ERR_DEVICE_TIMEOUT = 5  /* a kernel gave up waiting on an on-chip barrier   */
} nomas_status;

typedef enum { NOMAS_F32 = 0, NOMAS_BF16 = 1, NOMAS_INT8 = 2, NOMAS_FP8 = 3 } nomas_dtype;

/*
 * Persistent KV cache of num_blocks transformer blocks (the lifelong cache of
 * the orcarouter.ai explainer, section "Die Schleife"; windowed per "Das
 * Single-GPU-Preset" of the inferencekey.com RTX 4090 test).
 *
 * Layout (caller-allocated device memory):
 *   k, v       [num_blocks][heads][capacity_frames * grid_h * grid_w][head_dim]
 *              int8 codes (dtype NOMAS_INT8), E4M3 codes (NOMAS_FP8) or bf16
 *              values (NOMAS_BF16)
 *   k_scale,   [num_blocks][heads][capacity_frames * grid_h * grid_w] float32,
 *   v_scale    one scale per (block, head, token); NULL for NOMAS_BF16
 * Absolute latent frame f lives in frame-slot (f mod capacity_frames); token
 * (h, w) of that frame sits at slot (f mod capacity_frames)*grid_h*grid_w +
 * h*grid_w + w.  Resident slots are always [0, valid_frames*grid_h*grid_w).
 * INT8 codes: scale = fl32(absmax/127), code = clamp(rint(fl32(x *
 * fl32(127/absmax))), -127, 127), ties to even; an all-zero row has scale 0.
 * FP8 codes (a comparison format beside the pages' INT8): OCP E4M3 bytes,
 * scale = fl32(absmax/448), code = E4M3(fl32(x * fl32(448/absmax))), nearest
 * with ties to the even code, saturating at +-448; a NaN product (0 * inf,
 * only for a zero or tiny row) is coded 0.  Every call accepts a NOMAS_FP8
 * cache wherever it accepts NOMAS_INT8 (the archive included); the attention
 * dequantises value(code) * scale to bf16 in shared memory.
 *
 * past_frames > 0 is a sliding window of that many latent frames and requires
 * capacity_frames == past_frames; past_frames == 0 means no window (appending
 * beyond capacity_frames is NOMAS_ERR_CAPACITY).  total_frames and
 * valid_frames are host metadata maintained by append and reset; a caller
 * creating a descriptor sets them to 0.  Saving the struct and the device
 * buffers and restoring both resumes a session.
 */
typedef struct {
  int32_t num_blocks;      /* transformer blocks sharing this descriptor (>= 1)  */
  int32_t heads;           /* attention heads (>= 1)                              */
  int32_t head_dim;        /* must be 128                                         */
  int32_t grid_h;          /* latent rows per frame                               */
  int32_t grid_w;          /* latent columns per frame                            */
  int32_t capacity_frames; /* ring size in latent frames                          */
  int32_t past_frames;     /* window in latent frames; 0 = none                   */
  int32_t dtype;           /* nomas_dtype: NOMAS_INT8, NOMAS_FP8 or NOMAS_BF16    */
  void* k;                 /* device                                              */
  void* v;                 /* device                                              */
  float* k_scale;          /* device, INT8 / FP8 only                             */
  float* v_scale;          /* device, INT8 / FP8 only                             */
  int64_t total_frames;    /* absolute latent frames ever appended (host)         */
  int32_t valid_frames;    /* resident frames = min(total_frames, window) (host)  */
  int32_t reserved;        /* must be 0                                           */
} nomas_kvcache;

/* Library version (major*10000 + minor*100 + patch). Host only. */
int32_t nomas_version(void);

/* Human-readable name of a status. Host only; never NULL. */
const char* nomas_status_string(nomas_status s);

/* Check a descriptor's shape fields and pointers (no device access). */
nomas_status nomas_kvcache_validate(const nomas_kvcache* cache);

/* Device bytes the descriptor's k, v (and scales) need; 0 if invalid. Host only.
 * INT8 / FP8: 2 * blocks*heads*slots*(head_dim + 4); BF16: 2 * blocks*heads*slots*head_dim*2,
 * slots = capacity_frames*grid_h*grid_w. */
size_t nomas_kvcache_bytes(const nomas_kvcache* cache);

/*
 * What nomas_kvcache_append of n_frames would do, without doing it (host only).
 * first_frame: the first frame of the new segment that is written (frames
 * before it fall outside the window and are never written); slot_frame: the
 * ring frame-slot it goes to; new_total / new_valid: metadata afterwards.
 * Any output pointer may be NULL.  Returns NOMAS_ERR_CAPACITY when a cache
 * without a window would overflow.
 */
nomas_status nomas_kvcache_plan_append(const nomas_kvcache* cache, int32_t n_frames,
                                       int32_t* first_frame, int32_t* slot_frame,
                                       int64_t* new_total, int32_t* new_valid);

/*
 * 3D rotary position embedding, in place, on the video rows of Q (and K).
 * Model card: "3D RoPE" (inferencekey.com RTX 4090 test, "Modell und
 * Dateien").  Reading: head_dim splits into d_t, d_h, d_w contiguous chunks
 * (d_t + d_h + d_w <= head_dim, each even); inside the chunk of axis a, pair
 * (x[o+2i], x[o+2i+1]) rotates by pos_a * theta^(-2i/d_a):
 * (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos).  Video token n has positions
 * (t0 + n / (grid_h*grid_w), (n mod grid_h*grid_w) / grid_w, n mod grid_w).
 *
 *   q, k              device, [n_video..][heads][head_dim] of io_dt (F32 or
 *                     BF16), row stride row_stride_elems elements; rows
 *                     [0, n_video) are rotated, nothing else is touched.
 *                     k may be NULL.
 *   n_video           must equal frames*grid_h*grid_w
 *   t0                absolute latent frame of the segment's first frame
 *   theta             frequency base (> 0), e.g. 10000
 * Math in float32 (angles reduced with a compensated product), one rounding
 * to io_dt at the end.
 * NOMAS_ERR_UNSUPPORTED: head_dim != 128, t0 + frames >= 2^24, grid_h or
 * grid_w >= 2^24, heads > 2^19, n_video > 2^31 - 9.  NOMAS_ERR_INVALID_ARG:
 * other bad arguments (including q or k not 16-byte aligned, or a row stride
 * below heads*head_dim or not a multiple of 16 bytes).
 */
nomas_status nomas_rope3d_apply(void* q, void* k, nomas_dtype io_dt, int32_t n_video,
                                int32_t heads, int32_t head_dim, int64_t row_stride_elems,
                                int32_t frames, int32_t grid_h, int32_t grid_w, int64_t t0,
                                float theta, int32_t d_t, int32_t d_h, int32_t d_w,
                                cudaStream_t stream);

/*
 * Append a finished segment's K/V for all blocks (the KV-cache write stage,
 * "Zeiten" on the inferencekey.com RTX 4090 test page), quantising to INT8
 * (or FP8) with per-(block, head, token) scales or copying to BF16, into the
 * ring; frames
 * older than the window are never written (a segment longer than the window
 * writes only its last past_frames frames).  Updates cache->total_frames and
 * cache->valid_frames after a successful enqueue.
 *
 *   k, v                device, [num_blocks][n_frames*grid_h*grid_w][heads][head_dim]
 *                       of in_dt (F32 or BF16); block b starts at
 *                       b*block_stride_elems elements
 *   block_stride_elems  >= n_frames*grid_h*grid_w*heads*head_dim
 */
nomas_status nomas_kvcache_append(nomas_kvcache* cache, const void* k, const void* v,
                                  nomas_dtype in_dt, int32_t n_frames,
                                  int64_t block_stride_elems, cudaStream_t stream);

/*
 * The KV-write stage with position encoding (the "Schreiben des KV-Cache"
 * stage of the RTX 4090 guide, section "Zeiten"; positions continue from the
 * cached frames): nomas_kvcache_append of a segment whose keys have not been
 * rotated yet.  Frame f of the segment is rotated by 3D RoPE at positions
 * (total_frames + f, h, w) in float32, with the pair layout and frequencies of
 * nomas_rope3d_apply (theta, d_t, d_h, d_w as there), and the rotated row is
 * then quantised (INT8) or rounded to bf16 like any appended row; V is
 * appended unchanged.  One pass over the input instead of a RoPE pass over K
 * followed by an append.  With float32 input the stored bits equal those of
 * nomas_rope3d_apply (t0 = total_frames) followed by nomas_kvcache_append;
 * with bf16 input the rotated keys are not rounded to bf16 before they are
 * stored.  Arguments, errors and metadata updates as nomas_kvcache_append,
 * plus NOMAS_ERR_INVALID_ARG for a bad rotary split or theta and
 * NOMAS_ERR_UNSUPPORTED when total_frames + n_frames reaches 2^24.
 */
nomas_status nomas_kvcache_append_rope(nomas_kvcache* cache, const void* k, const void* v,
                                       nomas_dtype in_dt, int32_t n_frames,
                                       int64_t block_stride_elems, float theta, int32_t d_t,
                                       int32_t d_h, int32_t d_w, cudaStream_t stream);

/*
 * Host archive of every appended frame (the CPU KV archive of the low-memory
 * recipe: the GPU keeps the last past_frames latent frames, all earlier ones
 * live in host RAM; "System-RAM" on the inferencekey.com RTX 4090 test page
 * logs cpu_archive_gib growing by about 5.88 GiB per 30-frame segment).
 *
 * nomas_kvcache_archive_frame_bytes: host bytes one archived frame takes,
 * 2 * blocks * heads * grid_h * grid_w * (head_dim + 4); 0 for an invalid or
 * BF16 descriptor.  Host only.
 *
 * nomas_kvcache_append_archive: nomas_kvcache_append of an INT8 (or FP8) cache that
 * also copies every frame of the segment, once quantised, to host memory at
 * archive + *archive_used, in increasing frame order, and advances
 * *archive_used.  One archived frame is: K codes, V codes
 * ([blocks][heads][grid_h*grid_w][head_dim] bytes each), then K scales, V
 * scales ([blocks][heads][grid_h*grid_w] float32 each).  The segment is
 * appended in chunks of at most one window, so frames that fall out of the
 * window within the segment are still archived; the cache ends in the same
 * state as after nomas_kvcache_append.  The copies are asynchronous on
 * `stream` (pinned host memory makes them overlap other work); read the
 * archive after synchronising the stream.
 *
 *   archive, archive_bytes  caller-owned host buffer and its size
 *   archive_used            in/out: bytes already used
 * Returns NOMAS_ERR_UNSUPPORTED for a BF16 cache, NOMAS_ERR_CAPACITY (nothing
 * enqueued) when the archive or a cache without a window would overflow.
 */
size_t nomas_kvcache_archive_frame_bytes(const nomas_kvcache* cache);
nomas_status nomas_kvcache_append_archive(nomas_kvcache* cache, const void* k, const void* v, nomas_dtype in_dt,
                                          int32_t n_frames, int64_t block_stride_elems, void* archive,
                                          size_t archive_bytes, size_t* archive_used, cudaStream_t stream);

/*
 * How nomas_segment_attn divides its work.  A unit is one head x one block of
 * 256 query rows (BF16 cache, one CTA) or one head x two adjacent blocks (INT8
 * and FP8 caches, a pair of CTAs that share every dequantised key tile); units
 * are ordered head by head.  The first whole_units units run whole; every
 * later unit is cut into pieces_per_split_unit pieces of its key range, whose
 * partial outputs a second kernel merges in piece order.
 *
 *   num_splits = 0   automatic: the whole units fill the full waves of the
 *                    device's SMs and only the units of the last, partial wave
 *                    are cut (so they end together), or nothing is cut, or
 *                    every unit is, whichever a cost model of waves, per-unit
 *                    fixed cost and merge traffic finds cheapest
 *   num_splits = 1   nothing is cut
 *   num_splits = s   every unit is cut into s pieces (at most the number of
 *                    key tiles of 128 keys, and 64)
 *
 * nomas_segment_attn_workspace_bytes: device scratch the plan needs (0 when
 * nothing is cut): float32 partial outputs and log-sum-exps of every piece.
 * nomas_segment_attn_plan: the plan itself.  Both host only; for num_splits =
 * 0 they read the current device's SM count.
 */
typedef struct {
  int32_t units;                  /* heads x query units                         */
  int32_t whole_units;            /* units run whole                             */
  int32_t pieces_per_split_unit;  /* pieces of every later unit (1 = none cut)   */
  int32_t ctas_per_unit;          /* 1 (BF16 cache) or 2 (one-byte caches)        */
  int32_t work_items;             /* whole units + pieces                        */
  int32_t reserved;
  size_t workspace_bytes;         /* as nomas_segment_attn_workspace_bytes        */
} nomas_attn_plan;

nomas_status nomas_segment_attn_workspace_bytes(const nomas_kvcache* cache, int32_t n_video,
                                                int32_t n_text, int32_t num_splits,
                                                size_t* bytes);
nomas_status nomas_segment_attn_plan(const nomas_kvcache* cache, int32_t n_video, int32_t n_text,
                                     int32_t num_splits, nomas_attn_plan* plan);

/*
 * Segment attention of one block (the "segment-wise causal joint attention"
 * of the madebyagents.com model page over the lifelong cache of the
 * orcarouter.ai explainer): per head, O = softmax(s * Q K^T) V over the keys
 * [resident cache of `block` (dequantised if INT8 or FP8) ; current segment's K/V],
 * every current query seeing every key of that set.
 *
 *   q, k_cur, v_cur  device bf16 [n_video + n_text][heads][head_dim]
 *   softmax_scale    s > 0 (1/sqrt(128) in the model)
 *   out              device bf16 [n_video + n_text][heads][head_dim]
 *   lse              device float32 [heads][n_video + n_text] (natural log), or NULL
 *   workspace        device scratch of workspace_bytes (see
 *                    nomas_segment_attn_workspace_bytes), 256-byte aligned, or
 *                    NULL/0: with num_splits = 0 nothing is then cut
 *   num_splits       0 = automatic plan, 1 = none cut, s > 1 = every unit in s
 *                    pieces (see nomas_segment_attn_plan); s > 1 without enough
 *                    workspace is NOMAS_ERR_INVALID_ARG
 * BF16 tensor-core products with float32 accumulation and float32 softmax.
 * Results are bitwise reproducible for a given plan (num_splits on the same
 * device model).
 */
nomas_status nomas_segment_attn(const nomas_kvcache* cache, int32_t block, const void* q,
                                const void* k_cur, const void* v_cur, int32_t n_video,
                                int32_t n_text, float softmax_scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, int32_t num_splits,
                                cudaStream_t stream);

/*
 * nomas_segment_attn with a caller-chosen work plan (for example one tuned
 * for another SM count, or a fixed plan kept across devices for bitwise
 * reproducibility).  plan->units and plan->ctas_per_unit must equal what
 * nomas_segment_attn_plan reports for these arguments; 0 <= whole_units <=
 * units; 1 <= pieces_per_split_unit <= min(key tiles, 64) (ignored when
 * whole_units = units).  The workspace must hold what such a plan needs:
 * (units - whole_units) x pieces x ctas_per_unit x 256 rows of 516 bytes, each
 * of the two arrays rounded up to 256 bytes.  Anything else returns
 * NOMAS_ERR_INVALID_ARG without a launch.  Other arguments as
 * nomas_segment_attn.
 */
nomas_status nomas_segment_attn_planned(const nomas_kvcache* cache, int32_t block, const void* q,
                                        const void* k_cur, const void* v_cur, int32_t n_video,
                                        int32_t n_text, float softmax_scale, void* out, float* lse,
                                        void* workspace, size_t workspace_bytes,
                                        const nomas_attn_plan* plan, cudaStream_t stream);

/*
 * Block-sparse segment attention.  The single-GPU preset of the RTX 4090
 * guide lists a sparse attention backend that, after two dense denoising
 * steps, attends to a quarter of the candidate video key blocks (Hy-Nomas auf
 * einer RTX 4090, section "Das Single-GPU-Preset").  The pages give no block
 * size and no selection rule; this library reads them as follows.  A
 * candidate is a key tile of 128 resident cache slots (tile t = slots
 * [128 t, 128 t + 128) of the resident cache, the last one partial); the
 * current segment's own keys are always attended.  Queries form groups of 512
 * rows (g = row / 512).  For head h and group g, tile t scores
 * mean_query(h, g) . mean_key(h, t) (INT8 / FP8 keys dequantised), and the
 * k = min(T, ceil(keep_fraction * T)) best tiles are kept (equal scores: the
 * lower tile first), listed in increasing tile order.
 *
 * nomas_sparse_select_workspace_bytes: device scratch nomas_sparse_select
 * needs: the mean keys, float32 [heads][T][head_dim], 256-byte rounded.
 * Host only.
 *
 * nomas_sparse_select: compute the kept lists for one block.
 *   q               device bf16 [n_video + n_text][heads][head_dim] (the
 *                   queries that will attend, after RoPE)
 *   keep_fraction   in (0, 1]; 0.25 in the preset
 *   tiles           device int32 [heads][groups][max_keep]: row (h, g) gets
 *                   its kept tiles in its first counts[h, g] entries; the rest
 *                   of the row is left untouched
 *   counts          device int32 [heads][groups], groups = ceil((n_video + n_text) / 512)
 *   max_keep        row length of `tiles`; must be >= k
 *   reuse_key_means 0: compute the mean keys of the resident cache into the
 *                   workspace (one pass over the cache K).  Non-zero: the
 *                   workspace still holds the mean keys an earlier call
 *                   computed for this block with the cache unchanged since
 *                   (no append or reset), as across the denoising steps of
 *                   one turn; only the queries are read.  Stale means give a
 *                   valid but different list.
 *   workspace       device scratch, 256-byte aligned, of at least the bytes
 *                   nomas_sparse_select_workspace_bytes reports
 * Returns NOMAS_ERR_INVALID_ARG (nothing enqueued) for a bad argument and
 * NOMAS_ERR_UNSUPPORTED for more than 8192 resident tiles.  An empty cache
 * gives counts of 0.
 *
 * nomas_segment_attn_sparse: nomas_segment_attn where the queries of group g,
 * head h see only the cache tiles tiles[h, g, 0 .. counts[h, g]) plus every
 * current key.  Arguments as nomas_segment_attn, plus tiles, counts and
 * max_keep laid out as above (any increasing list of valid tiles, not only
 * one from nomas_sparse_select; counts are clamped to [0, min(max_keep, T)]).
 * A list entry outside [0, T) is clamped into the cache and records
 * NOMAS_ERR_INVALID_ARG in the device error word.  The workspace
 * nomas_segment_attn_workspace_bytes reports for the same split count
 * suffices.  With every tile kept the result equals nomas_segment_attn's.
 */
nomas_status nomas_sparse_select_workspace_bytes(const nomas_kvcache* cache, int32_t n_video,
                                                 int32_t n_text, size_t* bytes);
nomas_status nomas_sparse_select(const nomas_kvcache* cache, int32_t block, const void* q,
                                 int32_t n_video, int32_t n_text, float keep_fraction,
                                 int32_t* tiles, int32_t* counts, int32_t max_keep,
                                 int32_t reuse_key_means, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);
nomas_status nomas_segment_attn_sparse(const nomas_kvcache* cache, int32_t block, const void* q,
                                       const void* k_cur, const void* v_cur, int32_t n_video,
                                       int32_t n_text, float softmax_scale, const int32_t* tiles,
                                       const int32_t* counts, int32_t max_keep, void* out,
                                       float* lse, void* workspace, size_t workspace_bytes,
                                       int32_t num_splits, cudaStream_t stream);

/*
 * Scratch capacity, in bytes, of nomas_segment_attn_noalloc (one array per
 * device, held for the life of the process).
 */
#define NOMAS_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * nomas_segment_attn without a workspace argument: the split-KV scratch lives
 * in a static device array of NOMAS_NOALLOC_SCRATCH_BYTES inside the library,
 * and the call allocates nothing.  The pages have no counterpart; it exists
 * for callers that cannot allocate device memory on this path (an engine that
 * has reserved nearly all of HBM for its own pools, or a latency-bound loop
 * that cannot accept an allocation's implicit synchronisation).
 *
 * Arguments as nomas_segment_attn.  With num_splits = 0 the automatic plan is
 * used when its scratch fits; otherwise its split units are cut into fewer
 * pieces, down to none, until it fits, so the call always runs.  An explicit
 * num_splits > 1 whose scratch exceeds NOMAS_NOALLOC_SCRATCH_BYTES returns
 * NOMAS_ERR_CAPACITY and launches nothing (nomas_segment_attn_workspace_bytes
 * gives the need).  Every call shares the
 * array and it keeps the last call's contents (nothing in it must start at
 * zero); calls whose kernels overlap on the GPU race on it.  The first call on
 * a device looks up the array's address with that device current, so make it
 * before any stream capture.
 */
nomas_status nomas_segment_attn_noalloc(const nomas_kvcache* cache, int32_t block, const void* q,
                                        const void* k_cur, const void* v_cur, int32_t n_video,
                                        int32_t n_text, float softmax_scale, void* out, float* lse,
                                        int32_t num_splits, cudaStream_t stream);

/*
 * Camera cross-attention of the current segment's video tokens.  Camera
 * control enters as 4x4 extrinsic matrices grouped over four frames and fed
 * through cross-attention in every block (blog.authon.dev guide, section
 * "What Hy-Nomas is", model-card specs); one latent frame covers four video
 * frames (4x temporal compression, same list).  Reading: the camera encoder
 * (trained weights, upstream of this call) gives each latent frame n_cam
 * key/value tokens per head, and every video token of latent frame f attends
 * to exactly those: per head, O = softmax(s q K_f^T) V_f.  Text tokens are
 * not involved.
 *
 *   q            device bf16 [frames * grid_h * grid_w][heads][128]: the
 *                video rows (the first rows of a segment's Q tensor)
 *   k_cam, v_cam device bf16 [frames][n_cam][heads][128]
 *   n_cam        camera tokens per latent frame, 1 .. 16
 *   softmax_scale s > 0
 *   out          device bf16 [frames * grid_h * grid_w][heads][128]
 * All four pointers 16-byte aligned.  Scores and the weighted sum of V
 * accumulate in float32 on the tensor cores; the softmax runs in float32 and
 * its weights are rounded to bf16 for the weighted sum, as in
 * nomas_segment_attn; bf16 output.  NOMAS_ERR_UNSUPPORTED for n_cam > 16 or
 * more than 65535 heads or frames.
 */
nomas_status nomas_camera_cross_attn(const void* q, const void* k_cam, const void* v_cam,
                                     int32_t frames, int32_t grid_h, int32_t grid_w,
                                     int32_t heads, int32_t n_cam, float softmax_scale,
                                     void* out, cudaStream_t stream);

/*
 * BF16 copy of the resident window of an INT8 or FP8 cache.  The low-memory
 * preset keeps the cache in INT8 to fit a 24 GB card (Hy-Nomas auf einer RTX
 * 4090, section "Das Single-GPU-Preset"); the cache changes only when a
 * finished segment is appended (section "Zeiten"), while every denoising step
 * of the next segment attends over it.  A caller with memory to spare can
 * expand the window once per append and run those steps' attention over the
 * copy (nomas_segment_attn with dst), which gives the same values the
 * attention kernel dequantises itself: x_hat = bf16(fl32(code * scale)).
 *
 *   src  an INT8 or FP8 cache (not modified)
 *   dst  a BF16 cache of the same geometry (blocks, heads, head_dim, grid,
 *        capacity_frames, past_frames), buffers distinct from src's; caller-
 *        owned.  Its resident slots [0, valid_frames * grid_h * grid_w) of
 *        every (block, head) plane are overwritten, and its total_frames /
 *        valid_frames are set to src's when the call succeeds.
 * Stream-ordered, no allocation.  NOMAS_ERR_INVALID_ARG for a BF16 src, a
 * one-byte dst, mismatched geometry or shared buffers.
 */
nomas_status nomas_kvcache_expand(const nomas_kvcache* src, nomas_kvcache* dst, cudaStream_t stream);

/*
 * Start a new session (the resident service's new session_id, "Setup" and the
 * JSON turns on the inferencekey.com RTX 4090 test page): total_frames and
 * valid_frames to 0; with zero_memory != 0 also enqueue a kernel that clears
 * k, v and the scales.
 */
nomas_status nomas_kvcache_reset(nomas_kvcache* cache, int zero_memory, cudaStream_t stream);

/*
 * Self-test of the bounded-wait error path (no counterpart in the pages):
 * enqueue a one-warp kernel that waits up to limit_us microseconds (1 ..
 * 2,000,000) on an on-chip barrier that nothing arrives on, then records
 * NOMAS_ERR_DEVICE_TIMEOUT in the device error word and exits normally.  No
 * fault or hang is involved; the context stays usable.  Read the result with
 * nomas_device_error.  Returns NOMAS_ERR_INVALID_ARG for a limit out of range.
 */
nomas_status nomas_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream);

/*
 * The range-checked build (no counterpart in the pages).  The library also
 * ships as libnomas_checked.so, the same kernels compiled so that every
 * computed global-memory index (TMA tile origins, ring slots, cache rows and
 * scales, tile-list entries, output, partial and workspace rows) is checked
 * against its buffer before the access: a bad index records
 * NOMAS_ERR_INVALID_ARG in the device error word and the access is skipped;
 * nothing traps.
 *
 * nomas_bounds_checked: 1 in the checked build, 0 otherwise.
 * nomas_selftest_bounds_check: checked build only, enqueue a one-warp kernel
 * whose single range check fails on purpose (index 4 of a 4-element buffer),
 * so NOMAS_ERR_INVALID_ARG lands in the device error word with no access made.
 * Returns NOMAS_ERR_UNSUPPORTED, launching nothing, in the regular build.
 */
int32_t nomas_bounds_checked(void);
nomas_status nomas_selftest_bounds_check(cudaStream_t stream);

/*
 * Read the device-side error word of the current device (a status code set
 * by a kernel that gave up waiting, 0 if none), synchronously.  With clear != 0
 * the word is reset to 0.  *status receives NOMAS_OK or the recorded status.
 */
nomas_status nomas_device_error(nomas_status* status, int clear);

#ifdef __cplusplus
}
#endif

#endif /* NOMAS_H_ */
