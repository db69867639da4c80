/*
 * gqa_decode.h -- C ABI of libgqa_decode.so: single-token grouped-query decode
 * attention over a KV cache on NVIDIA GB300 (sm_103a).
 *
 * What is computed (restated from the "FlashInfer sm110_gqa_decode" article,
 * sections "Input contract", "Convenience API" and "Prepared continuous
 * decoding", and for FP8 from the "FP8 KV cache port on Jetson AGX Thor" blog,
 * section 1, patch 2):
 *
 *   Fixed geometry: 32 query heads, 8 KV heads, head_dim 128, one query token
 *   per request.  Query head h reads KV head g = h / 4 (the grouped view
 *   that splits the 32 heads into 8 groups of 4 consecutive heads).  For every batch row b and query head h:
 *     s_t   = q_scale * k_scale / sqrt(128) * dot(q[b,h,:], K[b,g,t,:]),  0 <= t < len[b]
 *     out[b,h,:] = v_scale * sum_t softmax(s)_t * V[b,g,t,:]
 *   k_scale = v_scale = 1 except on the e4m3 entry point.  Slots t >= len[b]
 *   are never read.  Arithmetic is FP32 (exp2-domain online softmax); the
 *   output is rounded once to fp16/bf16, round-to-nearest-even.
 *
 * Layouts (all dense, row-major, contiguous; element offsets):
 *   q    [batch, 32, 128]              fp16 or bf16 (gqa_dtype_t)
 *   kv   [batch, 2, 8, capacity, 128]  plane 0 = K, plane 1 = V; same dtype
 *                                      as q, e4m3 bytes (fp8 entry) or int8
 *                                      codes with bf16 row scales (int8 entry);
 *                                      a paged pool on the paged entries
 *   lens int32 [batch], device memory, read only by the kernels; the contract
 *        is 1 <= lens[b] <= capacity (see "Lengths" below)
 *   out  [batch, 32, 128]              same dtype as q (bf16 on the fp8 entry)
 *   q, kv, out and the workspace must be 16-byte aligned; lens 4-byte aligned.
 *
 * Pointers are device pointers unless stated.  `stream` is a cudaStream_t
 * (NULL = the legacy default stream).  Every launching call is asynchronous,
 * enqueues on `stream`, reads nothing back to the host and performs no host
 * synchronisation, except gqa_decode_get_status and
 * gqa_decode_noalloc_get_status (documented there).
 *
 * Ownership: the caller owns every buffer (q, kv, lens, out, workspace).  The
 * library never frees caller memory and keeps no pointer past the call.  The
 * only library-owned state is a per-device cache of the device check and of
 * kernel attributes, and the static scratch of gqa_decode_noalloc.
 *
 * Errors: every function validates its arguments before any CUDA call and
 * returns a gqa_status_t; no exception or abort crosses this ABI.  A
 * thread-local message with details of the last failure on the calling thread
 * is available from gqa_last_error().
 *
 * Lengths: read on the device only.  A length outside [1, capacity] is
 * clamped to [0, capacity] (0 produces a zero output row), never read out of
 * bounds, and flagged with GQA_FLAG_LENGTH_CLAMPED in the workspace header
 * (gqa_decode_get_status).
 *
 * Workspace (split-KV, the flash-decoding scheme of the article's
 * "num_splits" section): a caller-owned device buffer of
 * gqa_decode_workspace_size(batch, capacity, num_splits) bytes.  It holds a
 * 256-byte header (status flags) and FP32 partial results (unnormalised
 * output, running max in the log2 domain, softmax denominator) per
 * (b, query head, split slot).  How a row is cut is decided per call from the
 * sizes: into num_splits chunks of capacity (one CTA each), or, for grids of
 * more than one wave, into pieces of equal runs of one stream of all rows'
 * tiles (each row start weighs one more tile when some row is shorter than
 * a run) taken by the resident CTAs (lengths read on the device); either way
 * a row has at most num_splits pieces, and the results are deterministic.
 * With one piece per CTA, 2..8 splits that hold slots and a grid of one wave
 * at most, the splits of each (b, KV head) run as one thread-block cluster
 * and merge on chip through distributed shared memory: no partial is
 * written and stage 2 launches nothing.  Zero the header once before first use (gqa_decode_workspace_init).
 * Launches that may run concurrently (different streams or graphs) need
 * distinct workspaces; launches ordered on one stream may share one.
 */
#ifndef GQA_DECODE_H_
#define GQA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQA_NUM_Q_HEADS 32
#define GQA_NUM_KV_HEADS 8
#define GQA_HEAD_DIM 128
#define GQA_MAX_SPLITS 256
#define GQA_WORKSPACE_HEADER_BYTES 256

typedef enum {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARGUMENT = 1,   /* null pointer, size, dtype, scale, misalignment */
  GQA_ERR_UNSUPPORTED_DEVICE = 2, /* not a compute capability 10.3 (sm_103) device */
  GQA_ERR_WORKSPACE_TOO_SMALL = 3,
  GQA_ERR_ALIASING = 4,           /* out overlaps q, kv or lens */
  GQA_ERR_CUDA = 5                /* a CUDA runtime call failed (see gqa_last_error) */
} gqa_status_t;

typedef enum { GQA_F16 = 0, GQA_BF16 = 1 } gqa_dtype_t;

typedef enum { GQA_KV_F16 = 0, GQA_KV_BF16 = 1, GQA_KV_E4M3 = 2, GQA_KV_I8 = 3 } gqa_kv_format_t;

/* Bits of the status word in the workspace header. */
#define GQA_FLAG_LENGTH_CLAMPED 0x1u  /* some lens[b] was outside [1, capacity] */
#define GQA_FLAG_WAIT_TIMEOUT 0x2u    /* a pipeline wait gave up; outputs are invalid */
#define GQA_FLAG_PAGE_CLAMPED 0x4u    /* a block-table entry was outside [0, num_pages) (decode: clamped; append: not written) */
#define GQA_FLAG_SLOT_CLAMPED 0x8u    /* gqa_append_kv: a slot outside [0, capacity), not written */
#define GQA_FLAG_BOUNDS 0x10u         /* checked builds only (GQA_CHECKED): an access fell outside its
                                         buffer and was redirected inside it; the library has a bug */

/* Name of a status code (static string). */
const char* gqa_status_string(gqa_status_t status);

/* Details of the last failure on the calling thread ("" if none). */
const char* gqa_last_error(void);

/* Bytes of workspace needed for (batch, capacity, num_splits); 0 if the
 * arguments are invalid (batch, capacity < 1; num_splits outside
 * [1, GQA_MAX_SPLITS]).  num_splits = 1 needs only the 256-byte header. */
size_t gqa_decode_workspace_size(int batch, int capacity, int num_splits);

/* Host-only split planner (no CUDA call besides a cached SM-count query; safe
 * during stream capture once the device has been seen).  Picks the number of
 * KV splits from batch x capacity, the KV format and the SM count of `device`:
 * about 8 waves of (batch, KV head, split) work items over the worst case, or,
 * for latency-bound sizes (at most 16 tiles per resident CTA in all), about
 * sqrt(6 x tiles per row) capped at one wave.  Writes the chosen count
 * (1..GQA_MAX_SPLITS) to *num_splits_out. */
gqa_status_t gqa_decode_plan(int batch, int capacity, gqa_kv_format_t kv_format, int device,
                             int* num_splits_out);

/* The same planner with the SM count given: pure host arithmetic, no CUDA
 * call.  sm_count < 1 is invalid. */
gqa_status_t gqa_decode_plan_for(int batch, int capacity, gqa_kv_format_t kv_format, int sm_count,
                                 int* num_splits_out);

/* Split geometry (pure host arithmetic): tokens per split, rounded up to
 * whole 64-token (fp16/bf16) or 128-token (8-bit) tiles, and the number of
 * splits that hold slots, ceil(capacity / chunk) <= num_splits.  With one
 * piece per CTA, split s covers slots [s * chunk, min((s + 1) * chunk, len));
 * the balanced schedule cuts rows elsewhere but never into more pieces.
 * Stage 2 runs only when the effective count is above 1 and the splits do
 * not merge on chip (2..8 of them with one piece per CTA in a grid of one
 * wave whose clusters can all be resident at once do, in a thread-block
 * cluster). */
gqa_status_t gqa_decode_split_geometry(int capacity, int num_splits, gqa_kv_format_t kv_format,
                                       int* chunk_tokens_out, int* splits_effective_out);

/* Kernels one decode call of these sizes enqueues on its stream (host
 * arithmetic; no work is enqueued): 1 when a single split holds every slot
 * or the splits merge on chip in a thread-block cluster, else 2 (the split
 * kernel and the combine).  The on-chip merge also needs all its clusters
 * resident at once; once the current device has been set up by a call that
 * launches, and sm_count is its SM count, its cluster occupancy (queried at
 * set-up) decides that as the launches do, else only the SM count does.
 * The same for the contiguous and paged entries; q_len 1..4 as
 * gqa_decode_verify; num_splits 1..GQA_MAX_SPLITS after resolving 0;
 * sm_count < 1 is invalid.  Writes the count to *launches_out. */
gqa_status_t gqa_decode_launch_count_for(int batch, int capacity, gqa_kv_format_t kv_format, int q_len,
                                         int num_splits, int sm_count, int* launches_out);

/* Convenience call (the article's sm110_gqa_decode): plans the split count,
 * takes a stream-ordered workspace with cudaMallocAsync/cudaFreeAsync on
 * `stream`, and launches.  q_scale must be finite and >= 0 (0 gives the mean
 * of V).  Length-clamp flags are not observable through this call. */
gqa_status_t gqa_decode(const void* q, const void* kv, const int32_t* lens, void* out,
                        int batch, int capacity, gqa_dtype_t dtype, float q_scale,
                        void* stream);

/* Prepared call (the article's launch_sm110_gqa_decode_prepared): no
 * allocation and no host synchronisation, so it can be captured in a CUDA
 * graph.  q_scale must be finite and > 0 (as the article's prepare step
 * requires).  num_splits = 0 picks gqa_decode_plan's choice; otherwise
 * 1..GQA_MAX_SPLITS.  `workspace` must hold gqa_decode_workspace_size(batch,
 * capacity, num_splits) bytes (after resolving 0).  `out` must not overlap q,
 * kv or lens. */
gqa_status_t gqa_decode_prepared(const void* q, const void* kv, const int32_t* lens, void* out,
                                 int batch, int capacity, gqa_dtype_t dtype, float q_scale,
                                 int num_splits, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* FP8 KV cache (the blog's e4m3 port): kv holds float8 e4m3fn bytes (OCP FP8:
 * bias 7, no infinities, 0x7F/0xFF NaN), q and out are bf16.  k_scale
 * multiplies the scores, v_scale the normalised output; both finite and > 0.
 * q_scale finite and >= 0.  Other rules as gqa_decode_prepared. */
gqa_status_t gqa_decode_fp8kv(const void* q_bf16, const uint8_t* kv_e4m3, const int32_t* lens,
                              void* out_bf16, int batch, int capacity, float q_scale,
                              float k_scale, float v_scale, int num_splits, void* workspace,
                              size_t workspace_bytes, void* stream);

/* INT8 KV cache (the "Qwen3-VL official BF16 on Jetson Orin (SM87)" docs,
 * section "INT8 KV cache (kv_mode)": the cache kept as int8 codes, each
 * (position, KV head) row with its own bf16 scale).  kv_i8 holds int8 codes [batch, 2, 8,
 * capacity, 128]; kv_scales_bf16 holds bf16 scales [batch, 2, 8, capacity]
 * (plane 0 K rows, plane 1 V rows), 16-byte aligned, and capacity must be a
 * multiple of 8 (the scales are staged by 16-byte bulk copies); element (b, p, g, t, d)
 * of the cache is code * scale[b, p, g, t].  q and out are fp16 or bf16
 * (`dtype`).  The K row scale multiplies that slot's scores, the V row scale
 * its weight; scales of slots >= len[b] are never read.  q_scale finite and
 * >= 0.  Other rules as gqa_decode_prepared (no allocation, no host sync). */
gqa_status_t gqa_decode_int8kv(const void* q, const int8_t* kv_i8, const uint16_t* kv_scales_bf16,
                               const int32_t* lens, void* out, int batch, int capacity,
                               gqa_dtype_t dtype, float q_scale, int num_splits, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Paged KV cache.  The pages only say that a paged cache is gathered into
 * one contiguous prefix matrix before attention; this entry reads the pages
 * in place instead, with the same result.  Layout (this library's reading):
 *   kv_pages        [num_pages, 2, 8, page_size, 128] in `kv_format` (fp16,
 *                   bf16, e4m3 or int8), each (page, plane, KV head) block
 *                   contiguous
 *   kv_scales_pages int8 only (NULL otherwise): bf16 [num_pages, 2, 8,
 *                   page_size], the row scales of the same page rows,
 *                   16-byte aligned
 *   block_table     int32 [batch, max_pages_per_seq], device memory, read only
 *                   by the kernels: slot t of batch row b is row t % page_size
 *                   of page block_table[b][t / page_size]
 * page_size is a power of two in [16, 65536]; the capacity is
 * max_pages_per_seq * page_size (<= 2^30), and lengths follow the usual
 * contract against it.  Only the entries of pages holding slots < len[b] are
 * used; an entry outside [0, num_pages) is clamped and flagged with
 * GQA_FLAG_PAGE_CLAMPED, never dereferenced out of bounds.  q_len 1..4: q
 * and out are [batch, q_len, 32, 128] and query j attends slots
 * [0, len - q_len + j] (gqa_decode_verify); 1 is plain decode.  q/out dtype
 * `q_dtype` (must equal fp16/bf16 KV; either for 8-bit KV).  k_scale,
 * v_scale as gqa_decode_fp8kv (1 for the other formats).  Both stages, no
 * allocation, no host sync; the workspace as gqa_decode_prepared for batch
 * * q_len rows and capacity max_pages_per_seq * page_size. */
gqa_status_t gqa_decode_paged(const void* q, gqa_dtype_t q_dtype, const void* kv_pages,
                              gqa_kv_format_t kv_format, const uint16_t* kv_scales_pages,
                              const int32_t* block_table, int max_pages_per_seq, int num_pages,
                              int page_size, const int32_t* lens, void* out, int batch, int q_len,
                              float q_scale, float k_scale, float v_scale, int num_splits,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Verify window: q_len query tokens per request (1..4), the draft tokens of
 * speculative / multi-token-prediction decoding (the "FP8 KV cache port on
 * Jetson AGX Thor" blog, section 2, MTP).  The window's tokens are the last
 * q_len slots already written to the cache: query token j of row b sits at
 * slot len[b] - q_len + j and attends slots [0, len[b] - q_len + j] (causal
 * within the window).  q and out are [batch, q_len, 32, 128]; the workspace
 * holds gqa_decode_workspace_size(batch * q_len, capacity, num_splits) bytes.
 * Lengths must lie in [q_len, capacity]; a query with no slot (len below
 * q_len) gets a zero row and GQA_FLAG_LENGTH_CLAMPED.  kv_format: fp16 / bf16
 * (= q_dtype), e4m3 or int8 (kv_scales_bf16 as gqa_decode_int8kv, else NULL).
 * k_scale, v_scale as gqa_decode_fp8kv (1 unless e4m3).  q_scale finite and
 * >= 0.  Both stages, no allocation, no host sync. */
gqa_status_t gqa_decode_verify(const void* q, gqa_dtype_t q_dtype, const void* kv,
                               gqa_kv_format_t kv_format, const uint16_t* kv_scales_bf16,
                               const int32_t* lens, void* out, int batch, int capacity, int q_len,
                               float q_scale, float k_scale, float v_scale, int num_splits,
                               void* workspace, size_t workspace_bytes, void* stream);

/* The two stages of a prepared launch, for callers that schedule (or time)
 * them separately.  Stage 1 streams K/V once per (b, KV head, split) and
 * writes FP32 partials to the workspace, or the final output when
 * num_splits == 1 or when its 2..8 effective splits merge on chip (one
 * thread-block cluster per (b, KV head), one piece per CTA, one wave, every
 * cluster resident at once).  Stage 2 merges the partials of each (b, query
 * head) with a log-sum-exp combine and writes `out`; when stage 1 wrote the
 * output it launches nothing.  Both must be given the same geometry, scales
 * and workspace, in this order, on one stream, with the same device
 * current.  Validation as gqa_decode_prepared, except that
 * q_scale may be 0.  Stage 1 does not take an int8 cache (it has no scale
 * argument: use gqa_decode_int8kv); stage 2 accepts every format. */
gqa_status_t gqa_decode_split_stage(const void* q, gqa_dtype_t q_dtype, const void* kv,
                                    gqa_kv_format_t kv_format, const int32_t* lens, void* out,
                                    int batch, int capacity, float q_scale, float k_scale,
                                    float v_scale, int num_splits, void* workspace,
                                    size_t workspace_bytes, void* stream);
gqa_status_t gqa_decode_combine_stage(const int32_t* lens, void* out, gqa_dtype_t out_dtype,
                                      gqa_kv_format_t kv_format, int batch, int capacity,
                                      float v_scale, int num_splits, const void* workspace,
                                      size_t workspace_bytes, void* stream);

/* No-allocation variant of gqa_decode, for callers that cannot allocate
 * device memory at call time: code running inside a memory-budgeted runtime
 * or a custom allocator that forbids cudaMalloc on the decode path, plugins
 * handed only pre-existing buffers, or hosts that must not touch the
 * allocator between steps.  The pages have no counterpart to this call (their
 * convenience call allocates its workspace and their prepared call takes one
 * from the caller).
 *
 * The split-KV scratch lives in a file-scope static __device__ array of
 * GQA_STATIC_WORKSPACE_BYTES (16 MiB) that every GPU which loads this library
 * holds until the process exits.  The caller still passes q, kv, lens and out.
 * This call performs no cudaMalloc, cudaFree or other allocation; it launches
 * the two stages on `stream`.
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress, zeroes its 256-byte
 * header (the status word) with cudaMemsetAsync on `stream`, and caches the
 * address; make that first call before any stream capture.  A failed lookup
 * is reported (GQA_ERR_CUDA) and retried by the next call.  The cached
 * address belongs to the device's primary context: do not use this call (or
 * gqa_decode_noalloc_get_status) on a device after cudaDeviceReset.  Every
 * call on a device shares the one array, which keeps the last call's
 * contents: calls that may overlap on the GPU (different streams or graphs
 * without ordering) race and corrupt each other's results; order them on one
 * stream.  The partials need no clearing (each call writes before it reads);
 * the status flags (GQA_FLAG_LENGTH_CLAMPED, GQA_FLAG_WAIT_TIMEOUT) accumulate
 * over calls until gqa_decode_noalloc_get_status reads and clears them.
 *
 * num_splits = 0 takes gqa_decode_plan's choice, lowered if needed to the
 * largest split count whose scratch fits the array.  An explicit num_splits
 * whose scratch (gqa_decode_workspace_size) exceeds GQA_STATIC_WORKSPACE_BYTES
 * is rejected with GQA_ERR_WORKSPACE_TOO_SMALL.  q_scale finite and >= 0;
 * other rules as gqa_decode_prepared. */
#define GQA_STATIC_WORKSPACE_BYTES (16u << 20)
gqa_status_t gqa_decode_noalloc(const void* q, const void* kv, const int32_t* lens, void* out,
                                int batch, int capacity, gqa_dtype_t dtype, float q_scale,
                                int num_splits, void* stream);

/* The status word of the static scratch of gqa_decode_noalloc on the current
 * device (GQA_FLAG_* bits, accumulated since set-up or the last read): copies
 * it to *flags and clears it.  Like gqa_decode_get_status it synchronises
 * `stream`, so it is for checks outside the hot path, never inside a
 * capture.  Performs the static scratch's set-up if no call has yet (flags
 * are then 0).  The pages have no counterpart to this call. */
gqa_status_t gqa_decode_noalloc_get_status(void* stream, uint32_t* flags);

/* Test hook for the failure path (not for production use).  Launches stage 1
 * exactly as gqa_decode_split_stage does, except that the producer never
 * issues the copies of tile `skip_tile` (0-based, 64 tokens for fp16/bf16,
 * 128 for e4m3) of each split, so the consumers' wait on that tile runs out
 * after `wait_budget_ns` (1 ms .. 4 s).  Each affected CTA then sets
 * GQA_FLAG_WAIT_TIMEOUT in the workspace header, waits (bounded) for its own
 * copies in flight and returns; outputs and partials are invalid.  Lets a test
 * check that a stalled pipeline is reported to the host while the CUDA
 * context stays usable, without faulting or hanging the GPU. */
gqa_status_t gqa_decode_debug_skip_tile(const void* q, gqa_dtype_t q_dtype, const void* kv,
                                        gqa_kv_format_t kv_format, const int32_t* lens, void* out,
                                        int batch, int capacity, float q_scale, float k_scale,
                                        float v_scale, int num_splits, void* workspace,
                                        size_t workspace_bytes, int skip_tile,
                                        uint64_t wait_budget_ns, void* stream);

/* Test hook of the range-checked build (compiled with GQA_CHECKED; not for
 * production use).  From the next launch of this process on, the extents
 * that the split kernel's range checks compare against are cut short: the
 * KV cache (or page pool) by `kv_cut_bytes` and the int8 row scales by
 * `scales_cut_bytes` (each to 0 at most).  A cache access past the cut extent
 * then sets GQA_FLAG_BOUNDS and is redirected to an address inside the
 * buffer, as a real out-of-range access would be, so a test can see the
 * checks fire without any access leaving the real buffers; outputs of such
 * launches are invalid.  0, 0 restores the true extents.  The product build
 * has no range checks: there it accepts 0, 0 and rejects anything else with
 * GQA_ERR_INVALID_ARGUMENT.  The pages have no counterpart to this call. */
gqa_status_t gqa_decode_debug_cut_extents(uint64_t kv_cut_bytes, uint64_t scales_cut_bytes);

/* The step before decode: one new token per batch row (the "Qwen3-VL
 * official BF16 on Jetson Thor (SM110)" docs, "Runtime architecture": fused
 * kernels that normalise Q and K, rotate them and write the cache; decode
 * graphs keyed by (cache_pos,
 * rope_pos)).  For each query head and each KV head vector x of 128:
 *   y_d = x_d / sqrt(mean(x^2) + eps) * w_d     (w = q_norm_w or k_norm_w, [128])
 *   z_i = y_i cos a_i - y_{i+64} sin a_i,  z_{i+64} = y_{i+64} cos a_i + y_i sin a_i,
 *   a_i = positions[b] * rope_theta^(-i/64)     (rotate-half RoPE, i = 0..63)
 * q_out[b] <- z of the 32 query heads (dtype, RNE); the K plane of `kv` at
 * slot slots[b] <- z of the 8 key heads; the V plane at that slot <- v_proj
 * unchanged.  q_proj [batch,32,128], k_proj and v_proj [batch,8,128] and the
 * weights are `dtype`.  The cache format decides the write: fp16/bf16 (must
 * equal dtype; RNE), e4m3 (value / k_scale or / v_scale, RNE, saturating) or
 * int8 (codes round-to-nearest-even of value / scale with a fresh bf16 row
 * scale amax/127 written to kv_scales_bf16, clipped to +-127).  positions and
 * slots are int32 [batch] in device memory, read only by the kernel; a slot
 * outside [0, capacity) is not written and, when a workspace is given, sets
 * GQA_FLAG_SLOT_CLAMPED in its header (workspace may be NULL).  eps finite >= 0,
 * rope_theta finite > 0.  One launch, no allocation, no host sync.  A decode
 * that should see the new token uses len[b] = slots[b] + 1. */
gqa_status_t gqa_append_kv(const void* q_proj, const void* k_proj, const void* v_proj,
                           const void* q_norm_w, const void* k_norm_w, gqa_dtype_t dtype,
                           const int32_t* positions, const int32_t* slots, int batch, void* q_out,
                           void* kv, gqa_kv_format_t kv_format, uint16_t* kv_scales_bf16, int capacity,
                           float eps, float rope_theta, float k_scale, float v_scale, void* workspace,
                           size_t workspace_bytes, void* stream);

/* The same step on a paged cache (the layout of gqa_decode_paged): slot
 * slots[b] of row b is row slots[b] % page_size of page
 * block_table[b][slots[b] / page_size]; an int8 cache writes its fresh row
 * scale into kv_scales_pages [num_pages, 2, 8, page_size].  A slot outside
 * [0, max_pages_per_seq * page_size) sets GQA_FLAG_SLOT_CLAMPED and a
 * block-table entry outside [0, num_pages) sets GQA_FLAG_PAGE_CLAMPED; in both
 * cases nothing of that row is written to the cache (q_out still is).  Other
 * arguments and rules as gqa_append_kv. */
gqa_status_t gqa_append_kv_paged(const void* q_proj, const void* k_proj, const void* v_proj,
                                 const void* q_norm_w, const void* k_norm_w, gqa_dtype_t dtype,
                                 const int32_t* positions, const int32_t* slots, int batch,
                                 void* q_out, void* kv_pages, gqa_kv_format_t kv_format,
                                 uint16_t* kv_scales_pages, const int32_t* block_table,
                                 int max_pages_per_seq, int num_pages, int page_size, float eps,
                                 float rope_theta, float k_scale, float v_scale, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Zero the workspace header (status flags) on `stream`.  Asynchronous. */
gqa_status_t gqa_decode_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Debug only, never inside a capture: synchronises `stream`, copies the
 * status word of the workspace header to *flags (GQA_FLAG_* bits) and clears
 * it. */
gqa_status_t gqa_decode_get_status(void* workspace, size_t workspace_bytes, void* stream,
                                   uint32_t* flags);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H_ */
