/*
 * hpc_decode.h — C ABI of the load-balanced paged GQA decode-attention library
 * (libhpcdecode.so, CUDA for sm_103a).
 *
 * Sources the operations are taken from (two web posts about the HPC-Ops
 * attention backend):
 *   [vLLM]  "騰訊混元が vLLM に HPC オプス対応" (English text of the vLLM
 *           integration post), sections "The challenge: mixed-length decode
 *           in every batch" and "The solution: a per-step, load-balanced
 *           decode scheduler" (Assign / Compute and combine bullets).
 *   [SGL]   "腾讯HPC-Ops联手SGLang开源高性能MoE内核" (SGLang integration post),
 *           sections "Attention：变长decode的负载均衡", "围绕Live KV Work的调度"
 *           and "从HPC-Ops Kernel到SGLang".
 *
 * Conventions shared by every entry point:
 *   - All pointers named d_* or documented as "device" are CUDA device
 *     pointers owned by the caller.  The library never allocates or frees
 *     memory, never synchronises a stream (except hpc_decode_read_meta) and
 *     keeps no state between calls except a cached driver entry point and
 *     per-device launch facts (kernel attributes set, resident CTAs).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  Launch sizes depend only on
 *     host-known bounds, never on device data.
 *   - Kernels are launched as programmatic dependents of the previous kernel
 *     on the stream: they may become resident while it still runs, but none
 *     reads or writes caller data before that kernel has finished, with one
 *     exception internal to hpc_decode_step (and the entry points built on
 *     it): there the attention grid starts streaming its first tiles while
 *     the assign kernel it follows, which itself waited for everything
 *     before it, is still running.
 *   - The returned status covers host-side argument checks and the launch
 *     itself (cudaGetLastError).  Problems only visible on the device (bad
 *     seqlens, block-table entries out of range, a wait that timed out) are
 *     OR-ed as HPC_FLAG_* bits into map->meta[3], which the caller reads after
 *     the stream completes (hpc_decode_read_meta does that for you).
 *   - Fixed geometry: head_dim = 128, page (= tile) size = 64 tokens,
 *     G = Hq / Hkv query heads per KV head with 1 <= G <= 16.  Query head hq
 *     uses KV head hq / G (contiguous groups); one descriptor serves the
 *     whole group of its KV head ([vLLM] Compute and combine bullet).
 *   - Layouts are row-major:
 *       q         [B, Hq, 128]            bf16, or e4m3 for HPC_KV_FP8_E4M3
 *       q_scale   [B, Hq]                 fp32 (FP8 only): q = e4m3(q8) * q_scale
 *       k_cache,
 *       v_cache   [num_pages, 64, Hkv, 128]  bf16 or e4m3 (k = e4m3(k8) * k_scale)
 *       block_table [B, max_pages_per_req] int32 physical page ids; entries
 *                 past ceil(L_r / 64) are never read
 *       seqlens   [B] int32 live tokens per request (0 allowed)
 *       out       [B, Hq, 128] bf16
 *   - Base addresses of q, the caches, part_o and out must be 16-byte aligned.
 */
#ifndef HPC_DECODE_H
#define HPC_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void *hpc_stream_t; /* a cudaStream_t */

typedef enum {
    HPC_OK = 0,
    HPC_ERR_ARG = -1,         /* null pointer, negative size, misaligned pointer, bad enum */
    HPC_ERR_UNSUPPORTED = -2, /* head_dim != 128, G > 16, Hq % Hkv != 0, too large a batch */
    HPC_ERR_WORKSPACE = -3,   /* task-map capacity below what the plan may write */
    HPC_ERR_CUDA = -4         /* a CUDA runtime/driver call failed (launch, tensor map) */
} hpc_status;

typedef enum { HPC_KV_BF16 = 0, HPC_KV_FP8_E4M3 = 1 } hpc_kv_dtype;

/* Device-side error bits, OR-ed into meta[3]. */
#define HPC_FLAG_BAD_SEQLEN 1u   /* a seqlen < 0 or > 64 * max_pages_per_req; clamped */
#define HPC_FLAG_DESC_OVERFLOW 2u /* the plan needed more than cap_desc descriptors */
#define HPC_FLAG_BAD_PAGE 4u     /* a block-table entry outside [0, num_pages); page 0 read instead */
#define HPC_FLAG_TIMEOUT 8u      /* a pipeline wait hit its time limit; output invalid */

#define HPC_HEAD_DIM 128
#define HPC_PAGE_SIZE 64
#define HPC_MAX_GROUP 16
#define HPC_MAX_BATCH 16384
#define HPC_MAX_QUERY_ROWS 16 /* multi-query decode: q_len * G query rows per KV head at most */

/*
 * Task map: the device-side result of the assign step ([vLLM] Assign bullet;
 * [SGL] 围绕Live KV Work的调度).  All arrays are caller-owned device memory.
 *   desc        [cap_desc][4] int32 {kv_head, request, tile_begin, tile_end},
 *               tiles local to the request, bin-major order.
 *   bin_ptr     [num_ctas + 1] CSR offsets: CTA c drains
 *               desc[bin_ptr[c] .. bin_ptr[c+1]); an empty range is the
 *               terminator of an unused bin.
 *   chunk_count [Hkv * B] descriptors per unit u = kv_head * B + request.
 *   chunk_off   [Hkv * B] index of the unit's first descriptor; descriptor i
 *               writes split-buffer slot i.
 *   meta        [8] {total_tiles, budget, num_desc, error_flags, bin counter,
 *               reserved x3}; the bin counter is zeroed by the planners and
 *               left zero by every attention launch.
 * cap_desc, cap_bins and cap_units give the sizes of desc (entries of four
 * int32), bin_ptr and chunk_count / chunk_off, and are set by the caller.
 * B, Hkv, num_ctas (the number of bins), persistent, min_tiles and
 * max_pages (the planner's arguments) are written by the planners (the
 * host-side struct is updated) and read by hpc_decode_attn /
 * hpc_decode_combine, which check B and Hkv against their own arguments.
 * The attention kernel of a persistent map re-derives each CTA's first
 * descriptor from the sequence lengths so it can start before the map is
 * complete; the map and the sequence lengths must describe the same batch.
 * A persistent map (hpc_decode_plan) is drained by min(num_ctas, resident
 * CTAs) persistent CTAs: CTA c takes bin c first and, when there are more
 * bins than resident CTAs, pulls the remaining bins in order from the bin
 * counter, so faster SMs take more bins.  A static map
 * (hpc_decode_plan_static) launches one CTA per bin.
 */
typedef struct {
    int32_t *desc;
    int32_t *bin_ptr;
    int32_t *chunk_count;
    int32_t *chunk_off;
    int32_t *meta;
    int32_t cap_desc, cap_bins, cap_units;
    int32_t B, Hkv, num_ctas, persistent, min_tiles, max_pages;
} hpc_task_map;

/* Library version string (static storage). */
const char *hpc_decode_version(void);

/* Human-readable name of a status code (static storage). */
const char *hpc_status_string(hpc_status status);

/*
 * Number of persistent CTAs for the attention kernel on `device`: SM count x
 * resident CTAs per SM for that KV dtype's kernel.  Returns a negative
 * hpc_status on failure.  ([vLLM] "persistent kernel grid")
 */
int32_t hpc_decode_num_ctas(int32_t device, hpc_kv_dtype kv_dtype);

/*
 * Descriptor capacity that always suffices for hpc_decode_plan:
 * num_ctas + B * Hkv (a unit contributes one descriptor plus one per bin
 * boundary falling inside it, and there are at most num_ctas - 1 such
 * boundaries).  Returns -1 on negative arguments.
 */
int64_t hpc_decode_desc_capacity(int32_t B, int32_t Hkv, int32_t num_ctas);

/* Descriptor capacity for hpc_decode_plan_static: B * Hkv * num_splits. */
int64_t hpc_decode_static_capacity(int32_t B, int32_t Hkv, int32_t num_splits);

/*
 * Assign step ([vLLM] Assign bullet; [SGL] 围绕Live KV Work的调度): one CTA
 * cuts every request's live KV into 64-token tiles (n_r = ceil(L_r / 64)),
 * sums them over KV heads and requests (T = Hkv * sum n_r), sets the
 * per-CTA budget max(ceil(T / num_ctas), min_tiles_per_cta, 1), walks tiles
 * head-major / batch-minor and fills bins in order, spilling into the next
 * bin when one is full.  Writes the whole task map (every bin_ptr entry,
 * every chunk_count/chunk_off entry, desc[0 .. num_desc), meta[0..7]).
 * num_ctas is the number of bins: the pages' choice is one bin per
 * persistent CTA (hpc_decode_num_ctas); a small multiple of it lets the
 * attention kernel balance uneven SM speeds by pulling bins dynamically.
 * The map is meant to be built once per decode step and reused by every
 * layer's hpc_decode_attn / hpc_decode_combine.
 *   d_seqlens          device [B] int32
 *   B                  0 <= B <= HPC_MAX_BATCH
 *   Hkv                >= 1
 *   max_pages_per_req  block-table row length; a seqlen above 64 * this is
 *                      clamped and flagged HPC_FLAG_BAD_SEQLEN
 *   num_ctas           >= 1, the number of bins (see hpc_decode_num_ctas)
 *   min_tiles_per_cta  minimum-work floor (>= 0)
 *   map                cap_desc >= hpc_decode_desc_capacity(B, Hkv, num_ctas),
 *                      cap_bins >= num_ctas + 1 and cap_units >= B * Hkv,
 *                      else HPC_ERR_WORKSPACE
 */
hpc_status hpc_decode_plan(const int32_t *d_seqlens, int32_t B, int32_t Hkv,
                           int32_t max_pages_per_req, int32_t num_ctas,
                           int32_t min_tiles_per_cta, hpc_task_map *map, hpc_stream_t stream);

/*
 * In-house static split-KV comparator ([vLLM] "The challenge: mixed-length
 * decode in every batch", fixed number of splits; [SGL]
 * Attention：变长decode的负载均衡, strategy (1)).  Emits the same task-map
 * format with one bin (= one CTA) per (kv_head, request, split):
 * bin u * S + s of unit u = kv_head * B + request covers tiles
 * [s * k_r, min((s + 1) * k_r, n_r)) with k_r = ceil(n_r / S); empty splits
 * keep an empty descriptor (tile_begin == tile_end) and launch a CTA that
 * finds no work.  The map's num_ctas becomes B * Hkv * S, which is the grid
 * hpc_decode_attn then launches; meta[1] holds S.
 *   num_splits  S >= 1; cap_desc >= B * Hkv * S, cap_bins >= B * Hkv * S + 1,
 *               cap_units >= B * Hkv, else HPC_ERR_WORKSPACE.
 */
hpc_status hpc_decode_plan_static(const int32_t *d_seqlens, int32_t B, int32_t Hkv,
                                  int32_t max_pages_per_req, int32_t num_splits,
                                  hpc_task_map *map, hpc_stream_t stream);

/*
 * Persistent attention ([vLLM] Compute and combine bullet; [SGL]
 * 围绕Live KV Work的调度, execution paragraph): map->num_ctas CTAs; CTA c
 * drains bin c.  For descriptor i = (h, r, tb, te) it gathers K/V pages
 * block_table[r][tb .. te) of KV head h and computes, for the G query heads
 * h*G .. h*G+G-1 of request r, softmax attention over tokens
 * [64 tb, min(64 te, L_r)) with scores sm_scale * q.k, writing
 *     part_o[i][g][:]  = sum_j p_j v_j / sum_j p_j      (fp32, normalised)
 *     part_lse[i][g]   = log(sum_j exp(s_j))             (fp32, natural log)
 * Empty descriptors write nothing.  FP8: scores use q_scale[r][hq] * k_scale,
 * values v_scale; BF16 ignores the scales (pass NULL / 1).
 *   part_o    device [map->cap_desc, G, 128] fp32
 *   part_lse  device [map->cap_desc, G] fp32
 *   num_pages physical pages in each cache; a live block-table entry outside
 *             [0, num_pages) is replaced by page 0 (no out-of-bounds read) and
 *             flags HPC_FLAG_BAD_PAGE; that request's output is then invalid.
 */
hpc_status hpc_decode_attn(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                           const void *d_v_cache, int32_t num_pages, float k_scale, float v_scale,
                           hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                           int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                           int32_t Hq, int32_t Hkv, int32_t head_dim, float sm_scale,
                           const hpc_task_map *map, float *d_part_o, float *d_part_lse,
                           hpc_stream_t stream);

/*
 * hpc_decode_attn with the combine step folded into the same persistent
 * grid (the combine kernel's job, [vLLM] Compute and combine bullet, done
 * without a second launch).  A unit whose chunk count is 1 writes its BF16
 * output directly from the CTA that computed it; for a split unit every CTA
 * writes its partial, then counts the chunk in d_unit_done[u] (device-scope
 * fence before the atomic), and the CTA that brings the count to
 * chunk_count[u] merges the unit's partials into d_out exactly as
 * hpc_decode_combine does and resets the counter to 0 (chunks are counted,
 * and units merged, at the end of each CTA's work).  Nothing waits on
 * another CTA.  Requests with no live tokens get zero rows, as in
 * hpc_decode_combine.
 *   d_unit_done  device int32 [B * Hkv]; all zero before the call (clear it
 *                once after allocating); every completed call leaves it zero.
 *   d_out        device [B, Hq, 128] bf16
 * Other arguments as in hpc_decode_attn; part_o / part_lse are still needed
 * for the split units.
 */
hpc_status hpc_decode_attn_combine(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                                   const void *d_v_cache, int32_t num_pages, float k_scale,
                                   float v_scale, hpc_kv_dtype kv_dtype,
                                   const int32_t *d_block_table, int32_t max_pages_per_req,
                                   const int32_t *d_seqlens, int32_t B, int32_t Hq, int32_t Hkv,
                                   int32_t head_dim, float sm_scale, const hpc_task_map *map,
                                   float *d_part_o, float *d_part_lse, int32_t *d_unit_done,
                                   void *d_out, hpc_stream_t stream);

/*
 * Combine ([vLLM] Compute and combine bullet: "reads the chunk count for each
 * (head, request) pair"; [SGL] 围绕Live KV Work的调度: merge under the correct
 * global softmax normalisation).  For every (r, hq), with unit
 * u = (hq / G) * B + r, n = chunk_count[u], slots s = chunk_off[u] + i:
 *     M = max_i lse_i,  w_i = exp(lse_i - M),
 *     out[r][hq][:] = bf16_rn( sum_i w_i part_o[s_i] / sum_i w_i )
 * A unit with no chunks (L_r = 0) gets a zero row.
 *   d_out  device [B, Hq, 128] bf16
 */
hpc_status hpc_decode_combine(const float *d_part_o, const float *d_part_lse,
                              const hpc_task_map *map, int32_t B, int32_t Hq, int32_t Hkv,
                              int32_t head_dim, void *d_out, hpc_stream_t stream);

/* ------------------------------------------------------------------------
 * Multi-query decode (q_len > 1: the speculative / MTP layer of Hy3, vLLM
 * post "A Quick Word on Hy3-series models"; the pages' next-step item of
 * extend shapes with few query tokens).  Each request's last q_len live
 * tokens are queries; the caller has written their K and V into the cache
 * (L_r counts them).  Query token i of request r attends the live tokens
 * j < L_r - q_len + 1 + i (everything before it and itself).  The task map is
 * the same as for q_len = 1 (tiles count KV tokens); every descriptor serves
 * R = q_len * G query rows rho = i * G + g of its KV head, and each KV tile is
 * read once for all of them.  Layouts:
 *   q         [B, q_len, Hq, 128]   bf16, or e4m3 with q_scale [B, q_len, Hq]
 *   out       [B, q_len, Hq, 128]   bf16
 *   part_o    [cap, R, 128] fp32,   part_lse [cap, R] fp32 (R = q_len * G)
 * Requires 1 <= q_len and q_len * G <= HPC_MAX_QUERY_ROWS
 * (HPC_ERR_UNSUPPORTED otherwise).  A query row that sees no token (L_r <
 * q_len) is written as zeros.  Otherwise as the q_len = 1 calls, which are
 * these with q_len = 1.
 * ---------------------------------------------------------------------- */
hpc_status hpc_decode_attn_mq(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                              const void *d_v_cache, int32_t num_pages, float k_scale,
                              float v_scale, hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                              int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                              int32_t Hq, int32_t Hkv, int32_t head_dim, int32_t q_len,
                              float sm_scale, const hpc_task_map *map, float *d_part_o,
                              float *d_part_lse, hpc_stream_t stream);

hpc_status hpc_decode_attn_combine_mq(const void *d_q, const float *d_q_scale,
                                      const void *d_k_cache, const void *d_v_cache,
                                      int32_t num_pages, float k_scale, float v_scale,
                                      hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                                      int32_t max_pages_per_req, const int32_t *d_seqlens,
                                      int32_t B, int32_t Hq, int32_t Hkv, int32_t head_dim,
                                      int32_t q_len, float sm_scale, const hpc_task_map *map,
                                      float *d_part_o, float *d_part_lse, int32_t *d_unit_done,
                                      void *d_out, hpc_stream_t stream);

hpc_status hpc_decode_combine_mq(const float *d_part_o, const float *d_part_lse,
                                 const hpc_task_map *map, int32_t B, int32_t Hq, int32_t Hkv,
                                 int32_t head_dim, int32_t q_len, void *d_out,
                                 hpc_stream_t stream);

hpc_status hpc_decode_step_mq(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                              const void *d_v_cache, int32_t num_pages, float k_scale,
                              float v_scale, hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                              int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                              int32_t Hq, int32_t Hkv, int32_t head_dim, int32_t q_len,
                              float sm_scale, int32_t num_ctas, int32_t min_tiles_per_cta,
                              int32_t num_splits, hpc_task_map *map, float *d_part_o,
                              float *d_part_lse, int32_t *d_unit_done, void *d_out,
                              hpc_stream_t stream);

/*
 * One whole decode step of one layer on device buffers: hpc_decode_plan
 * (when num_splits == 0) or hpc_decode_plan_static (num_splits >= 1), then
 * either hpc_decode_attn_combine (d_unit_done != NULL) or hpc_decode_attn
 * followed by hpc_decode_combine (d_unit_done == NULL), all on `stream`.
 * Arguments as in those calls.  In a real model the plan is built once per
 * step and shared by all layers; this call rebuilds it every time.
 */
hpc_status hpc_decode_step(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                           const void *d_v_cache, int32_t num_pages, float k_scale, float v_scale,
                           hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                           int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                           int32_t Hq, int32_t Hkv, int32_t head_dim, float sm_scale,
                           int32_t num_ctas, int32_t min_tiles_per_cta, int32_t num_splits,
                           hpc_task_map *map, float *d_part_o, float *d_part_lse,
                           int32_t *d_unit_done, void *d_out, hpc_stream_t stream);

/*
 * hpc_decode_step with the per-step inputs and the output in host memory:
 * brings h_q, h_q_scale (FP8 only), h_seqlens and h_block_table into the
 * caller's device staging buffers d_q, d_q_scale, d_seqlens, d_block_table,
 * runs the step, and copies d_out back into h_out.  When every input is
 * pinned host memory with a device alias, one copy kernel reads them all
 * through their aliases (16-byte vectors where both addresses are 16-byte
 * aligned, bytes otherwise) and the assign kernel launches behind it as a
 * programmatic dependent; otherwise each array is one cudaMemcpyAsync
 * (synchronous for pageable memory).  The KV caches stay device-resident, as
 * they are in serving.  Pinned inputs are read asynchronously: the caller
 * rewrites them only after `stream` has passed the step.  The host output is
 * complete once `stream` has finished.
 */
hpc_status hpc_decode_step_host(const void *h_q, const float *h_q_scale, const int32_t *h_seqlens,
                                const int32_t *h_block_table, void *h_out, void *d_q,
                                float *d_q_scale, int32_t *d_seqlens, int32_t *d_block_table,
                                void *d_out, const void *d_k_cache, const void *d_v_cache,
                                int32_t num_pages, float k_scale, float v_scale,
                                hpc_kv_dtype kv_dtype, int32_t max_pages_per_req, int32_t B,
                                int32_t Hq, int32_t Hkv, int32_t head_dim, float sm_scale,
                                int32_t num_ctas, int32_t min_tiles_per_cta, int32_t num_splits,
                                hpc_task_map *map, float *d_part_o, float *d_part_lse,
                                int32_t *d_unit_done, hpc_stream_t stream);

/*
 * Layout of the packed per-step input of hpc_decode_step_host_packed: one
 * buffer holding the query, the FP8 query scales (FP8 only), the seqlens and
 * the block table, each section starting on a 16-byte boundary.  Writes the
 * byte offsets {q, q_scale (-1 for BF16), seqlens, block_table} to offsets[4]
 * and returns the total size in bytes (-1 for invalid arguments).  Sections
 * are laid out exactly as the separate arrays of hpc_decode_step.
 */
int64_t hpc_decode_packed_layout(int32_t B, int32_t Hq, int32_t max_pages_per_req,
                                 hpc_kv_dtype kv_dtype, int64_t offsets[4]);

/*
 * hpc_decode_step_host with the per-step inputs in ONE host buffer h_in
 * (the layout of hpc_decode_packed_layout) brought into the caller's device
 * staging buffer d_in (same size, 16-byte aligned), the step on the device
 * sections, and one device-to-host copy of d_out into h_out.  Pinned h_in
 * (with a 16-byte-aligned device alias) is read by a copy kernel through its
 * alias, one 16-byte load per thread, with the assign kernel launched as its
 * programmatic dependent (the caller rewrites h_in only after `stream` has
 * passed the step); pageable h_in goes through the copy engine
 * (cudaMemcpyAsync, synchronous for pageable memory).  The same bytes move as
 * with the separate buffers, in one transfer each way.  With d_out NULL (and
 * d_unit_done given: the combine fused into the attention grid) the kernels
 * store the BF16 output straight into h_out, which must then be pinned host
 * memory with a device alias (cudaHostAlloc memory under unified addressing;
 * HPC_ERR_ARG otherwise): no separate copy out.
 */
hpc_status hpc_decode_step_host_packed(const void *h_in, void *d_in, void *h_out, void *d_out,
                                       const void *d_k_cache, const void *d_v_cache,
                                       int32_t num_pages, float k_scale, float v_scale,
                                       hpc_kv_dtype kv_dtype, int32_t max_pages_per_req,
                                       int32_t B, int32_t Hq, int32_t Hkv, int32_t head_dim,
                                       float sm_scale, int32_t num_ctas,
                                       int32_t min_tiles_per_cta, int32_t num_splits,
                                       hpc_task_map *map, float *d_part_o, float *d_part_lse,
                                       int32_t *d_unit_done, hpc_stream_t stream);

/*
 * Size of the scratch array compiled into the library for
 * hpc_decode_step_noalloc.
 */
#define HPC_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * hpc_decode_step for callers that cannot allocate device memory.  The
 * posts describe nothing like it; it exists for callers that may not call
 * cudaMalloc when they run attention (code under an allocator they do not
 * own, plug-ins whose host forbids device allocation after start-up, tools
 * that must leave the memory state untouched).  They pass only the inputs
 * and the output; the task map and the split buffer live in one
 * HPC_NOALLOC_SCRATCH_BYTES array inside the library, which every GPU that
 * loads the library holds until the process exits.  The call allocates
 * nothing and frees nothing.
 *   Arguments as in hpc_decode_step (load-balanced plan only), plus
 *   d_out       device [B, Hq, 128] bf16, written
 *   d_meta_out  device int32[4] or NULL: receives the step's
 *               {total_tiles, budget, num_desc, error_flags}
 * Limits: the scratch must hold (num_ctas + B*Hkv) descriptors with their
 * partials, G * 516 + 16 bytes each (about 4.2 KB at G = 8, roughly 1,900
 * descriptors; 8.3 KB at G = 16, roughly 1,000); larger problems get
 * HPC_ERR_WORKSPACE before anything is launched, and unsupported shapes the
 * same status as hpc_decode_step.
 * The first call in a CUDA context looks up the array's device address in
 * that context (with its device current) and caches it under the context's
 * id; make that first call before any stream capture.  A device reset or a
 * different current context (cuCtxSetCurrent) makes the next call look the
 * address up again.  All calls share the one array and leave their contents
 * in it: calls that overlap on the GPU (other streams, other host threads)
 * race and must be serialised by the caller.
 */
hpc_status hpc_decode_step_noalloc(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                                   const void *d_v_cache, int32_t num_pages, float k_scale,
                                   float v_scale, hpc_kv_dtype kv_dtype,
                                   const int32_t *d_block_table, int32_t max_pages_per_req,
                                   const int32_t *d_seqlens, int32_t B, int32_t Hq, int32_t Hkv,
                                   int32_t head_dim, float sm_scale, int32_t num_ctas,
                                   int32_t min_tiles_per_cta, void *d_out, int32_t *d_meta_out,
                                   hpc_stream_t stream);

/* ------------------------------------------------------------------------
 * Fused attention prologue (HpcRopeNorm).
 *
 * vLLM integration post, "A fused attention prologue"; SGLang post, the
 * paragraph on the Hy3 FP8 prologue: starting from the fused QKV projection
 * of the new tokens, one kernel applies QK-Norm and RoPE in the model's
 * order (Hy3 normalises first), writes K and V straight into the paged
 * cache and, for FP8, emits the query as E4M3 with one scale per
 * (token, head), which hpc_decode_attn takes as it is (q, q_scale).
 *
 * The posts give no constants; the op takes them as parameters and uses
 * the standard definitions:
 *   RMS norm of a head row x:  x / sqrt(mean(x^2) + eps) * w, with one BF16
 *     weight vector w[128] for all query heads and one for all key heads;
 *   RoPE over the whole head: frequency i < 64 is base^(-2i/128); the pair
 *     (a, b) turns by pos * freq_i into (a cos - b sin, b cos + a sin);
 *     pairs are (i, i + 64) for HPC_ROPE_HALVES, (2i, 2i + 1) for
 *     HPC_ROPE_INTERLEAVED;
 *   V is not normalised or rotated;
 *   FP8 query: scale = amax / 448 over the head row (1 for an all-zero
 *     row), codes = E4M3 round-to-nearest-even of y / scale (saturating);
 *   FP8 K and V: E4M3 of y / k_scale and v / v_scale (saturating).
 * The arithmetic is fp32.  The rotation angle pos * freq is formed as an
 * exact fp32 product plus its rounding error against an fp64 frequency and
 * reduced modulo 2 pi in extended precision, so every position below 2^24
 * keeps an angle error of a few 1e-7 rad; max_pages_per_req * 64 must not
 * exceed 2^24 (HPC_ERR_UNSUPPORTED).
 * ---------------------------------------------------------------------- */
typedef enum { HPC_ROPE_HALVES = 0, HPC_ROPE_INTERLEAVED = 1 } hpc_rope_layout;

typedef struct {
    float eps;           /* RMS-norm epsilon, finite, >= 0 */
    float rope_base;     /* RoPE base, finite, > 0 */
    int32_t rope_layout; /* hpc_rope_layout */
    int32_t norm_first;  /* 1: QK-Norm then RoPE (Hy3); 0: RoPE then QK-Norm */
    const double *freq;  /* device fp64 [64] from hpc_rope_frequencies(rope_base), 16-byte
                            aligned, or NULL: every CTA then builds the table itself in fp64,
                            which costs a couple of microseconds at the start of the kernel */
} hpc_rope_norm_params;

/*
 * Writes the 64 RoPE frequencies rope_base^(-2i/128), i = 0..63, in fp64 into
 * d_freq (device, 16-byte aligned, caller-owned): the table a model builds
 * once and passes to every hpc_rope_norm call through params->freq.
 * Asynchronous on `stream`; HPC_ERR_ARG for a non-positive or non-finite base.
 */
hpc_status hpc_rope_frequencies(float rope_base, double *d_freq, hpc_stream_t stream);

/*
 * Runs the prologue for num_tokens new tokens.
 *   d_qkv          device bf16 [num_tokens, qkv_row_stride]; a token's row
 *                  holds Hq query heads, then Hkv key heads, then Hkv value
 *                  heads, 128 elements each; qkv_row_stride (elements) is
 *                  >= (Hq + 2 Hkv) * 128 and a multiple of 8
 *   d_q_norm_w, d_k_norm_w  device bf16 [128]
 *   d_positions    device int32 [num_tokens]: the token's position in its
 *                  request, which is both its RoPE position and its cache slot
 *   d_token_req    device int32 [num_tokens] (the token's request) or NULL,
 *                  meaning token t belongs to request t (decode)
 *   d_block_table  device int32 [B, max_pages_per_req]
 *   d_k_cache, d_v_cache  device [num_pages, 64, Hkv, 128] of kv_dtype;
 *                  token t of request r at position p is written to page
 *                  block_table[r, p / 64], slot p % 64; nothing else changes
 *   d_q_out        device [num_tokens, Hq, 128]: bf16 (BF16 KV) or e4m3 (FP8 KV)
 *   d_q_scale_out  device fp32 [num_tokens, Hq]: FP8 only (NULL for BF16)
 *   d_flags        device int32 or NULL: OR-ed with HPC_FLAG_BAD_SEQLEN when
 *                  a token's request or position is out of range and with
 *                  HPC_FLAG_BAD_PAGE when its page is outside [0, num_pages);
 *                  such a token still gets its query but writes no cache slot
 * All device pointers 16-byte aligned; the caller owns every buffer.  Two
 * tokens that name the same cache slot leave either one's row there.
 * Asynchronous on `stream`.  The kernel waits for the preceding kernel on
 * the stream to finish before it reads anything (it may be launched early
 * as a programmatic dependent of it) and lets its own dependents start only
 * when it has finished, so an attention launch that follows sees the new
 * cache rows.  Returns HPC_ERR_ARG / HPC_ERR_UNSUPPORTED on bad arguments
 * (head_dim != 128, Hq % Hkv != 0), HPC_ERR_CUDA if the launch fails.
 */
hpc_status hpc_rope_norm(const void *d_qkv, int64_t qkv_row_stride, const void *d_q_norm_w,
                         const void *d_k_norm_w, const int32_t *d_positions,
                         const int32_t *d_token_req, int32_t num_tokens, int32_t Hq, int32_t Hkv,
                         int32_t head_dim, const int32_t *d_block_table,
                         int32_t max_pages_per_req, int32_t B, void *d_k_cache, void *d_v_cache,
                         int32_t num_pages, hpc_kv_dtype kv_dtype, float k_scale, float v_scale,
                         void *d_q_out, float *d_q_scale_out, int32_t *d_flags,
                         const hpc_rope_norm_params *params, hpc_stream_t stream);

/*
 * Self-test of the bounded waits every kernel here relies on (each waits on
 * a barrier for at most a time limit, then raises HPC_FLAG_TIMEOUT and leaves
 * instead of hanging): launches one CTA that waits on a shared-memory barrier
 * nothing completes, with a limit of limit_us microseconds (1 .. 10^6).  When
 * the limit passes the kernel ORs HPC_FLAG_TIMEOUT into *d_flags (device
 * int32) and returns; the context stays usable.  HPC_ERR_ARG for a null flag
 * word or a limit out of range.  Asynchronous on `stream`.
 */
hpc_status hpc_selftest_wait_timeout(int32_t *d_flags, int32_t limit_us, hpc_stream_t stream);

/* ------------------------------------------------------------------------
 * Router GEMM with FP32 weights on BF16 tensor cores (SGLang post, section
 * "Router GEMM：在路由精度与吞吐量之间取得平衡", and its summary bullet): the
 * FP32 router weight W is split once into W_high, its BF16 truncation (low 16
 * bits dropped), and W_low, the round-to-nearest BF16 of (W - W_high) * 256,
 * so W ~ W_high + W_low / 256; the scores are
 *     S = X W_high^T + (X W_low^T) / 256,
 * both products accumulated in FP32 (tcgen05 tensor cores, TMEM
 * accumulators), the 1/256 applied in the epilogue.  The split keeps every
 * weight within 2^-16 of its magnitude.
 * ---------------------------------------------------------------------- */

/*
 * Splits d_w (device fp32 [N, K], row-major: experts x hidden, a Linear
 * layer's weight) into d_w_hi and d_w_lo (device bf16 [N, K]).  Done once,
 * when the weights are loaded.  Asynchronous on `stream`.
 */
hpc_status hpc_router_split(const float *d_w, int32_t N, int32_t K, void *d_w_hi, void *d_w_lo,
                            hpc_stream_t stream);

/*
 * Bytes of the fp32 workspace hpc_router_gemm uses on the current device for
 * this shape (split-K partials when tokens are few); 0 when it needs none,
 * -1 for a shape it does not support.
 */
int64_t hpc_router_workspace_bytes(int32_t M, int32_t N, int32_t K);

/*
 * The launch hpc_router_gemm makes for this shape on the current device with
 * a full workspace, in plan[4] (host int32): plan[0] = 1 for the tensor-core
 * kernel, 0 for the few-token CUDA-core kernel (M <= 16); plan[1] = experts
 * per CTA; plan[2] = K splits; plan[3] = CTAs launched.  HPC_ERR_ARG /
 * HPC_ERR_UNSUPPORTED as hpc_router_gemm; HPC_ERR_CUDA when the tensor-core
 * plan needs a device and none is present.
 */
hpc_status hpc_router_plan(int32_t M, int32_t N, int32_t K, int32_t *plan);

/*
 * S = X W_high^T + (X W_low^T) / 256 for d_x (device bf16 [M, K], row-major
 * tokens x hidden) into d_out (device fp32 [M, N]).  K must be a multiple of
 * 64 and N of 16 (HPC_ERR_UNSUPPORTED otherwise); all pointers 16-byte
 * aligned.  d_workspace (hpc_router_workspace_bytes bytes, or less: the call
 * then uses fewer K splits, down to none) holds split-K partials, which a
 * second kernel sums in a fixed order, so the result is deterministic.
 * d_flags (device int32 or NULL) gets HPC_FLAG_TIMEOUT if a pipeline wait
 * timed out (output invalid).  Asynchronous on `stream`; reads X only after
 * the previous kernel on the stream has finished.
 */
hpc_status hpc_router_gemm(const void *d_x, const void *d_w_hi, const void *d_w_lo, int32_t M,
                           int32_t N, int32_t K, float *d_out, void *d_workspace,
                           int64_t workspace_bytes, int32_t *d_flags, hpc_stream_t stream);

/* ------------------------------------------------------------------------
 * Extend / prefill attention (vLLM post, "Attention: HPC-Ops vs
 * FlashAttention / Triton / FlashInfer", Table 4's prefill and extend rows):
 * many new query tokens per request over the paged BF16 cache, on tcgen05
 * tensor cores.  Request r holds L_r live tokens (d_seqlens, device); its
 * last q_len tokens are the queries, already written into the cache, and
 * query token i (position L_r - q_len + i) attends the tokens j <= L_r -
 * q_len + i (causal).  A prefill is L_r = q_len; an extend has a cached
 * prefix.  No task map: one CTA per (request, query head, 128 query tokens).
 *   d_q        [B, q_len, Hq, 128] bf16, 16-byte aligned
 *   caches     [num_pages, 64, Hkv, 128] bf16 (as for decode)
 *   d_out      [B, q_len, Hq, 128] bf16, written for every query row; a row
 *              that sees no token (L_r < q_len) is written as zeros
 * Query head hq reads KV head hq / (Hq / Hkv); Hq % Hkv must be 0 and
 * head_dim 128 (HPC_ERR_UNSUPPORTED otherwise).  d_flags (device int32 or
 * NULL) gets HPC_FLAG_BAD_SEQLEN for a length outside [0, 64 *
 * max_pages_per_req] (clamped), HPC_FLAG_BAD_PAGE for a page outside [0,
 * num_pages) (not read; that request's output is invalid) and
 * HPC_FLAG_TIMEOUT if a pipeline wait timed out.  Asynchronous on `stream`;
 * reads its inputs only after the previous kernel on the stream has
 * finished.  The caller owns all memory.
 * ---------------------------------------------------------------------- */
hpc_status hpc_prefill_attn(const void *d_q, const void *d_k_cache, const void *d_v_cache,
                            int32_t num_pages, const int32_t *d_block_table,
                            int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                            int32_t Hq, int32_t Hkv, int32_t head_dim, int32_t q_len,
                            float sm_scale, void *d_out, int32_t *d_flags, hpc_stream_t stream);

/*
 * Synchronises `stream` and copies map->meta into host_meta[4]
 * ({total_tiles, budget, num_desc, error_flags}).
 */
hpc_status hpc_decode_read_meta(const hpc_task_map *map, int32_t host_meta[4],
                                hpc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HPC_DECODE_H */
