// Internal declarations shared by the kernels' translation units and the
// host-side entry points.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "hpc_decode.h"

namespace hpc {

constexpr int kHeadDim = 128;
constexpr int kTile = 64;  // tokens per tile = tokens per page
constexpr int kMaxRows = 16;  // query rows of one KV head in a descriptor: q_len * G
constexpr int kConsumerWarps = 4;  // consumer warps per tile of a stage
constexpr int kPlanThreads = 1024;

// Stage flags written by the producer for the consumers.
constexpr int kFirst = 1;  // first tile of a descriptor (Q is in this stage)
constexpr int kLast = 2;   // last tile of a descriptor
constexpr int kEnd = 4;    // terminator: the bin is drained

struct AttnParams {
    const int32_t *bin_ptr;
    const int4 *desc;
    const int32_t *chunk_count;
    const int32_t *chunk_off;
    const int32_t *seqlens;
    const int32_t *block_table;
    const void *q;
    const float *q_scale;
    float *part_o;
    float *part_lse;
    int32_t *meta;
    int32_t *unit_done;  // fused mode: per-unit chunk counters (zero between launches)
    void *out;           // fused mode: BF16 output; nullptr = write partials only
    int *bin_counter;  // dynamic bins: next bin to pull, minus the grid size
    int num_bins;      // bins in the task map (>= the grid size)
    int min_tiles;     // floor the map was planned with (load-balanced maps)
    int fly;           // 1: derive the first descriptor from the seqlens (load-balanced maps)
    int B, Hq, Hkv, G, max_pages, num_pages;
    int q_len;  // query tokens per request (the last q_len live tokens; causal among them)
    int R;      // query rows per KV head: q_len * G (row rho = i * G + g)
    float score_scale;  // sm_scale * log2(e), times k_scale for FP8
    float v_scale;      // 1 for BF16
};

// Attention kernel configuration for one KV dtype and row-block count nb
// (query rows per KV head R <= 8 nb; nb = 1 or 2).
struct AttnConfig {
    const void *kernel;
    int smem_bytes;
    int threads;
};

AttnConfig attn_config_bf16(int nb);
AttnConfig attn_config_fp8(int nb);

cudaError_t launch_attn_bf16(int nb, const CUtensorMap &tk, const CUtensorMap &tv,
                             const AttnParams &p, int grid, cudaStream_t s);
cudaError_t launch_attn_fp8(int nb, const CUtensorMap &tk, const CUtensorMap &tv,
                            const AttnParams &p, int grid, cudaStream_t s);

// bt_prefetch (or null): a block table [B, max_pages] the kernel warms in L2
// for the attention grid that follows it.
cudaError_t launch_assign(const int32_t *seqlens, int B, int Hkv, int max_pages, int num_ctas,
                          int floor, const hpc_task_map &map, cudaStream_t s,
                          const int32_t *bt_prefetch = nullptr);
cudaError_t launch_static_plan(const int32_t *seqlens, int B, int Hkv, int max_pages,
                               int num_splits, const hpc_task_map &map, cudaStream_t s);
int assign_smem_bytes(int B);

// cuTensorMapEncodeTiled from the driver (nullptr when unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// TMA tensor map over one paged cache [num_pages, 64, Hkv, 128] (BF16: one
// 64-dim half of one head's page per load, 128-byte swizzle; FP8: the whole
// 128-byte rows of one head's page).
hpc_status cache_tensor_map(CUtensorMap *m, const void *base, int32_t num_pages, int32_t Hkv,
                            bool fp8);

cudaError_t launch_combine(const float *part_o, const float *part_lse, const hpc_task_map &map,
                           int B, int Hq, int Hkv, int q_len, void *out, cudaStream_t s);

}  // namespace hpc
