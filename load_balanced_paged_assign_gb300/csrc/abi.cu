// Host side of the C ABI declared in include/hpc_decode.h: argument checks,
// TMA tensor maps over the paged caches, and kernel launches.  No device
// memory is allocated or freed here and no stream is synchronised except by
// hpc_decode_read_meta.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

using namespace hpc;

namespace {

constexpr float kLog2eF = 1.4426950408889634f;
constexpr int kMaxDevices = 64;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// Per-device "dynamic shared memory attribute already raised" bits.
std::atomic<unsigned> g_attr_done[kMaxDevices];

cudaError_t prepare_kernel(const AttnConfig &cfg, int which) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned bit = 1u << which;
    if (dev >= 0 && dev < kMaxDevices && (g_attr_done[dev].load() & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(cfg.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             cfg.smem_bytes);
    if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) g_attr_done[dev].fetch_or(bit);
    return e;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

hpc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA; }

hpc_status check_shapes(int32_t B, int32_t Hq, int32_t Hkv, int32_t head_dim,
                        int32_t max_pages) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || max_pages <= 0) return HPC_ERR_ARG;
    if (head_dim != HPC_HEAD_DIM) return HPC_ERR_UNSUPPORTED;
    if (Hq % Hkv != 0 || Hq / Hkv > HPC_MAX_GROUP) return HPC_ERR_UNSUPPORTED;
    if (B > HPC_MAX_BATCH) return HPC_ERR_UNSUPPORTED;
    // every tile count and tile index must fit comfortably in int32
    if ((int64_t)B * max_pages * Hkv >= (int64_t)1 << 30) return HPC_ERR_UNSUPPORTED;
    return HPC_OK;
}

hpc_status check_map(const hpc_task_map *map, bool need_units) {
    if (!map || !map->desc || !map->bin_ptr || !map->meta) return HPC_ERR_ARG;
    if (need_units && (!map->chunk_count || !map->chunk_off)) return HPC_ERR_ARG;
    if (map->cap_desc < 0 || map->cap_bins < 0 || map->cap_units < 0) return HPC_ERR_ARG;
    if (!aligned16(map->desc)) return HPC_ERR_ARG;
    return HPC_OK;
}

// Tensor map over one paged cache, [num_pages, 64, Hkv, 128].
//  BF16: rank 5 {64 dims, 2 halves, Hkv, 64 tokens, pages}, box {64, 1, 1, 64, 1}:
//        each load brings one 64-dim half of one head's page as 64 rows of
//        128 B (the 128-byte swizzle span), so a row index is a token index.
//  FP8:  rank 4 {128 dims, Hkv, 64 tokens, pages}, box {128, 1, 64, 1}.
hpc_status make_cache_map(CUtensorMap *m, const void *base, int32_t num_pages, int32_t Hkv,
                          bool fp8) {
    auto encode = encoder();
    if (!encode) return HPC_ERR_CUDA;
    std::memset(m, 0, sizeof(*m));
    const cuuint64_t row = (cuuint64_t)Hkv * HPC_HEAD_DIM * (fp8 ? 1 : 2);  // bytes per token
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    CUresult r;
    if (fp8) {
        cuuint64_t dims[4] = {HPC_HEAD_DIM, (cuuint64_t)Hkv, HPC_PAGE_SIZE, (cuuint64_t)num_pages};
        cuuint64_t strides[3] = {HPC_HEAD_DIM, row, row * HPC_PAGE_SIZE};
        cuuint32_t box[4] = {HPC_HEAD_DIM, 1, HPC_PAGE_SIZE, 1};
        r = encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides,
                   box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[5] = {64, 2, (cuuint64_t)Hkv, HPC_PAGE_SIZE, (cuuint64_t)num_pages};
        cuuint64_t strides[4] = {128, 2 * 128, row, row * HPC_PAGE_SIZE};
        cuuint32_t box[5] = {64, 1, 1, HPC_PAGE_SIZE, 1};
        r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides,
                   box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS ? HPC_OK : HPC_ERR_CUDA;
}

// Resident CTAs of the attention kernel per device and variant (KV dtype x
// row blocks; cached).
std::atomic<int> g_capacity[kMaxDevices][4];

int resident_ctas(const AttnConfig &cfg, int which) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    int c = g_capacity[dev][which].load();
    if (c > 0) return c;
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cfg.kernel, cfg.threads,
                                                      cfg.smem_bytes) != cudaSuccess ||
        per_sm < 1)
        return -1;
    c = sms * per_sm;
    g_capacity[dev][which].store(c);
    return c;
}

// Kernel variant: KV dtype x row blocks (nb = 1: up to 8 query rows per KV
// head, 2: up to 16).
int variant_of(hpc_kv_dtype dt, int nb) { return (dt == HPC_KV_FP8_E4M3 ? 1 : 0) + 2 * (nb - 1); }

const AttnConfig &config_for(hpc_kv_dtype dt, int nb = 1) {
    static const AttnConfig cfg[4] = {attn_config_bf16(1), attn_config_fp8(1),
                                      attn_config_bf16(2), attn_config_fp8(2)};
    return cfg[variant_of(dt, nb)];
}

// Shared body of hpc_decode_attn (unit_done == out == nullptr: partials only)
// and hpc_decode_attn_combine (fused combine).
hpc_status launch_attention(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                            const void *d_v_cache, int32_t num_pages, float k_scale,
                            float v_scale, hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                            int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                            int32_t Hq, int32_t Hkv, int32_t head_dim, float sm_scale,
                            const hpc_task_map *map, float *d_part_o, float *d_part_lse,
                            int32_t *d_unit_done, void *d_out, bool after_plan, int32_t q_len,
                            hpc_stream_t stream) {
    hpc_status st = check_shapes(B, Hq, Hkv, head_dim, max_pages_per_req);
    if (st != HPC_OK) return st;
    if (q_len < 1) return HPC_ERR_ARG;
    if (q_len * (Hq / Hkv) > HPC_MAX_QUERY_ROWS) return HPC_ERR_UNSUPPORTED;
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_ARG;
    const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
    if (num_pages <= 0 || !d_k_cache || !d_v_cache || !d_part_o || !d_part_lse)
        return HPC_ERR_ARG;
    if (B > 0 && (!d_q || !d_block_table || !d_seqlens)) return HPC_ERR_ARG;
    if (fp8 && B > 0 && !d_q_scale) return HPC_ERR_ARG;
    if (!aligned16(d_q) || !aligned16(d_k_cache) || !aligned16(d_v_cache) ||
        !aligned16(d_part_o))
        return HPC_ERR_ARG;
    if (!std::isfinite(sm_scale) || (fp8 && (!std::isfinite(k_scale) || !std::isfinite(v_scale))))
        return HPC_ERR_ARG;
    st = check_map(map, false);
    if (st != HPC_OK) return st;
    if (map->B != B || map->Hkv != Hkv || map->num_ctas < 1 || map->num_ctas >= map->cap_bins)
        return HPC_ERR_ARG;

    CUtensorMap tk, tv;
    st = make_cache_map(&tk, d_k_cache, num_pages, Hkv, fp8);
    if (st == HPC_OK) st = make_cache_map(&tv, d_v_cache, num_pages, Hkv, fp8);
    if (st != HPC_OK) return st;

    AttnParams p;
    p.bin_ptr = map->bin_ptr;
    p.desc = reinterpret_cast<const int4 *>(map->desc);
    p.chunk_count = map->chunk_count;
    p.chunk_off = map->chunk_off;
    p.unit_done = d_unit_done;
    p.out = d_out;
    p.seqlens = d_seqlens;
    p.block_table = d_block_table;
    p.q = d_q;
    p.q_scale = d_q_scale;
    p.part_o = d_part_o;
    p.part_lse = d_part_lse;
    p.meta = map->meta;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.max_pages = max_pages_per_req;
    p.num_pages = num_pages;
    p.q_len = q_len;
    p.R = q_len * p.G;
    p.score_scale = sm_scale * kLog2eF * (fp8 ? k_scale : 1.f);
    p.v_scale = fp8 ? v_scale : 1.f;

    const int nb = p.R > 8 ? 2 : 1;
    const AttnConfig &cfg = config_for(kv_dtype, nb);
    cudaError_t e = prepare_kernel(cfg, variant_of(kv_dtype, nb));
    if (e != cudaSuccess) return HPC_ERR_CUDA;
    int grid = map->num_ctas;  // static map: one CTA per bin
    if (map->persistent) {     // persistent: resident CTAs, extra bins pulled dynamically
        const int cap = resident_ctas(cfg, variant_of(kv_dtype, nb));
        if (cap < 1) return HPC_ERR_CUDA;
        grid = std::min(grid, cap);
    }
    const bool pulls_bins = map->persistent && map->num_ctas > grid;
    p.num_bins = map->num_ctas;
    p.bin_counter = map->meta + 4;
    p.min_tiles = map->min_tiles;
    // The first descriptor is derived in-kernel, and streamed before the grid
    // waits on its predecessor, only right behind this library's own assign
    // kernel: that kernel waited for everything before it, so the caller's
    // inputs are complete.  Behind any other kernel (a reused map) every read
    // waits.  The map must be load-balanced and planned for this block table.
    // Not with more bins than CTAs: a CTA pulls its next bin once it has read
    // the map, and a derived first descriptor that spans the whole bin would
    // delay that read to the bin's end, so the CTAs whose first bin is one
    // descriptor would pull late and the others take more bins than their share.
    p.fly = after_plan && map->persistent && map->max_pages == max_pages_per_req && !pulls_bins
                ? 1
                : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = fp8 ? launch_attn_fp8(nb, tk, tv, p, grid, s) : launch_attn_bf16(nb, tk, tv, p, grid, s);
    return cuda_status(e);
}

// hpc_decode_attn_combine's checks and launch; after_plan as in launch_attention.
hpc_status attn_combine(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                        const void *d_v_cache, int32_t num_pages, float k_scale, float v_scale,
                        hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                        int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                        int32_t Hq, int32_t Hkv, int32_t head_dim, float sm_scale,
                        const hpc_task_map *map, float *d_part_o, float *d_part_lse,
                        int32_t *d_unit_done, void *d_out, bool after_plan, int32_t q_len,
                        hpc_stream_t stream) {
    if (B > 0 && (!d_unit_done || !d_out)) return HPC_ERR_ARG;
    if (!aligned16(d_out)) return HPC_ERR_ARG;
    if (!map || !map->chunk_count || !map->chunk_off) return HPC_ERR_ARG;
    if ((int64_t)B * Hkv > map->cap_units) return HPC_ERR_ARG;
    return launch_attention(d_q, d_q_scale, d_k_cache, d_v_cache, num_pages, k_scale, v_scale,
                            kv_dtype, d_block_table, max_pages_per_req, d_seqlens, B, Hq, Hkv,
                            head_dim, sm_scale, map, d_part_o, d_part_lse, d_unit_done, d_out,
                            after_plan, q_len, stream);
}

// hpc_decode_combine_mq's checks and launch.
hpc_status combine_impl(const float *d_part_o, const float *d_part_lse, const hpc_task_map *map,
                        int32_t B, int32_t Hq, int32_t Hkv, int32_t head_dim, int32_t q_len,
                        void *d_out, hpc_stream_t stream) {
    hpc_status st = check_shapes(B, Hq, Hkv, head_dim, 1);
    if (st != HPC_OK) return st;
    if (q_len < 1) return HPC_ERR_ARG;
    if (q_len * (Hq / Hkv) > HPC_MAX_QUERY_ROWS) return HPC_ERR_UNSUPPORTED;
    if (!d_part_o || !d_part_lse || (B > 0 && !d_out)) return HPC_ERR_ARG;
    if (!aligned16(d_part_o) || !aligned16(d_out)) return HPC_ERR_ARG;
    st = check_map(map, true);
    if (st != HPC_OK) return st;
    if (map->B != B || map->Hkv != Hkv || (int64_t)B * Hkv > map->cap_units) return HPC_ERR_ARG;
    return cuda_status(launch_combine(d_part_o, d_part_lse, *map, B, Hq, Hkv, q_len, d_out,
                                      static_cast<cudaStream_t>(stream)));
}

// The packed per-step inputs, from pinned host memory read through its device
// alias into the device buffer: one 16-byte load per thread, so the transfer
// is a single round trip over the CPU-GPU link.  It lets the grid after it
// (the assign kernel, a programmatic dependent that reads nothing before
// griddepcontrol.wait) launch at once instead of behind a copy-engine
// transfer.  Launched as an ordinary kernel: the previous step's grids may
// still read the device buffer until they end.
constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy_in_kernel(const int4 *__restrict__ src,
                                                               int4 *__restrict__ dst, int64_t n) {
    grid_launch_dependents();
    for (int64_t i = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * kCopyThreads)
        dst[i] = src[i];
}

// Up to four host arrays copied by one launch (grid row y = array y), each
// as 16-byte vectors when both ends are 16-byte aligned, else byte by byte.
struct CopySegments {
    const char *src[4];
    char *dst[4];
    int64_t bytes[4];
};

__global__ void __launch_bounds__(kCopyThreads) copy_in_segments_kernel(const CopySegments c) {
    grid_launch_dependents();
    const int y = blockIdx.y;  // selected without indexing the parameter block
    const char *src = y == 0 ? c.src[0] : y == 1 ? c.src[1] : y == 2 ? c.src[2] : c.src[3];
    char *dst = y == 0 ? c.dst[0] : y == 1 ? c.dst[1] : y == 2 ? c.dst[2] : c.dst[3];
    const int64_t bytes = y == 0 ? c.bytes[0] : y == 1 ? c.bytes[1] : y == 2 ? c.bytes[2] : c.bytes[3];
    const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
    const int64_t first = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x;
    const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0;
    int64_t done = 0;
    if (vec) {
        const int64_t n = bytes / 16;
        for (int64_t i = first; i < n; i += stride)
            reinterpret_cast<int4 *>(dst)[i] = reinterpret_cast<const int4 *>(src)[i];
        done = n * 16;
    }
    for (int64_t i = done + first; i < bytes; i += stride) dst[i] = src[i];
}

// The device alias of a pinned (page-locked, mapped) host buffer, or null for
// pageable memory.
const void *host_alias(const void *h) {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, h) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return pa.type == cudaMemoryTypeHost ? pa.devicePointer : nullptr;
}

}  // namespace

namespace hpc {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return encoder(); }
hpc_status cache_tensor_map(CUtensorMap *m, const void *base, int32_t num_pages, int32_t Hkv,
                            bool fp8) {
    return make_cache_map(m, base, num_pages, Hkv, fp8);
}
}  // namespace hpc

extern "C" {

const char *hpc_decode_version(void) { return "hpc_decode 0.1 (sm_103a)"; }

const char *hpc_status_string(hpc_status s) {
    switch (s) {
        case HPC_OK: return "ok";
        case HPC_ERR_ARG: return "invalid argument";
        case HPC_ERR_UNSUPPORTED: return "unsupported shape";
        case HPC_ERR_WORKSPACE: return "workspace too small";
        case HPC_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

int64_t hpc_decode_desc_capacity(int32_t B, int32_t Hkv, int32_t num_ctas) {
    if (B < 0 || Hkv < 0 || num_ctas < 0) return -1;
    return (int64_t)num_ctas + (int64_t)B * Hkv;
}

int64_t hpc_decode_static_capacity(int32_t B, int32_t Hkv, int32_t num_splits) {
    if (B < 0 || Hkv < 0 || num_splits < 0) return -1;
    return (int64_t)B * Hkv * num_splits;
}

int32_t hpc_decode_num_ctas(int32_t device, hpc_kv_dtype kv_dtype) {
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_ARG;
    int prev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return HPC_ERR_CUDA;
    if (device != prev && cudaSetDevice(device) != cudaSuccess) return HPC_ERR_CUDA;
    const AttnConfig &cfg = config_for(kv_dtype);
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = prepare_kernel(cfg, kv_dtype == HPC_KV_FP8_E4M3 ? 1 : 0);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cfg.kernel, cfg.threads,
                                                          cfg.smem_bytes);
    if (device != prev) cudaSetDevice(prev);
    if (e != cudaSuccess || per_sm < 1) return HPC_ERR_CUDA;
    return sms * per_sm;
}

namespace {
// The load-balanced plan; bt_prefetch (the step's block table, or null) is
// warmed in L2 by the assign kernel for the attention grid that follows.
hpc_status plan_impl(const int32_t *d_seqlens, int32_t B, int32_t Hkv, int32_t max_pages_per_req,
                     int32_t num_ctas, int32_t min_tiles_per_cta, hpc_task_map *map,
                     hpc_stream_t stream, const int32_t *bt_prefetch) {
    if (B < 0 || Hkv <= 0 || max_pages_per_req <= 0 || num_ctas < 1 || min_tiles_per_cta < 0)
        return HPC_ERR_ARG;
    if (min_tiles_per_cta >= (1 << 29)) return HPC_ERR_ARG;
    if (B > 0 && !d_seqlens) return HPC_ERR_ARG;
    if (B > HPC_MAX_BATCH) return HPC_ERR_UNSUPPORTED;
    if ((int64_t)B * max_pages_per_req * Hkv >= (int64_t)1 << 30) return HPC_ERR_UNSUPPORTED;
    hpc_status st = check_map(map, true);
    if (st != HPC_OK) return st;
    if ((int64_t)num_ctas + 1 > map->cap_bins || (int64_t)B * Hkv > map->cap_units ||
        (int64_t)map->cap_desc < hpc_decode_desc_capacity(B, Hkv, num_ctas))
        return HPC_ERR_WORKSPACE;
    hpc_task_map m = *map;
    m.B = B;
    m.Hkv = Hkv;
    m.num_ctas = num_ctas;
    m.persistent = 1;
    m.min_tiles = min_tiles_per_cta;
    m.max_pages = max_pages_per_req;
    st = cuda_status(launch_assign(d_seqlens, B, Hkv, max_pages_per_req, num_ctas,
                                   min_tiles_per_cta, m, static_cast<cudaStream_t>(stream),
                                   bt_prefetch));
    if (st == HPC_OK) *map = m;
    return st;
}
}  // namespace

hpc_status hpc_decode_plan(const int32_t *d_seqlens, int32_t B, int32_t Hkv,
                           int32_t max_pages_per_req, int32_t num_ctas,
                           int32_t min_tiles_per_cta, hpc_task_map *map, hpc_stream_t stream) {
    return plan_impl(d_seqlens, B, Hkv, max_pages_per_req, num_ctas, min_tiles_per_cta, map,
                     stream, nullptr);
}

hpc_status hpc_decode_plan_static(const int32_t *d_seqlens, int32_t B, int32_t Hkv,
                                  int32_t max_pages_per_req, int32_t num_splits,
                                  hpc_task_map *map, hpc_stream_t stream) {
    if (B < 0 || Hkv <= 0 || max_pages_per_req <= 0 || num_splits < 1) return HPC_ERR_ARG;
    if (B > 0 && !d_seqlens) return HPC_ERR_ARG;
    if (B > HPC_MAX_BATCH) return HPC_ERR_UNSUPPORTED;
    if ((int64_t)B * max_pages_per_req * Hkv >= (int64_t)1 << 30) return HPC_ERR_UNSUPPORTED;
    hpc_status st = check_map(map, true);
    if (st != HPC_OK) return st;
    const int64_t bins = hpc_decode_static_capacity(B, Hkv, num_splits);
    if (bins >= ((int64_t)1 << 31) - 1) return HPC_ERR_UNSUPPORTED;
    if (bins > map->cap_desc || bins + 1 > map->cap_bins || (int64_t)B * Hkv > map->cap_units)
        return HPC_ERR_WORKSPACE;
    if (bins == 0) return HPC_ERR_ARG;  // a grid needs at least one CTA
    hpc_task_map m = *map;
    m.B = B;
    m.Hkv = Hkv;
    m.num_ctas = (int32_t)bins;
    m.persistent = 0;
    m.min_tiles = num_splits;
    m.max_pages = max_pages_per_req;
    st = cuda_status(launch_static_plan(d_seqlens, B, Hkv, max_pages_per_req, num_splits, m,
                                        static_cast<cudaStream_t>(stream)));
    if (st == HPC_OK) *map = m;
    return st;
}

hpc_status hpc_decode_attn_mq(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                              const void *d_v_cache, int32_t num_pages, float k_scale,
                              float v_scale, hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                              int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                              int32_t Hq, int32_t Hkv, int32_t head_dim, int32_t q_len,
                              float sm_scale, const hpc_task_map *map, float *d_part_o,
                              float *d_part_lse, hpc_stream_t stream) {
    return launch_attention(d_q, d_q_scale, d_k_cache, d_v_cache, num_pages, k_scale, v_scale,
                            kv_dtype, d_block_table, max_pages_per_req, d_seqlens, B, Hq, Hkv,
                            head_dim, sm_scale, map, d_part_o, d_part_lse, nullptr, nullptr,
                            false, q_len, stream);
}

hpc_status hpc_decode_attn(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                           const void *d_v_cache, int32_t num_pages, float k_scale, float v_scale,
                           hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                           int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                           int32_t Hq, int32_t Hkv, int32_t head_dim, float sm_scale,
                           const hpc_task_map *map, float *d_part_o, float *d_part_lse,
                           hpc_stream_t stream) {
    return hpc_decode_attn_mq(d_q, d_q_scale, d_k_cache, d_v_cache, num_pages, k_scale, v_scale,
                              kv_dtype, d_block_table, max_pages_per_req, d_seqlens, B, Hq, Hkv,
                              head_dim, 1, sm_scale, map, d_part_o, d_part_lse, stream);
}

hpc_status hpc_decode_attn_combine_mq(const void *d_q, const float *d_q_scale,
                                      const void *d_k_cache, const void *d_v_cache,
                                      int32_t num_pages, float k_scale, float v_scale,
                                      hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                                      int32_t max_pages_per_req, const int32_t *d_seqlens,
                                      int32_t B, int32_t Hq, int32_t Hkv, int32_t head_dim,
                                      int32_t q_len, float sm_scale, const hpc_task_map *map,
                                      float *d_part_o, float *d_part_lse, int32_t *d_unit_done,
                                      void *d_out, hpc_stream_t stream) {
    return attn_combine(d_q, d_q_scale, d_k_cache, d_v_cache, num_pages, k_scale, v_scale,
                        kv_dtype, d_block_table, max_pages_per_req, d_seqlens, B, Hq, Hkv,
                        head_dim, sm_scale, map, d_part_o, d_part_lse, d_unit_done, d_out, false,
                        q_len, stream);
}

hpc_status hpc_decode_attn_combine(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                                   const void *d_v_cache, int32_t num_pages, float k_scale,
                                   float v_scale, hpc_kv_dtype kv_dtype,
                                   const int32_t *d_block_table, int32_t max_pages_per_req,
                                   const int32_t *d_seqlens, int32_t B, int32_t Hq, int32_t Hkv,
                                   int32_t head_dim, float sm_scale, const hpc_task_map *map,
                                   float *d_part_o, float *d_part_lse, int32_t *d_unit_done,
                                   void *d_out, hpc_stream_t stream) {
    return hpc_decode_attn_combine_mq(d_q, d_q_scale, d_k_cache, d_v_cache, num_pages, k_scale,
                                      v_scale, kv_dtype, d_block_table, max_pages_per_req,
                                      d_seqlens, B, Hq, Hkv, head_dim, 1, sm_scale, map, d_part_o,
                                      d_part_lse, d_unit_done, d_out, stream);
}

hpc_status hpc_decode_combine_mq(const float *d_part_o, const float *d_part_lse,
                                 const hpc_task_map *map, int32_t B, int32_t Hq, int32_t Hkv,
                                 int32_t head_dim, int32_t q_len, void *d_out,
                                 hpc_stream_t stream) {
    return combine_impl(d_part_o, d_part_lse, map, B, Hq, Hkv, head_dim, q_len, d_out, stream);
}

hpc_status hpc_decode_combine(const float *d_part_o, const float *d_part_lse,
                              const hpc_task_map *map, int32_t B, int32_t Hq, int32_t Hkv,
                              int32_t head_dim, void *d_out, hpc_stream_t stream) {
    return combine_impl(d_part_o, d_part_lse, map, B, Hq, Hkv, head_dim, 1, d_out, stream);
}

hpc_status hpc_decode_step_mq(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                              const void *d_v_cache, int32_t num_pages, float k_scale,
                              float v_scale, hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                              int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                              int32_t Hq, int32_t Hkv, int32_t head_dim, int32_t q_len,
                              float sm_scale, int32_t num_ctas, int32_t min_tiles_per_cta,
                              int32_t num_splits, hpc_task_map *map, float *d_part_o,
                              float *d_part_lse, int32_t *d_unit_done, void *d_out,
                              hpc_stream_t stream) {
    hpc_status st = check_shapes(B, Hq, Hkv, head_dim, max_pages_per_req);
    if (st != HPC_OK) return st;
    if (num_splits < 0 || q_len < 1) return HPC_ERR_ARG;
    if (q_len * (Hq / Hkv) > HPC_MAX_QUERY_ROWS) return HPC_ERR_UNSUPPORTED;
    st = num_splits == 0 ? plan_impl(d_seqlens, B, Hkv, max_pages_per_req, num_ctas,
                                     min_tiles_per_cta, map, stream, d_block_table)
                         : hpc_decode_plan_static(d_seqlens, B, Hkv, max_pages_per_req,
                                                  num_splits, map, stream);
    if (st != HPC_OK) return st;
    // the attention grid follows the assign kernel directly (after_plan)
    if (d_unit_done)  // fused: the attention grid also performs the combine
        return attn_combine(d_q, d_q_scale, d_k_cache, d_v_cache, num_pages, k_scale, v_scale,
                            kv_dtype, d_block_table, max_pages_per_req, d_seqlens, B, Hq, Hkv,
                            head_dim, sm_scale, map, d_part_o, d_part_lse, d_unit_done, d_out,
                            true, q_len, stream);
    st = launch_attention(d_q, d_q_scale, d_k_cache, d_v_cache, num_pages, k_scale, v_scale,
                          kv_dtype, d_block_table, max_pages_per_req, d_seqlens, B, Hq, Hkv,
                          head_dim, sm_scale, map, d_part_o, d_part_lse, nullptr, nullptr, true,
                          q_len, stream);
    if (st != HPC_OK) return st;
    return combine_impl(d_part_o, d_part_lse, map, B, Hq, Hkv, head_dim, q_len, d_out, stream);
}

hpc_status hpc_decode_step(const void *d_q, const float *d_q_scale, const void *d_k_cache,
                           const void *d_v_cache, int32_t num_pages, float k_scale, float v_scale,
                           hpc_kv_dtype kv_dtype, const int32_t *d_block_table,
                           int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
                           int32_t Hq, int32_t Hkv, int32_t head_dim, float sm_scale,
                           int32_t num_ctas, int32_t min_tiles_per_cta, int32_t num_splits,
                           hpc_task_map *map, float *d_part_o, float *d_part_lse,
                           int32_t *d_unit_done, void *d_out, hpc_stream_t stream) {
    return hpc_decode_step_mq(d_q, d_q_scale, d_k_cache, d_v_cache, num_pages, k_scale, v_scale,
                              kv_dtype, d_block_table, max_pages_per_req, d_seqlens, B, Hq, Hkv,
                              head_dim, 1, sm_scale, num_ctas, min_tiles_per_cta, num_splits,
                              map, d_part_o, d_part_lse, d_unit_done, d_out, stream);
}

hpc_status hpc_decode_step_host(const void *h_q, const float *h_q_scale, const int32_t *h_seqlens,
                                const int32_t *h_block_table, void *h_out, void *d_q,
                                float *d_q_scale, int32_t *d_seqlens, int32_t *d_block_table,
                                void *d_out, const void *d_k_cache, const void *d_v_cache,
                                int32_t num_pages, float k_scale, float v_scale,
                                hpc_kv_dtype kv_dtype, int32_t max_pages_per_req, int32_t B,
                                int32_t Hq, int32_t Hkv, int32_t head_dim, float sm_scale,
                                int32_t num_ctas, int32_t min_tiles_per_cta, int32_t num_splits,
                                hpc_task_map *map, float *d_part_o, float *d_part_lse,
                                int32_t *d_unit_done, hpc_stream_t stream) {
    hpc_status st = check_shapes(B, Hq, Hkv, head_dim, max_pages_per_req);
    if (st != HPC_OK) return st;
    const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
    if (B > 0 && (!h_q || !h_seqlens || !h_block_table || !h_out || !d_q || !d_seqlens ||
                  !d_block_table || !d_out))
        return HPC_ERR_ARG;
    if (fp8 && B > 0 && (!h_q_scale || !d_q_scale)) return HPC_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t q_bytes = (size_t)B * Hq * HPC_HEAD_DIM * (fp8 ? 1 : 2);
    const size_t out_bytes = (size_t)B * Hq * HPC_HEAD_DIM * 2;
    cudaError_t e = cudaSuccess;
    if (B > 0) {
        // all inputs pinned: one copy kernel reads them through their device
        // aliases (the assign kernel launches behind it as a programmatic
        // dependent); otherwise one copy-engine transfer per array
        const void *hs[4] = {h_q, fp8 ? h_q_scale : nullptr, h_seqlens, h_block_table};
        void *ds[4] = {d_q, fp8 ? d_q_scale : nullptr, d_seqlens, d_block_table};
        const int64_t nb[4] = {(int64_t)q_bytes, fp8 ? (int64_t)B * Hq * 4 : 0, (int64_t)B * 4,
                               (int64_t)B * max_pages_per_req * 4};
        CopySegments cs = {};
        int n = 0;
        int64_t widest = 0;
        bool pinned = true;
        for (int i = 0; i < 4 && pinned; ++i) {
            if (nb[i] == 0) continue;
            const void *a = host_alias(hs[i]);
            if (!a) pinned = false;
            cs.src[n] = static_cast<const char *>(a);
            cs.dst[n] = static_cast<char *>(ds[i]);
            cs.bytes[n] = nb[i];
            widest = std::max(widest, (nb[i] + 15) / 16);
            ++n;
        }
        if (pinned) {
            const int gx = (int)std::min<int64_t>((widest + kCopyThreads - 1) / kCopyThreads, 1024);
            copy_in_segments_kernel<<<dim3(gx, n), kCopyThreads, 0, s>>>(cs);
            e = cudaGetLastError();
        } else {
            for (int i = 0; i < 4 && e == cudaSuccess; ++i)
                if (nb[i] > 0)
                    e = cudaMemcpyAsync(ds[i], hs[i], (size_t)nb[i], cudaMemcpyHostToDevice, s);
        }
        if (e != cudaSuccess) return HPC_ERR_CUDA;
    }
    st = hpc_decode_step(d_q, d_q_scale, d_k_cache, d_v_cache, num_pages, k_scale, v_scale,
                         kv_dtype, d_block_table, max_pages_per_req, d_seqlens, B, Hq, Hkv,
                         head_dim, sm_scale, num_ctas, min_tiles_per_cta, num_splits, map,
                         d_part_o, d_part_lse, d_unit_done, d_out, stream);
    if (st != HPC_OK) return st;
    if (B > 0) e = cudaMemcpyAsync(h_out, d_out, out_bytes, cudaMemcpyDeviceToHost, s);
    return cuda_status(e);
}

int64_t hpc_decode_packed_layout(int32_t B, int32_t Hq, int32_t max_pages_per_req,
                                 hpc_kv_dtype kv_dtype, int64_t offsets[4]) {
    if (B < 0 || Hq <= 0 || max_pages_per_req <= 0 || !offsets) return -1;
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return -1;
    const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
    auto up16 = [](int64_t x) { return (x + 15) & ~int64_t(15); };
    int64_t off = 0;
    offsets[0] = off;
    off = up16(off + (int64_t)B * Hq * HPC_HEAD_DIM * (fp8 ? 1 : 2));
    offsets[1] = fp8 ? off : -1;
    if (fp8) off = up16(off + (int64_t)B * Hq * 4);
    offsets[2] = off;
    off = up16(off + (int64_t)B * 4);
    offsets[3] = off;
    off = up16(off + (int64_t)B * max_pages_per_req * 4);
    return off;
}

hpc_status hpc_decode_step_host_packed(const void *h_in, void *d_in, void *h_out, void *d_out,
                                       const void *d_k_cache, const void *d_v_cache,
                                       int32_t num_pages, float k_scale, float v_scale,
                                       hpc_kv_dtype kv_dtype, int32_t max_pages_per_req,
                                       int32_t B, int32_t Hq, int32_t Hkv, int32_t head_dim,
                                       float sm_scale, int32_t num_ctas,
                                       int32_t min_tiles_per_cta, int32_t num_splits,
                                       hpc_task_map *map, float *d_part_o, float *d_part_lse,
                                       int32_t *d_unit_done, hpc_stream_t stream) {
    hpc_status st = check_shapes(B, Hq, Hkv, head_dim, max_pages_per_req);
    if (st != HPC_OK) return st;
    int64_t off[4];
    const int64_t bytes = hpc_decode_packed_layout(B, Hq, max_pages_per_req, kv_dtype, off);
    if (bytes < 0) return HPC_ERR_ARG;
    if (B > 0 && (!h_in || !d_in || !h_out)) return HPC_ERR_ARG;
    if (B > 0 && !d_out && !d_unit_done) return HPC_ERR_ARG;  // direct output needs the fused combine
    if (B > 0 && !aligned16(d_in)) return HPC_ERR_ARG;
    // d_out null: the attention grid (combine fused) stores the output straight
    // into h_out through its device alias (pinned host memory under unified
    // addressing), with no separate copy
    void *out = d_out;
    const bool to_host = B > 0 && d_out == nullptr;
    if (to_host) {
        out = const_cast<void *>(host_alias(h_out));
        if (!out || !aligned16(out)) return HPC_ERR_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
    char *d = static_cast<char *>(d_in);
    if (B > 0) {
        // pinned input: copied by copy_in_kernel; pageable: by the copy engine
        const void *src = host_alias(h_in);
        if (src && aligned16(src)) {
            const int64_t n = bytes / 16;  // the layout's size is a multiple of 16
            const int grid = (int)std::min<int64_t>((n + kCopyThreads - 1) / kCopyThreads, 1024);
            copy_in_kernel<<<grid, kCopyThreads, 0, s>>>(static_cast<const int4 *>(src),
                                                          static_cast<int4 *>(d_in), n);
            if (cudaGetLastError() != cudaSuccess) return HPC_ERR_CUDA;
        } else if (cudaMemcpyAsync(d_in, h_in, (size_t)bytes, cudaMemcpyHostToDevice, s) !=
                   cudaSuccess) {
            return HPC_ERR_CUDA;
        }
    }
    st = hpc_decode_step(d + off[0], fp8 ? reinterpret_cast<const float *>(d + off[1]) : nullptr,
                         d_k_cache, d_v_cache, num_pages, k_scale, v_scale, kv_dtype,
                         reinterpret_cast<const int32_t *>(d + off[3]), max_pages_per_req,
                         reinterpret_cast<const int32_t *>(d + off[2]), B, Hq, Hkv, head_dim,
                         sm_scale, num_ctas, min_tiles_per_cta, num_splits, map, d_part_o,
                         d_part_lse, d_unit_done, out, stream);
    if (st != HPC_OK || B == 0 || to_host) return st;
    return cuda_status(cudaMemcpyAsync(h_out, d_out, (size_t)B * Hq * HPC_HEAD_DIM * 2,
                                       cudaMemcpyDeviceToHost, s));
}

hpc_status hpc_decode_read_meta(const hpc_task_map *map, int32_t host_meta[4],
                                hpc_stream_t stream) {
    if (!map || !map->meta || !host_meta) return HPC_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(host_meta, map->meta, 4 * sizeof(int32_t),
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

}  // extern "C"
