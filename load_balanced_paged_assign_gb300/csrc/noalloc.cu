// hpc_decode_step_noalloc: a whole decode step (assign, attention, combine)
// whose scratch — the task map and the split buffer of partial outputs —
// lives in a fixed array compiled into this library instead of memory the
// caller allocates.
//
// Who needs this: callers that cannot call cudaMalloc at the point where
// they run decode attention — for example code running under an allocator
// they do not control, plug-ins whose host framework forbids device
// allocation after start-up, or tools that must not perturb the memory state
// they observe.  Such a caller passes only its inputs and the output buffer.
//
// The array is HPC_NOALLOC_SCRATCH_BYTES (8 MiB) of device memory that every
// GPU using the library holds from load to process exit.  All calls on a
// device share it and it keeps the last call's contents, so two calls whose
// work overlaps on the GPU (different streams, or different host threads)
// race on it and corrupt each other; serialise them.  Nothing in it needs to
// start at zero: the assign kernel rewrites every part of the task map that
// the later kernels read, and every partial is written before it is read.
#include <mutex>

#include "internal.h"

namespace {

constexpr int64_t kScratchBytes = HPC_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// The array's device address is a property of the CUDA context the library's
// module is loaded in, not of the device ordinal: a cudaDeviceReset, or a
// caller that makes another context current (cuCtxSetCurrent), loads the
// module again at another address.  So the cached address is keyed by the
// context's unique id (cuCtxGetId, never reused within a process) and looked
// up again whenever the current context differs.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct ScratchEntry {
    unsigned long long ctx_id;  // context the address belongs to
    void *addr;                 // null: nothing cached
};

std::mutex g_mutex;
ScratchEntry g_cache[kMaxDevices];  // per device, guarded by g_mutex
std::once_flag g_fn_once;
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

// Unique id of the context current on this thread; false when there is none
// or the driver does not provide the calls (then nothing is cached).
bool current_context_id(unsigned long long *id) {
    std::call_once(g_fn_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
    });
    CUcontext ctx = nullptr;
    if (!g_ctx_current || !g_ctx_id || g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Device address of the array in the current context.  Looked up with
// cudaGetSymbolAddress the first time a context calls (with that context's
// device current); the symbol name itself is only a host stand-in and must
// never be handed to a kernel.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    std::lock_guard<std::mutex> lock(g_mutex);
    ScratchEntry &c = g_cache[dev];
    if (have_id && c.addr && c.ctx_id == id) {
        *out = c.addr;
        return cudaSuccess;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);  // makes the device's context current if none was
    if (e != cudaSuccess) return e;
    if (!have_id) have_id = current_context_id(&id);
    c = have_id ? ScratchEntry{id, p} : ScratchEntry{0, nullptr};
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" hpc_status hpc_decode_step_noalloc(
    const void *d_q, const float *d_q_scale, const void *d_k_cache, const void *d_v_cache,
    int32_t num_pages, float k_scale, float v_scale, hpc_kv_dtype kv_dtype,
    const int32_t *d_block_table, int32_t max_pages_per_req, const int32_t *d_seqlens, int32_t B,
    int32_t Hq, int32_t Hkv, int32_t head_dim, float sm_scale, int32_t num_ctas,
    int32_t min_tiles_per_cta, void *d_out, int32_t *d_meta_out, hpc_stream_t stream) {
    // The shape checks of hpc_decode_step, first, so that an unsupported shape
    // gets the same status there and here.
    if (B < 0 || Hq <= 0 || Hkv <= 0 || max_pages_per_req <= 0 || num_ctas < 1) return HPC_ERR_ARG;
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_ARG;
    if (head_dim != HPC_HEAD_DIM) return HPC_ERR_UNSUPPORTED;
    if (Hq % Hkv != 0 || Hq / Hkv > HPC_MAX_GROUP) return HPC_ERR_UNSUPPORTED;
    if (B > HPC_MAX_BATCH) return HPC_ERR_UNSUPPORTED;
    // Scratch layout: desc | bin_ptr | chunk_count | chunk_off | meta | part_o | part_lse,
    // sized in 64-bit arithmetic (no term can wrap: num_ctas < 2^31, B * Hkv < 2^31,
    // G <= 16) and checked against the array before anything is narrowed.
    const int64_t cap = hpc_decode_desc_capacity(B, Hkv, num_ctas);
    const int64_t units = (int64_t)B * Hkv > 0 ? (int64_t)B * Hkv : 1;
    const int64_t G = Hq / Hkv;
    const int64_t off_bins = align256(cap * 16);
    const int64_t off_count = off_bins + align256(((int64_t)num_ctas + 1) * 4);
    const int64_t off_off = off_count + align256(units * 4);
    const int64_t off_meta = off_off + align256(units * 4);
    const int64_t off_part_o = off_meta + 256;
    const int64_t off_part_lse = off_part_o + align256(cap * G * HPC_HEAD_DIM * 4);
    const int64_t need = off_part_lse + align256(cap * G * 4);
    if (cap < 0 || need > kScratchBytes) return HPC_ERR_WORKSPACE;  // too large for the array

    void *base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return HPC_ERR_CUDA;
    unsigned char *s = static_cast<unsigned char *>(base);
    hpc_task_map map;
    map.desc = reinterpret_cast<int32_t *>(s);
    map.bin_ptr = reinterpret_cast<int32_t *>(s + off_bins);
    map.chunk_count = reinterpret_cast<int32_t *>(s + off_count);
    map.chunk_off = reinterpret_cast<int32_t *>(s + off_off);
    map.meta = reinterpret_cast<int32_t *>(s + off_meta);
    map.cap_desc = (int32_t)cap;  // < 2^19: the layout fits the array
    map.cap_bins = num_ctas + 1;
    map.cap_units = (int32_t)units;
    map.B = map.Hkv = map.num_ctas = map.persistent = map.min_tiles = map.max_pages = 0;
    hpc_status st = hpc_decode_step(
        d_q, d_q_scale, d_k_cache, d_v_cache, num_pages, k_scale, v_scale, kv_dtype,
        d_block_table, max_pages_per_req, d_seqlens, B, Hq, Hkv, head_dim, sm_scale, num_ctas,
        min_tiles_per_cta, 0, &map, reinterpret_cast<float *>(s + off_part_o),
        reinterpret_cast<float *>(s + off_part_lse), nullptr, d_out, stream);
    if (st != HPC_OK || !d_meta_out) return st;
    return cudaMemcpyAsync(d_meta_out, map.meta, 4 * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HPC_OK
               : HPC_ERR_CUDA;
}
