// Assign step: builds the load-balanced task map on the device from the
// device-side sequence lengths (HPC-Ops vLLM post, "The solution: a per-step,
// load-balanced decode scheduler", Assign bullet; SGLang post, 围绕Live KV
// Work的调度).  Also the static fixed-split plan used as the in-house
// comparator (vLLM post, "The challenge: mixed-length decode in every batch").
//
// One CTA of 1024 threads.  Everything is integer arithmetic, so the map is
// deterministic and independent of thread timing.  Instead of walking tiles
// one by one, each unit u = h * B + r computes its chunk list in closed form
// from its first global tile index S_u: it touches bins S_u / budget ..
// (S_u + n_r - 1) / budget, one descriptor per bin.  A prefix sum over the
// units' chunk counts places the descriptors, and each bin's CSR offset is
// found by locating the unit that owns the bin's first tile.

#include "internal.h"
#include "ptx.cuh"

namespace hpc {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Inclusive block-wide prefix sum over blockDim.x (a multiple of 32) values;
// also returns the block total.  Uses `scratch` (32 ints) and synchronises.
__device__ int block_inclusive_scan(int v, int *scratch, int &total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += y;
    }
    if (lane == 31) scratch[wid] = v;
    __syncthreads();
    if (wid == 0) {
        int w = lane < nwarps ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        scratch[lane] = w;
    }
    __syncthreads();
    if (wid > 0) v += scratch[wid - 1];
    total = scratch[nwarps - 1];
    __syncthreads();
    return v;
}

__device__ __forceinline__ int tiles_of(int L) { return (L + kTile - 1) / kTile; }

// Reads seqlens[r], clamps it to [0, 64 * max_pages] and flags bad values.
__device__ __forceinline__ int live_len(const int32_t *seqlens, int r, int max_pages,
                                        unsigned &flags) {
    int L = seqlens[r];
    const int cap = max_pages * kTile;
    if (L < 0 || L > cap) {
        flags |= HPC_FLAG_BAD_SEQLEN;
        L = L < 0 ? 0 : cap;
    }
    return L;
}

constexpr size_t kPrefetchMaxBytes = 4u << 20;  // block-table bytes warmed in L2 at most

__global__ void __launch_bounds__(kPlanThreads)
    assign_kernel(const int32_t *__restrict__ seqlens, int B, int Hkv, int max_pages,
                  int num_ctas, int floor, int4 *__restrict__ desc, int32_t *__restrict__ bin_ptr,
                  int32_t *__restrict__ chunk_count, int32_t *__restrict__ chunk_off,
                  int32_t *__restrict__ meta, int cap_desc, const int32_t *bt_prefetch) {
    extern __shared__ int s_end[];  // [B] inclusive prefix of tiles per request
    __shared__ int s_scan[32];
    __shared__ unsigned s_flags;
    const int tid = threadIdx.x;
    grid_dependency_wait();    // launched as a dependent: the previous grid is done
    grid_launch_dependents();  // the attention grid may start its prologue now
    if (bt_prefetch) {
        // the step's block table into L2 (no registers held, nothing waited
        // for): the attention grid looks up the pages of its first tiles
        // while this kernel still runs
        const size_t bytes = min((size_t)B * max_pages * 4, kPrefetchMaxBytes);
        const char *bt = reinterpret_cast<const char *>(bt_prefetch);
        for (size_t off = (size_t)tid * 128; off < bytes; off += (size_t)blockDim.x * 128)
            prefetch_l2(bt + off);
    }
    if (tid == 0) s_flags = 0;
    unsigned flags = 0;

    // a1: tiles per request, n_r = ceil(L_r / 64), and their running sum.
    int carry = 0;
    for (int base = 0; base < B; base += blockDim.x) {
        const int r = base + tid;
        const int n = r < B ? tiles_of(live_len(seqlens, r, max_pages, flags)) : 0;
        int chunk_total;
        const int incl = block_inclusive_scan(n, s_scan, chunk_total);
        if (r < B) s_end[r] = carry + incl;
        carry += chunk_total;
    }
    __syncthreads();  // s_end complete
    const int N = carry;  // tiles per KV head; the host keeps Hkv * N < 2^30
    const int T = Hkv * N;

    // a2: budget = max(ceil(T / C), floor, 1).
    const int budget = max((T + num_ctas - 1) / num_ctas, max(floor, 1));

    // a3: chunk counts per unit (head-major, batch-minor), their offsets, the
    // descriptors, and the CSR offset of every used bin: bin b starts with
    // the descriptor that holds global tile b * budget.
    const int units = Hkv * B;
    carry = 0;
    for (int base = 0; base < units; base += blockDim.x) {
        const int u = base + tid;
        int cnt = 0, h = 0, r = 0, n = 0, S = 0;
        if (u < units) {
            h = u / B;
            r = u - h * B;
            n = s_end[r] - (r ? s_end[r - 1] : 0);
            S = h * N + s_end[r] - n;  // global index of the unit's first tile
            cnt = n ? (S + n - 1) / budget - S / budget + 1 : 0;
        }
        int chunk_total;
        const int incl = block_inclusive_scan(cnt, s_scan, chunk_total);
        if (u < units) {
            const int off = carry + incl - cnt;
            chunk_count[u] = cnt;
            chunk_off[u] = off;
            const int first_bin = S / budget;
            for (int i = 0; i < cnt; ++i) {
                const long long bin = first_bin + i;
                const long long bin_lo = bin * budget;
                const int lo = (int)max((long long)S, bin_lo);
                const int hi = (int)min((long long)(S + n), bin_lo + budget);
                if (off + i < cap_desc) {
                    desc[off + i] = make_int4(h, r, lo - S, hi - S);
                    if (lo == bin_lo) bin_ptr[bin] = off + i;  // first descriptor of its bin
                } else {
                    flags |= HPC_FLAG_DESC_OVERFLOW;
                }
            }
        }
        carry += chunk_total;
    }
    const int num_desc = carry;
    if (flags) atomicOr(&s_flags, flags);
    __syncthreads();
    const bool overflow = (s_flags & HPC_FLAG_DESC_OVERFLOW) != 0;
    // bins past the last tile are empty; an overflowing map is emptied entirely
    const int used = overflow ? 0 : (T + budget - 1) / budget;
    for (int b = used + tid; b <= num_ctas; b += blockDim.x) bin_ptr[b] = overflow ? 0 : num_desc;
    if (overflow)
        for (int b = tid; b < num_ctas; b += blockDim.x) bin_ptr[b] = 0;
    if (tid == 0) {
        meta[0] = T;
        meta[1] = budget;
        meta[2] = overflow ? 0 : num_desc;
        meta[3] = (int)s_flags;
        meta[4] = meta[5] = meta[6] = meta[7] = 0;  // bin counter of the attention kernel
    }
}

// Static split-KV plan: bin u * S + s is split s of unit u.
__global__ void __launch_bounds__(kPlanThreads)
    static_plan_kernel(const int32_t *__restrict__ seqlens, int B, int Hkv, int max_pages,
                       int S, int4 *__restrict__ desc, int32_t *__restrict__ bin_ptr,
                       int32_t *__restrict__ chunk_count, int32_t *__restrict__ chunk_off,
                       int32_t *__restrict__ meta) {
    __shared__ int s_scan[32];
    __shared__ unsigned s_flags;
    const int tid = threadIdx.x;
    grid_dependency_wait();
    grid_launch_dependents();
    if (tid == 0) s_flags = 0;
    unsigned flags = 0;
    int N = 0;
    for (int base = 0; base < B; base += blockDim.x) {
        const int r = base + tid;
        const int n = r < B ? tiles_of(live_len(seqlens, r, max_pages, flags)) : 0;
        int chunk_total;
        block_inclusive_scan(n, s_scan, chunk_total);
        N += chunk_total;
    }
    const int units = Hkv * B;
    const int bins = units * S;
    for (int b = tid; b < bins; b += blockDim.x) {
        const int u = b / S, s = b - u * S;
        const int h = u / B, r = u - h * B;
        unsigned ignored = 0;
        const int n = tiles_of(live_len(seqlens, r, max_pages, ignored));
        const int k = (n + S - 1) / S;
        desc[b] = make_int4(h, r, min(s * k, n), min((s + 1) * k, n));
        bin_ptr[b] = b;
        if (s == 0) {
            chunk_count[u] = k ? (n + k - 1) / k : 0;
            chunk_off[u] = u * S;
        }
    }
    if (flags) atomicOr(&s_flags, flags);
    __syncthreads();
    if (tid == 0) {
        bin_ptr[bins] = bins;
        meta[0] = Hkv * N;
        meta[1] = S;
        meta[2] = bins;
        meta[3] = (int)s_flags;
        meta[4] = meta[5] = meta[6] = meta[7] = 0;
    }
}

}  // namespace

int assign_smem_bytes(int B) { return (B > 0 ? B : 1) * (int)sizeof(int); }

// Smallest multiple of 32 threads covering the largest loop (capped at 1024):
// small batches are planned by a few warps, with cheaper barriers.
static int plan_threads(int B, int Hkv, int num_ctas) {
    const long long work = max((long long)B * Hkv, (long long)num_ctas + 1);
    const long long t = (work + 31) / 32 * 32;
    return (int)min(max(t, 64LL), (long long)kPlanThreads);
}

cudaError_t launch_assign(const int32_t *seqlens, int B, int Hkv, int max_pages, int num_ctas,
                          int floor, const hpc_task_map &map, cudaStream_t s,
                          const int32_t *bt_prefetch) {
    const int smem = assign_smem_bytes(B);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(assign_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(plan_threads(B, Hkv, num_ctas));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, assign_kernel, seqlens, B, Hkv, max_pages, num_ctas, floor,
                              reinterpret_cast<int4 *>(map.desc), map.bin_ptr, map.chunk_count,
                              map.chunk_off, map.meta, map.cap_desc, bt_prefetch);
}

cudaError_t launch_static_plan(const int32_t *seqlens, int B, int Hkv, int max_pages,
                               int num_splits, const hpc_task_map &map, cudaStream_t s) {
    static_plan_kernel<<<1, kPlanThreads, 0, s>>>(seqlens, B, Hkv, max_pages, num_splits,
                                                  reinterpret_cast<int4 *>(map.desc), map.bin_ptr,
                                                  map.chunk_count, map.chunk_off, map.meta);
    return cudaGetLastError();
}

}  // namespace hpc
