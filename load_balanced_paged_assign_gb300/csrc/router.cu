// Router GEMM with FP32 weights on BF16 tensor cores: the hi/lo split of the
// SGLang post's router-GEMM section ("Router GEMM：在路由精度与吞吐量之间取得平衡").
// Each FP32 weight is split once into W_high (its BF16 truncation) and W_low
// (the BF16 of the residual times 256); one kernel then computes
// S = X W_high^T + (X W_low^T) / 256 for BF16 hidden states X, loading every
// activation tile once for both products and accumulating both in FP32.
//
// GB300 design (tcgen05 + TMEM + TMA):
//   * a CTA owns a 128-row block of X (tokens) and up to 256 experts; its K
//     range is the whole hidden size or, when the grid would leave SMs idle
//     (few tokens), one of S equal slices (split-K);
//   * warp 0 streams 64-wide K blocks of X, W_high and W_low into a ring of
//     shared-memory stages with 2-D TMA loads (128-byte swizzle, K-major);
//   * one thread of warp 1 issues tcgen05.mma (kind::f16, BF16 in, FP32
//     accumulate) per 16-wide K step, twice: into the W_high accumulator and
//     into the W_low accumulator, both in TMEM (hi at column 0, lo after it);
//     tcgen05.commit releases each stage when its MMAs are done;
//   * warps 2-5 wait for the last commit, read both accumulators with
//     tcgen05.ld (warp w reads TMEM lanes 32 (w mod 4) ..), form
//     hi + lo / 256 (exact scaling), stage it in the freed ring (32-column
//     chunks, 128-byte swizzle) and write each chunk with a TMA tensor store,
//     as FP32 scores or as a split's partial (rows past M and columns past N
//     fall outside the tensor map and are not written);
//   * with split-K a second kernel sums the partials in a fixed order, so the
//     result is deterministic;
//   * up to 16 tokens the product is a weight-bound matrix-vector product:
//     a CUDA-core kernel reads the split weights once with no split-K pass.
// Every mbarrier wait is bounded; on a timeout the CTA raises the error
// flag, waits (bounded) for its copies in flight, frees its TMEM and leaves.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"
#include "tcgen05.cuh"

namespace hpc {
namespace {

constexpr int kBM = 128;        // tokens per CTA (UMMA M)
constexpr int kBK = 64;         // K per stage (one 128-byte swizzle row of BF16)
constexpr int kUK = 16;         // K per MMA instruction (kind::f16)
constexpr int kMaxBN = 256;     // experts per CTA (UMMA N limit at M = 128)
constexpr int kThreads = 192;   // producer, MMA, 4 epilogue warps
constexpr int kMaxStages = 4;
constexpr int kRingBytes = 200 * 1024;  // shared memory given to the stages at most
constexpr int kSmemFloor = 120 * 1024;  // keeps one CTA per SM: TMEM is never contended

struct RouterArgs {
    int32_t *flags;   // optional error word
    int M, N, K;
    int bn;           // experts per CTA (multiple of 32, <= 256)
    int kb_per_split; // K blocks per split
    int splits;
    int stages;
    int bar_off;      // shared-memory offset of the barriers (after the ring and the staging tile)
    int lo_col;       // TMEM column of the W_low accumulator
    uint32_t tmem_cols;
};

__host__ __device__ inline int stage_bytes(int bn) { return kBM * kBK * 2 + 2 * bn * kBK * 2; }

__global__ void __launch_bounds__(kThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tx,
                       const __grid_constant__ CUtensorMap thi,
                       const __grid_constant__ CUtensorMap tlo,
                       const __grid_constant__ CUtensorMap tout, const RouterArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int sb = stage_bytes(a.bn);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.bar_off);
    uint64_t *empty = full + kMaxStages;
    uint64_t *tmem_full = empty + kMaxStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tmem_full + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * a.bn, split = blockIdx.z;
    const int kb0 = split * a.kb_per_split, nkb = a.kb_per_split;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tmem_full, 1);
        *abort = 0;
        fence_barrier_init();
        prefetch_tensormap(&tx);
        prefetch_tensormap(&thi);
        prefetch_tensormap(&tlo);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dependency_wait();  // X may come from the kernel before this one
    // with split-K the reduction kernel follows: let it be scheduled now (it
    // waits for this grid's completion before reading the partials), so its
    // launch latency overlaps this kernel
    if (a.splits > 1) grid_launch_dependents();

    bool ok = true;
    int issued = 0;  // (producer lane) stages whose copies were issued
    // The producer and MMA roles: the whole warp takes every (bounded) wait
    // and lane 0 issues, so no lane is parked at a warp barrier while
    // another polls (parked lanes slow the SM's other warps).
    if (warp == 0) {
        const uint64_t stream = policy_evict_first(), keep = policy_evict_last();
        for (int i = 0; i < nkb; ++i) {
            const int s = i % a.stages;
            if (!mbar_wait_warp(&empty[s], ((i / a.stages) & 1u) ^ 1u, abort)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                uint8_t *st = smem + s * sb;
                const int k = (kb0 + i) * kBK;
                mbar_arrive_expect_tx(&full[s], (uint32_t)sb);
                tma_load_2d(st, &tx, &full[s], k, m0, stream);
                tma_load_2d(st + kBM * kBK * 2, &thi, &full[s], k, n0, keep);
                tma_load_2d(st + kBM * kBK * 2 + a.bn * kBK * 2, &tlo, &full[s], k, n0, keep);
            }
            __syncwarp();
            ++issued;
        }
    } else if (warp == 1) {
        const uint32_t idesc = idesc_bf16_f32(kBM, a.bn);
        for (int i = 0; i < nkb; ++i) {
            const int s = i % a.stages;
            if (!mbar_wait_warp(&full[s], (i / a.stages) & 1u, abort)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + s * sb);
                const uint32_t sh = sa + kBM * kBK * 2, sl = sh + a.bn * kBK * 2;
#pragma unroll
                for (int k = 0; k < kBK / kUK; ++k) {
                    const uint64_t da = smem_desc_k128(sa + k * kUK * 2);
                    const bool acc = (i | k) != 0;
                    umma_bf16(tmem, da, smem_desc_k128(sh + k * kUK * 2), idesc, acc);
                    umma_bf16(tmem + a.lo_col, da, smem_desc_k128(sl + k * kUK * 2), idesc, acc);
                }
                umma_commit(&empty[s]);  // the stage is free once these MMAs have read it
            }
            __syncwarp();
        }
        // every MMA issued has completed (also after a timeout: TMEM is
        // only freed once this arrives)
        if (lane == 0) umma_commit(tmem_full);
    } else {
        // epilogue: TMEM lane quarter q = warp mod 4 holds rows 32 q .. 32 q + 31.
        // The ring is free once the last commit has arrived; each warp stages
        // its 32 rows there as 32-column chunks (128-byte rows, 128-byte
        // swizzle: a warp's 16-byte writes fill whole bank rows) and stores
        // each chunk with one TMA tensor store.  Rows past M and columns past
        // N fall outside the tensor map and are not written.
        const int q = warp & 3;
        // (after an abort, copies may still land in the ring: nothing is staged)
        // every lane waits; the verdict is warp-uniform (the TMEM loads below are
        // warp-collective)
        const bool waited = mbar_wait_warp(tmem_full, 0, abort);
        const bool live = __all_sync(0xffffffffu, waited && !*abort);
        if (live) {
            tc_fence_after();
            const uint32_t row = tmem + ((uint32_t)(32 * q) << 16);
            const int chunks = a.bn / 32;
            uint8_t *stage_out = smem + (size_t)q * chunks * 4096;
            for (int c = 0; c < chunks; ++c) {
                float v[64];
                tmem_ld32x2(row + 32 * c, row + a.lo_col + 32 * c, v);
                uint8_t *line = stage_out + c * 4096 + lane * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4 *>(line + ((j ^ (lane & 7)) << 4)) =
                        make_float4(v[4 * j] + v[32 + 4 * j] * (1.0f / 256.0f),
                                    v[4 * j + 1] + v[32 + 4 * j + 1] * (1.0f / 256.0f),
                                    v[4 * j + 2] + v[32 + 4 * j + 2] * (1.0f / 256.0f),
                                    v[4 * j + 3] + v[32 + 4 * j + 3] * (1.0f / 256.0f));
                fence_proxy_async_smem();  // the writes are seen by the TMA store
                __syncwarp();
                if (lane == 0 && !*abort) {
                    tma_store_3d(&tout, stage_out + c * 4096, n0 + 32 * c, m0 + 32 * q, split);
                    bulk_commit_group();
                }
            }
            if (lane == 0) bulk_wait_all();  // the scores are written, the staging is free
            __syncwarp();
        } else {
            ok = false;
        }
    }

    if (!ok || *abort) {
        if (a.flags && lane == 0) atomicOr(a.flags, (int)HPC_FLAG_TIMEOUT);
        // no copy may land after the CTA has left: wait (bounded) for the last
        // copy issued into each stage
        if (warp == 0 && lane == 0) {
            for (int i = max(0, issued - a.stages); i < issued; ++i) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&full[i % a.stages], (i / a.stages) & 1u) &&
                       globaltimer_ns() - t0 < 1000000000ull) {
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // no MMA may still write TMEM when it is freed (bounded, like every wait)
        {
            volatile int no_abort = 0;
            mbar_wait(tmem_full, 0, &no_abort);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// out[i] = sum over at most 8 splits, in split order: one thread per float4,
// its loads all in flight together.
__global__ void __launch_bounds__(256)
    router_reduce_few_kernel(const float4 *__restrict__ partials, float4 *__restrict__ out,
                             size_t n4, int splits) {
    grid_dependency_wait();
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    float4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
        v[c] = c < splits ? __ldcg(partials + (size_t)c * n4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc = v[0];
#pragma unroll
    for (int c = 1; c < 8; ++c) acc = add4(acc, v[c]);
    out[i] = acc;
}

// out[i] = sum over splits s of partials[s][i] (more than 8).  A block takes 32 float4s;
// its eight warp-rows of threads g = 0..7 each sum the splits s = g mod 8
// (all their loads in flight together), and the eight sums are combined in
// the order g = 0..7 through shared memory, so the result does not depend on
// timing.
__global__ void __launch_bounds__(256)
    router_reduce_kernel(const float4 *__restrict__ partials, float4 *__restrict__ out,
                         size_t n4, int splits) {
    __shared__ float4 part[8][32];
    grid_dependency_wait();
    const int e = threadIdx.x & 31, g = threadIdx.x >> 5;
    const size_t i = (size_t)blockIdx.x * 32 + e;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < n4) {
        float4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int sp = g + 8 * c;
            v[c] = sp < splits ? __ldcg(partials + (size_t)sp * n4 + i)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int sp = g + 64; sp < splits; sp += 8) acc = add4(acc, __ldcg(partials + (size_t)sp * n4 + i));
#pragma unroll
        for (int c = 0; c < 8; ++c) acc = add4(acc, v[c]);
    }
    part[g][e] = acc;
    __syncthreads();
    if (g == 0 && i < n4) {
        float4 sum = part[0][e];
#pragma unroll
        for (int c = 1; c < 8; ++c) sum = add4(sum, part[c][e]);
        out[i] = sum;
    }
}

// Few tokens (M <= kGemvMaxM): the product is bound by reading the split
// weights (2 N K BF16), so CUDA cores do it with no split-K pass.  A CTA owns
// kGemvExperts experts over the whole K and one 256-thread group per eight
// tokens (the groups read the same weights, the second time from L1); in a
// group, warp w takes every eighth 256-wide K block and a lane 8 consecutive
// K.  Both products are accumulated separately in FP32 (as the method
// states) and reduced in a fixed order: lanes by shuffles, then warps 0..7
// through shared memory.
constexpr int kGemvMaxM = 16;
constexpr int kGemvExperts = 2;
constexpr int kGemvRows = 8;  // tokens per 256-thread group at most

__device__ __forceinline__ void bf16x8(uint4 v, float (&f)[8]) {
    f[0] = bf16lo_to_f32(v.x), f[1] = bf16hi_to_f32(v.x);
    f[2] = bf16lo_to_f32(v.y), f[3] = bf16hi_to_f32(v.y);
    f[4] = bf16lo_to_f32(v.z), f[5] = bf16hi_to_f32(v.z);
    f[6] = bf16lo_to_f32(v.w), f[7] = bf16hi_to_f32(v.w);
}

template <int MM>  // tokens per group (M <= MM * groups)
__global__ void __launch_bounds__(256 * (kGemvMaxM / kGemvRows))
    router_gemv_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ whi,
                       const uint4 *__restrict__ wlo, float *__restrict__ out, int M, int N,
                       int K) {
    __shared__ float red[kGemvMaxM / kGemvRows][8][MM][kGemvExperts][2];
    grid_dependency_wait();
    const int grp = threadIdx.x >> 8, tid = threadIdx.x & 255;
    const int warp = tid >> 5, lane = tid & 31;
    const int m0 = grp * MM;
    const int n0 = blockIdx.x * kGemvExperts;
    const int K8 = K / 8;  // 16-byte vectors per row
    float acc[MM][kGemvExperts][2];
#pragma unroll
    for (int m = 0; m < MM; ++m)
#pragma unroll
        for (int e = 0; e < kGemvExperts; ++e) acc[m][e][0] = acc[m][e][1] = 0.f;
    // U K vectors per step, all their loads issued before any use (U = 2 when
    // the registers allow: twice the bytes in flight per thread)
    constexpr int U = MM <= 4 ? 2 : 1;
    for (int v0 = warp * 32 + lane; v0 < K8; v0 += 256 * U) {
        uint4 wv[U][kGemvExperts][2], xp[U][MM];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 256 * u;
            const bool in = v < K8;
#pragma unroll
            for (int e = 0; e < kGemvExperts; ++e) {
                const int n = min(n0 + e, N - 1);
                wv[u][e][0] = in ? __ldg(whi + (size_t)n * K8 + v) : make_uint4(0u, 0u, 0u, 0u);
                wv[u][e][1] = in ? __ldg(wlo + (size_t)n * K8 + v) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int m = 0; m < MM; ++m)
                xp[u][m] = in && m0 + m < M ? __ldg(x + (size_t)(m0 + m) * K8 + v)
                                            : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float h[kGemvExperts][8], l[kGemvExperts][8];
#pragma unroll
            for (int e = 0; e < kGemvExperts; ++e) {
                bf16x8(wv[u][e][0], h[e]);
                bf16x8(wv[u][e][1], l[e]);
            }
#pragma unroll
            for (int m = 0; m < MM; ++m) {
                float xv[8];
                bf16x8(xp[u][m], xv);
#pragma unroll
                for (int e = 0; e < kGemvExperts; ++e)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        acc[m][e][0] = fmaf(xv[j], h[e][j], acc[m][e][0]);
                        acc[m][e][1] = fmaf(xv[j], l[e][j], acc[m][e][1]);
                    }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MM; ++m)
#pragma unroll
        for (int e = 0; e < kGemvExperts; ++e)
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                float t = acc[m][e][p];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (lane == 0) red[grp][warp][m][e][p] = t;
            }
    __syncthreads();
    if (tid < MM * kGemvExperts) {
        const int m = tid / kGemvExperts, e = tid - m * kGemvExperts;
        if (m0 + m < M && n0 + e < N) {
            float hi = 0.f, lo = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                hi += red[grp][w][m][e][0];
                lo += red[grp][w][m][e][1];
            }
            out[(size_t)(m0 + m) * N + n0 + e] = hi + lo * (1.0f / 256.0f);
        }
    }
}

__global__ void router_split_kernel(const float *__restrict__ w, size_t n,
                                    __nv_bfloat16 *__restrict__ hi,
                                    __nv_bfloat16 *__restrict__ lo) {
    grid_dependency_wait();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const uint32_t bits = __float_as_uint(w[i]) & 0xFFFF0000u;  // truncation
        const float h = __uint_as_float(bits);
        hi[i] = __ushort_as_bfloat16((unsigned short)(bits >> 16));
        lo[i] = __float2bfloat16_rn((w[i] - h) * 256.0f);  // residual and scaling exact
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

hpc_status cuda_status_of(cudaError_t e) { return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA; }

template <int MM>
cudaError_t launch_gemv_m(const void *x, const void *hi, const void *lo, float *out, int M, int N,
                          int K, cudaStream_t s) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + kGemvExperts - 1) / kGemvExperts);
    cfg.blockDim = dim3(256 * ((M + MM - 1) / MM));  // one group per MM tokens
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, router_gemv_kernel<MM>, static_cast<const uint4 *>(x),
                              static_cast<const uint4 *>(hi), static_cast<const uint4 *>(lo),
                              out, M, N, K);
}

cudaError_t launch_gemv(const void *x, const void *hi, const void *lo, float *out, int M, int N,
                        int K, cudaStream_t s) {
    if (M <= 1) return launch_gemv_m<1>(x, hi, lo, out, M, N, K, s);
    if (M <= 4) return launch_gemv_m<4>(x, hi, lo, out, M, N, K, s);
    return launch_gemv_m<kGemvRows>(x, hi, lo, out, M, N, K, s);  // 8 tokens per group
}

std::mutex g_mu;
int g_smem_set[64];  // dynamic shared memory already allowed, per device
int g_sms[64];

int sm_count(int dev) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (dev < 0 || dev >= 64) return 0;
    if (!g_sms[dev]) cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    return g_sms[dev];
}

struct Plan {
    int bn, n_tiles, m_tiles, splits, kb_per_split, stages, bar_off, smem;
};

// Ring depth and shared-memory layout for the plan's tile: the stages, then
// (overlapping them) the epilogue's staging tile of 128 x bn FP32 scores,
// then the barriers.
void size_ring(Plan &p) {
    const int sb = stage_bytes(p.bn);
    p.stages = std::min(kMaxStages, std::max(2, kRingBytes / sb));
    p.stages = std::max(1, std::min(p.stages, p.kb_per_split));
    p.bar_off = std::max(p.stages * sb, kBM * p.bn * 4);
    p.smem = std::max(kSmemFloor, p.bar_off + 2 * kMaxStages * 8 + 8 + 16 + 1024);
}

Plan plan_for(int M, int N, int K, int sms) {
    Plan p;
    p.n_tiles = (N + kMaxBN - 1) / kMaxBN;
    // experts per CTA: a multiple of 32 (whole 32-column store chunks); the
    // last tile's rows past N read as zeros and its columns past N are not stored
    p.bn = (((N + p.n_tiles - 1) / p.n_tiles + 31) / 32) * 32;
    p.m_tiles = (M + kBM - 1) / kBM;
    const int kbs = K / kBK;
    // split K when the tiles alone would leave SMs idle; every split keeps
    // at least one K block and the splits divide the K blocks evenly
    int want = std::max(1, sms / std::max(1, p.m_tiles * p.n_tiles));
    want = std::min(want, kbs);
    while (kbs % want) --want;
    p.splits = want;
    p.kb_per_split = kbs / want;
    size_ring(p);
    return p;
}

}  // namespace
}  // namespace hpc

using namespace hpc;

extern "C" hpc_status hpc_router_split(const float *d_w, int32_t N, int32_t K, void *d_w_hi,
                                       void *d_w_lo, hpc_stream_t stream) {
    if (N <= 0 || K <= 0 || !d_w || !d_w_hi || !d_w_lo) return HPC_ERR_ARG;
    const size_t n = (size_t)N * K;
    const int threads = 256;
    const int grid = (int)std::min<size_t>((n + threads - 1) / threads, 4096);
    router_split_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        d_w, n, static_cast<__nv_bfloat16 *>(d_w_hi), static_cast<__nv_bfloat16 *>(d_w_lo));
    return cudaGetLastError() == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}

extern "C" int64_t hpc_router_workspace_bytes(int32_t M, int32_t N, int32_t K) {
    if (M < 0 || N <= 0 || K <= 0 || K % kBK || N % 16 || M == 0) return M == 0 ? 0 : -1;
    if (M <= kGemvMaxM) return 0;  // the few-token path needs no partials
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    const Plan p = plan_for(M, N, K, sm_count(dev));
    return p.splits > 1 ? (int64_t)p.splits * M * N * 4 : 0;
}

extern "C" hpc_status hpc_router_plan(int32_t M, int32_t N, int32_t K, int32_t *plan) {
    if (!plan || M < 0 || N <= 0 || K <= 0) return HPC_ERR_ARG;
    if (K % kBK || N % 16) return HPC_ERR_UNSUPPORTED;
    plan[0] = plan[1] = plan[2] = plan[3] = 0;
    if (M == 0) return HPC_OK;
    if (M <= kGemvMaxM) {
        plan[3] = (N + kGemvExperts - 1) / kGemvExperts;
        return HPC_OK;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return HPC_ERR_CUDA;
    const Plan p = plan_for(M, N, K, sm_count(dev));
    plan[0] = 1;
    plan[1] = p.bn;
    plan[2] = p.splits;
    plan[3] = p.m_tiles * p.n_tiles * p.splits;
    return HPC_OK;
}

extern "C" hpc_status hpc_router_gemm(const void *d_x, const void *d_w_hi, const void *d_w_lo,
                                      int32_t M, int32_t N, int32_t K, float *d_out,
                                      void *d_workspace, int64_t workspace_bytes,
                                      int32_t *d_flags, hpc_stream_t stream) {
    if (M < 0 || N <= 0 || K <= 0) return HPC_ERR_ARG;
    if (K % kBK || N % 16) return HPC_ERR_UNSUPPORTED;
    if ((int64_t)M * K >= ((int64_t)1 << 31) || (int64_t)N * K >= ((int64_t)1 << 31))
        return HPC_ERR_UNSUPPORTED;
    if (M == 0) return HPC_OK;
    if (!d_x || !d_w_hi || !d_w_lo || !d_out) return HPC_ERR_ARG;
    if (!aligned16(d_x) || !aligned16(d_w_hi) || !aligned16(d_w_lo) || !aligned16(d_out))
        return HPC_ERR_ARG;
    if (M <= kGemvMaxM) return cuda_status_of(launch_gemv(d_x, d_w_hi, d_w_lo, d_out, M, N, K,
                                                          static_cast<cudaStream_t>(stream)));
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return HPC_ERR_CUDA;
    Plan p = plan_for(M, N, K, sm_count(dev));
    if (p.splits > 1) {
        const int64_t need = (int64_t)p.splits * M * N * 4;
        if (!d_workspace || workspace_bytes < need || !aligned16(d_workspace)) {
            // not enough room for the partials: fewer splits
            const int64_t per = (int64_t)M * N * 4;
            int fit = d_workspace && aligned16(d_workspace) ? (int)(workspace_bytes / per) : 1;
            const int kbs = K / kBK;
            fit = std::max(1, std::min(fit, p.splits));
            while (kbs % fit) --fit;
            p.splits = fit;
            p.kb_per_split = kbs / fit;
            size_ring(p);
        }
    }
    auto encode = tensor_map_encoder();
    if (!encode) return HPC_ERR_CUDA;
    CUtensorMap tx, thi, tlo;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
        const cuuint32_t es[2] = {1, 1};
        if (encode(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(d_x), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return HPC_ERR_CUDA;
    }
    for (int w = 0; w < 2; ++w) {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)p.bn};
        const cuuint32_t es[2] = {1, 1};
        if (encode(w ? &tlo : &thi, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void *>(w ? d_w_lo : d_w_hi), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return HPC_ERR_CUDA;
    }
    // scores (one split) or the splits' partials, [splits, M, N] FP32, stored
    // in 32 x 32 tiles with the 128-byte swizzle of the staging chunks
    CUtensorMap tout;
    {
        void *base = p.splits > 1 ? d_workspace : static_cast<void *>(d_out);
        const cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)p.splits};
        const cuuint64_t strides[2] = {(cuuint64_t)N * 4, (cuuint64_t)M * N * 4};
        const cuuint32_t box[3] = {32, 32, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (encode(&tout, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return HPC_ERR_CUDA;
    }
    RouterArgs a;
    a.flags = d_flags;
    a.M = M;
    a.N = N;
    a.K = K;
    a.bn = p.bn;
    a.kb_per_split = p.kb_per_split;
    a.splits = p.splits;
    a.stages = p.stages;
    a.bar_off = p.bar_off;
    a.lo_col = p.bn;  // a multiple of 32
    a.tmem_cols = 32;
    while (a.tmem_cols < (uint32_t)(a.lo_col + p.bn)) a.tmem_cols <<= 1;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (p.smem > g_smem_set[dev]) {
            if (cudaFuncSetAttribute(router_gemm_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     p.smem) != cudaSuccess)
                return HPC_ERR_CUDA;
            g_smem_set[dev] = p.smem;
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.m_tiles, p.n_tiles, p.splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, router_gemm_kernel, tx, thi, tlo, tout, a);
    if (e == cudaSuccess && p.splits > 1) {
        const size_t n4 = (size_t)M * N / 4;
        const bool few = p.splits <= 8;
        cudaLaunchConfig_t rc = {};
        rc.gridDim = dim3((unsigned)(few ? (n4 + 255) / 256 : (n4 + 31) / 32));
        rc.blockDim = dim3(256);
        rc.stream = s;
        rc.attrs = attr;
        rc.numAttrs = 1;
        e = cudaLaunchKernelEx(&rc, few ? router_reduce_few_kernel : router_reduce_kernel,
                               reinterpret_cast<const float4 *>(d_workspace),
                               reinterpret_cast<float4 *>(d_out), n4, p.splits);
    }
    return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}
