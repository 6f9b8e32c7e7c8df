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
//     tcgen05.ld (warp w reads TMEM lanes 32 (w mod 4) ..), and write
//     hi + lo / 256 (exact scaling) as FP32 scores, or as a split's partial;
//   * with split-K a second kernel sums the partials in split order, so the
//     result is deterministic.
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
constexpr int kSmemFloor = 120 * 1024;  // keeps one CTA per SM: TMEM is never contended

struct RouterArgs {
    float *out;       // [M, N] scores (splits == 1)
    float *partials;  // [splits, M, N] (splits > 1)
    int32_t *flags;   // optional error word
    int M, N, K;
    int bn;           // experts per CTA (multiple of 16, <= 256)
    int kb_per_split; // K blocks of 64 per split
    int splits;
    int stages;
    int lo_col;       // TMEM column of the W_low accumulator
    uint32_t tmem_cols;
};

__host__ __device__ inline int stage_bytes(int bn) { return kBM * kBK * 2 + 2 * bn * kBK * 2; }

__global__ void __launch_bounds__(kThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tx,
                       const __grid_constant__ CUtensorMap thi,
                       const __grid_constant__ CUtensorMap tlo, const RouterArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int sb = stage_bytes(a.bn);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.stages * sb);
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

    bool ok = true;
    int issued = 0;  // (producer lane) stages whose copies were issued
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t stream = policy_evict_first(), keep = policy_evict_last();
            for (int i = 0; i < nkb; ++i) {
                const int s = i % a.stages;
                if (!mbar_wait(&empty[s], ((i / a.stages) & 1u) ^ 1u, abort)) {
                    ok = false;
                    break;
                }
                uint8_t *st = smem + s * sb;
                const int k = (kb0 + i) * kBK;
                mbar_arrive_expect_tx(&full[s], (uint32_t)sb);
                tma_load_2d(st, &tx, &full[s], k, m0, stream);
                tma_load_2d(st + kBM * kBK * 2, &thi, &full[s], k, n0, keep);
                tma_load_2d(st + kBM * kBK * 2 + a.bn * kBK * 2, &tlo, &full[s], k, n0, keep);
                ++issued;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBM, a.bn);
            for (int i = 0; i < nkb; ++i) {
                const int s = i % a.stages;
                if (!mbar_wait(&full[s], (i / a.stages) & 1u, abort)) {
                    ok = false;
                    break;
                }
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
            // every MMA issued has completed (also after a timeout: TMEM is
            // only freed once this arrives)
            umma_commit(tmem_full);
        }
    } else {
        // epilogue: TMEM lane quarter q = warp mod 4 holds rows 32 q .. 32 q + 31
        const int q = warp & 3;
        int live = 1;
        if (lane == 0) live = mbar_wait(tmem_full, 0, abort) ? 1 : 0;
        live = __shfl_sync(0xffffffffu, live, 0);
        if (live) {
            mbar_try_wait(tmem_full, 0);  // every lane observes the completed phase
            tc_fence_after();
            const int m = m0 + 32 * q + lane;
            const uint32_t row = tmem + ((uint32_t)(32 * q) << 16);
            float *dst = a.splits == 1 ? a.out + (size_t)m * a.N
                                       : a.partials + ((size_t)split * a.M + m) * a.N;
            for (int c = 0; c < a.bn; c += 16) {
                float hi[16], lo[16];
                tmem_ld16x2(row + c, row + a.lo_col + c, hi, lo);
                if (m < a.M && n0 + c < a.N && !*abort) {
                    float4 *d4 = reinterpret_cast<float4 *>(dst + n0 + c);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        d4[j] = make_float4(hi[4 * j] + lo[4 * j] * (1.0f / 256.0f),
                                            hi[4 * j + 1] + lo[4 * j + 1] * (1.0f / 256.0f),
                                            hi[4 * j + 2] + lo[4 * j + 2] * (1.0f / 256.0f),
                                            hi[4 * j + 3] + lo[4 * j + 3] * (1.0f / 256.0f));
                }
            }
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
        if (lane == 0) {
            volatile int no_abort = 0;
            mbar_wait(tmem_full, 0, &no_abort);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// out[i] = sum over splits s of partials[s][i], in split order.
__global__ void router_reduce_kernel(const float4 *__restrict__ partials, float4 *__restrict__ out,
                                     size_t n4, int splits) {
    grid_dependency_wait();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        float4 acc = partials[i];
        for (int s = 1; s < splits; ++s) {
            const float4 v = partials[(size_t)s * n4 + i];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        out[i] = acc;
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
    int bn, n_tiles, m_tiles, splits, kb_per_split, stages, smem;
};

Plan plan_for(int M, int N, int K, int sms) {
    Plan p;
    p.n_tiles = (N + kMaxBN - 1) / kMaxBN;
    p.bn = ((N / p.n_tiles + 15) / 16) * 16;
    p.m_tiles = (M + kBM - 1) / kBM;
    const int kbs = K / kBK;
    // split K when the tiles alone would leave SMs idle; every split keeps
    // at least one K block and the splits divide the K blocks evenly
    int want = std::max(1, sms / std::max(1, p.m_tiles * p.n_tiles));
    want = std::min(want, kbs);
    while (kbs % want) --want;
    p.splits = want;
    p.kb_per_split = kbs / want;
    const int sb = stage_bytes(p.bn);
    p.stages = std::min(kMaxStages, std::max(2, (200 * 1024) / sb));
    p.stages = std::min(p.stages, std::max(1, p.kb_per_split));
    p.stages = std::max(p.stages, 1);
    p.smem = std::max(kSmemFloor, p.stages * sb + 2 * kMaxStages * 8 + 8 + 16 + 1024);
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
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    const Plan p = plan_for(M, N, K, sm_count(dev));
    return p.splits > 1 ? (int64_t)p.splits * M * N * 4 : 0;
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
            p.stages = std::min(kMaxStages, std::max(2, (200 * 1024) / stage_bytes(p.bn)));
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
    RouterArgs a;
    a.out = d_out;
    a.partials = static_cast<float *>(d_workspace);
    a.flags = d_flags;
    a.M = M;
    a.N = N;
    a.K = K;
    a.bn = p.bn;
    a.kb_per_split = p.kb_per_split;
    a.splits = p.splits;
    a.stages = p.stages;
    a.lo_col = ((p.bn + 31) / 32) * 32;
    a.tmem_cols = 32;
    while (a.tmem_cols < (uint32_t)(a.lo_col + p.bn)) a.tmem_cols <<= 1;
    p.smem = std::max(kSmemFloor, a.stages * stage_bytes(p.bn) + 2 * kMaxStages * 8 + 8 + 16 +
                                      1024);
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, router_gemm_kernel, tx, thi, tlo, a);
    if (e == cudaSuccess && p.splits > 1) {
        const size_t n4 = (size_t)M * N / 4;
        cudaLaunchConfig_t rc = {};
        rc.gridDim = dim3((unsigned)std::min<size_t>((n4 + 255) / 256, 4096));
        rc.blockDim = dim3(256);
        rc.stream = s;
        rc.attrs = attr;
        rc.numAttrs = 1;
        e = cudaLaunchKernelEx(&rc, router_reduce_kernel,
                               reinterpret_cast<const float4 *>(d_workspace),
                               reinterpret_cast<float4 *>(d_out), n4, p.splits);
    }
    return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}
