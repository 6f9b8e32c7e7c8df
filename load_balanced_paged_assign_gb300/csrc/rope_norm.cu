// Fused attention prologue (HpcRopeNorm): QK-Norm, RoPE, the paged KV-cache
// write and, for FP8, the per-(token, head) E4M3 query.
//
// The op is described in the vLLM integration post ("A fused attention
// prologue") and the SGLang post (the Hy3 FP8 prologue paragraph): from the
// fused QKV projection it normalises and rotates the query and key heads in
// the model's order, writes K and V straight into the paged cache, and emits
// the FP8 query with its scale for the attention kernel.
//
// It is a pure streaming op (about 2.5 KB in and 2 KB out per token at the
// TP8 Hy3 shape, 20 KB in per token at TP1), so the design is about keeping
// enough bytes in flight:
//   * persistent CTAs of 8 warps stride over tokens; a warp owns whole
//     128-dim head rows (4 dims per lane, 8-byte loads) and issues the loads
//     of up to 8 of its rows before it processes any;
//   * the 64 rotation angles of a token are computed once per CTA by two
//     warps while the loads are in flight: the frequency table base^(-2i/128)
//     is built once per CTA in fp64, the angle pos * freq is reduced modulo
//     2 pi in fp64 (a few double operations), and only the reduced angle, in
//     half turns, goes through fp32 sincospif, so positions in the hundreds
//     of thousands keep fp32 accuracy;
//   * the RMS and the FP8 amax are warp reductions, the rotation partner of
//     a dim is in the same lane (interleaved pairs) or 16 lanes away (halves);
//   * one __syncthreads per token (the angle table and the token's cache
//     slot are double-buffered in shared memory).
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace hpc {
namespace {

constexpr int kRnWarps = 8;
constexpr int kRnThreads = 32 * kRnWarps;
constexpr int kRowsInFlight = 8;  // head rows a warp loads before processing them
constexpr double kInvPi = 0.3183098861837907;

struct RopeNormArgs {
    const uint16_t *qkv;
    int64_t stride;  // elements between token rows
    const uint16_t *q_w;
    const uint16_t *k_w;
    const int32_t *positions;
    const int32_t *token_req;
    const int32_t *block_table;
    void *k_cache;
    void *v_cache;
    void *q_out;
    float *q_scale_out;
    int32_t *flags;
    double base;
    float eps;
    float k_scale;
    float v_scale;
    int N, Hq, Hkv, R;  // R = Hq + 2 Hkv head rows per token
    int B, max_pages, num_pages;
    int layout;
    int norm_first;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// E4M3 (round to nearest even, saturating) of four values -> 4 bytes, v[0] lowest.
__device__ __forceinline__ uint32_t to_e4m3x4(const float (&v)[4]) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v[1]), "f"(v[0]));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v[3]), "f"(v[2]));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ uint2 to_bf16x4(const float (&v)[4]) {
    return make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
}

// Rotates this lane's four dims in place; cs holds (cos, sin) per frequency.
__device__ __forceinline__ void rotate(float (&v)[4], const float2 *cs, int lane, int layout) {
    if (layout == HPC_ROPE_HALVES) {
        // dims 4*lane + k; pairs (i, i + 64): lanes 0-15 hold the first
        // elements, lanes 16-31 the second ones of the same frequencies
        const bool second = lane >= 16;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float other = __shfl_xor_sync(0xffffffffu, v[k], 16);
            const float2 c = cs[(4 * lane + k) & 63];
            v[k] = second ? fmaf(v[k], c.x, other * c.y) : fmaf(v[k], c.x, -other * c.y);
        }
    } else {
        // pairs (2i, 2i + 1): dims 4*lane.. hold frequencies 2*lane and 2*lane + 1
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float2 c = cs[2 * lane + k];
            const float a = v[2 * k], b = v[2 * k + 1];
            v[2 * k] = fmaf(a, c.x, -b * c.y);
            v[2 * k + 1] = fmaf(b, c.x, a * c.y);
        }
    }
}

__device__ __forceinline__ void unpack4(uint2 raw, float (&x)[4]) {
    x[0] = bf16lo_to_f32(raw.x);
    x[1] = bf16hi_to_f32(raw.x);
    x[2] = bf16lo_to_f32(raw.y);
    x[3] = bf16hi_to_f32(raw.y);
}

template <bool FP8>
__device__ __forceinline__ void process_row(const RopeNormArgs &a, int t, int j, uint2 raw,
                                            const float2 *cs, long long slot,
                                            const float (&wq)[4], const float (&wk)[4],
                                            int lane) {
    float x[4];
    unpack4(raw, x);
    constexpr int kElem = FP8 ? 1 : 2;
    if (j >= a.Hq + a.Hkv) {  // value head: straight into the cache
        if (slot < 0) return;
        const int h = j - a.Hq - a.Hkv;
        char *dst = static_cast<char *>(a.v_cache) +
                    ((slot * a.Hkv + h) * kHeadDim + 4 * lane) * kElem;
        if (FP8) {
            float y[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) y[k] = x[k] / a.v_scale;
            *reinterpret_cast<uint32_t *>(dst) = to_e4m3x4(y);
        } else {
            *reinterpret_cast<uint2 *>(dst) = raw;
        }
        return;
    }
    const bool is_q = j < a.Hq;
    float w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = is_q ? wq[k] : wk[k];
    // the rotation keeps the row's norm, so the RMS of x serves both orders
    const float ss = warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]);
    const float inv = 1.0f / sqrtf(ss * (1.0f / kHeadDim) + a.eps);
    float y[4];
    if (a.norm_first) {
#pragma unroll
        for (int k = 0; k < 4; ++k) y[k] = x[k] * inv * w[k];
        rotate(y, cs, lane, a.layout);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) y[k] = x[k];
        rotate(y, cs, lane, a.layout);
#pragma unroll
        for (int k = 0; k < 4; ++k) y[k] = y[k] * inv * w[k];
    }
    if (is_q) {
        const size_t row = (size_t)t * a.Hq + j;
        if (FP8) {
            const float amax =
                warp_max(fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3]))));
            const float scale = amax > 0.f ? amax / 448.0f : 1.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) y[k] = y[k] / scale;
            reinterpret_cast<uint32_t *>(a.q_out)[row * (kHeadDim / 4) + lane] = to_e4m3x4(y);
            if (lane == 0) a.q_scale_out[row] = scale;
        } else {
            reinterpret_cast<uint2 *>(a.q_out)[row * (kHeadDim / 4) + lane] = to_bf16x4(y);
        }
        return;
    }
    if (slot < 0) return;
    const int h = j - a.Hq;
    char *dst =
        static_cast<char *>(a.k_cache) + ((slot * a.Hkv + h) * kHeadDim + 4 * lane) * kElem;
    if (FP8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) y[k] = y[k] / a.k_scale;
        *reinterpret_cast<uint32_t *>(dst) = to_e4m3x4(y);
    } else {
        *reinterpret_cast<uint2 *>(dst) = to_bf16x4(y);
    }
}

template <bool FP8>
__global__ void __launch_bounds__(kRnThreads) rope_norm_kernel(const RopeNormArgs a) {
    __shared__ double s_freq[kHeadDim / 2];
    __shared__ float2 s_cs[2][kHeadDim / 2];
    __shared__ long long s_slot[2];  // token's (page * 64 + offset), or -1: no cache write
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // Everything this grid reads may come from the kernel before it.
    grid_dependency_wait();
    if (tid < kHeadDim / 2) s_freq[tid] = pow(a.base, -(double)(2 * tid) / kHeadDim);
    float wq[4], wk[4];
    {
        const uint2 rq = reinterpret_cast<const uint2 *>(a.q_w)[lane];
        const uint2 rk = reinterpret_cast<const uint2 *>(a.k_w)[lane];
        unpack4(rq, wq);
        unpack4(rk, wk);
    }
    __syncthreads();

    int it = 0;
    for (int t = blockIdx.x; t < a.N; t += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint2 *row0 = reinterpret_cast<const uint2 *>(a.qkv + (size_t)t * a.stride);
        uint2 raw[kRowsInFlight];
#pragma unroll
        for (int k = 0; k < kRowsInFlight; ++k) {
            const int j = warp + k * kRnWarps;
            if (j < a.R) raw[k] = __ldcs(row0 + (size_t)j * (kHeadDim / 4) + lane);
        }
        if (tid < kHeadDim / 2) {
            const int pos = a.positions[t];
            // the angle in half turns, reduced to [-1, 1] exactly in fp64
            const double turns = (double)pos * s_freq[tid] * kInvPi;
            const double r = fma(-2.0, rint(0.5 * turns), turns);
            float sn, c;
            sincospif((float)r, &sn, &c);
            s_cs[buf][tid] = make_float2(c, sn);
        } else if (tid == kHeadDim / 2) {
            const int pos = a.positions[t];
            const int req = a.token_req ? a.token_req[t] : t;
            long long slot = -1;
            if (req < 0 || req >= a.B || pos < 0 || pos >= a.max_pages * kTile) {
                if (a.flags) atomicOr(a.flags, (int)HPC_FLAG_BAD_SEQLEN);
            } else {
                const int page = a.block_table[(size_t)req * a.max_pages + pos / kTile];
                if (page < 0 || page >= a.num_pages) {
                    if (a.flags) atomicOr(a.flags, (int)HPC_FLAG_BAD_PAGE);
                } else {
                    slot = (long long)page * kTile + (pos % kTile);
                }
            }
            s_slot[buf] = slot;
        }
        __syncthreads();
        const float2 *cs = s_cs[buf];
        const long long slot = s_slot[buf];
        for (int base = warp;;) {
#pragma unroll
            for (int k = 0; k < kRowsInFlight; ++k) {
                const int j = base + k * kRnWarps;
                if (j < a.R) process_row<FP8>(a, t, j, raw[k], cs, slot, wq, wk, lane);
            }
            base += kRowsInFlight * kRnWarps;
            if (base >= a.R) break;
#pragma unroll
            for (int k = 0; k < kRowsInFlight; ++k) {
                const int j = base + k * kRnWarps;
                if (j < a.R) raw[k] = __ldcs(row0 + (size_t)j * (kHeadDim / 4) + lane);
            }
        }
    }
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_grid_cap[kMaxDevices][2];  // resident CTAs per device and dtype (0: unknown)

template <bool FP8>
int grid_cap() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) {
        const int c = g_grid_cap[dev][FP8].load();
        if (c > 0) return c;
    }
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rope_norm_kernel<FP8>, kRnThreads,
                                                      0) != cudaSuccess ||
        per_sm < 1)
        return 0;
    const int cap = sms * per_sm;
    if (dev >= 0 && dev < kMaxDevices) g_grid_cap[dev][FP8].store(cap);
    return cap;
}

template <bool FP8>
cudaError_t launch(const RopeNormArgs &a, cudaStream_t s) {
    const int cap = grid_cap<FP8>();
    if (cap < 1) return cudaErrorUnknown;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(a.N, cap));
    cfg.blockDim = dim3(kRnThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rope_norm_kernel<FP8>, a);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite_positive(float x) { return std::isfinite(x) && x > 0.f; }

}  // namespace
}  // namespace hpc

extern "C" hpc_status hpc_rope_norm(const void *d_qkv, int64_t qkv_row_stride,
                                    const void *d_q_norm_w, const void *d_k_norm_w,
                                    const int32_t *d_positions, const int32_t *d_token_req,
                                    int32_t num_tokens, int32_t Hq, int32_t Hkv,
                                    int32_t head_dim, const int32_t *d_block_table,
                                    int32_t max_pages_per_req, int32_t B, void *d_k_cache,
                                    void *d_v_cache, int32_t num_pages, hpc_kv_dtype kv_dtype,
                                    float k_scale, float v_scale, void *d_q_out,
                                    float *d_q_scale_out, int32_t *d_flags,
                                    const hpc_rope_norm_params *params, hpc_stream_t stream) {
    using namespace hpc;
    if (!params || num_tokens < 0 || Hq <= 0 || Hkv <= 0 || B < 0 || max_pages_per_req <= 0 ||
        num_pages <= 0)
        return HPC_ERR_ARG;
    if (head_dim != HPC_HEAD_DIM || Hq % Hkv != 0) return HPC_ERR_UNSUPPORTED;
    if (Hq + 2 * Hkv > 4096) return HPC_ERR_UNSUPPORTED;
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_ARG;
    const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
    if (!std::isfinite(params->eps) || params->eps < 0.f || !finite_positive(params->rope_base))
        return HPC_ERR_ARG;
    if (params->rope_layout != HPC_ROPE_HALVES && params->rope_layout != HPC_ROPE_INTERLEAVED)
        return HPC_ERR_ARG;
    if (params->norm_first != 0 && params->norm_first != 1) return HPC_ERR_ARG;
    if (fp8 && (!finite_positive(k_scale) || !finite_positive(v_scale))) return HPC_ERR_ARG;
    if ((int64_t)B * max_pages_per_req >= (int64_t)1 << 31) return HPC_ERR_UNSUPPORTED;
    if ((int64_t)max_pages_per_req * kTile >= (int64_t)1 << 31) return HPC_ERR_UNSUPPORTED;
    if (num_tokens == 0) return HPC_OK;
    if (!d_qkv || !d_q_norm_w || !d_k_norm_w || !d_positions || !d_block_table || !d_k_cache ||
        !d_v_cache || !d_q_out || (fp8 && !d_q_scale_out))
        return HPC_ERR_ARG;
    if (qkv_row_stride < (int64_t)(Hq + 2 * Hkv) * HPC_HEAD_DIM || qkv_row_stride % 8 != 0)
        return HPC_ERR_ARG;
    if (!aligned16(d_qkv) || !aligned16(d_q_norm_w) || !aligned16(d_k_norm_w) ||
        !aligned16(d_k_cache) || !aligned16(d_v_cache) || !aligned16(d_q_out))
        return HPC_ERR_ARG;
    if (!d_token_req && num_tokens > B) return HPC_ERR_ARG;  // token t is request t

    RopeNormArgs a;
    a.qkv = static_cast<const uint16_t *>(d_qkv);
    a.stride = qkv_row_stride;
    a.q_w = static_cast<const uint16_t *>(d_q_norm_w);
    a.k_w = static_cast<const uint16_t *>(d_k_norm_w);
    a.positions = d_positions;
    a.token_req = d_token_req;
    a.block_table = d_block_table;
    a.k_cache = d_k_cache;
    a.v_cache = d_v_cache;
    a.q_out = d_q_out;
    a.q_scale_out = d_q_scale_out;
    a.flags = d_flags;
    a.base = (double)params->rope_base;
    a.eps = params->eps;
    a.k_scale = fp8 ? k_scale : 1.f;
    a.v_scale = fp8 ? v_scale : 1.f;
    a.N = num_tokens;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.R = Hq + 2 * Hkv;
    a.B = B;
    a.max_pages = max_pages_per_req;
    a.num_pages = num_pages;
    a.layout = params->rope_layout;
    a.norm_first = params->norm_first;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = fp8 ? launch<true>(a, s) : launch<false>(a, s);
    return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}
