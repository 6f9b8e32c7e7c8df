// Fused attention prologue (HpcRopeNorm): QK-Norm, RoPE, the paged KV-cache
// write and, for FP8, the per-(token, head) E4M3 query.
//
// The op is described in the vLLM integration post ("A fused attention
// prologue") and the SGLang post (the Hy3 FP8 prologue paragraph): from the
// fused QKV projection it normalises and rotates the query and key heads in
// the model's order, writes K and V straight into the paged cache, and emits
// the FP8 query with its scale for the attention kernel.
//
// It is a pure streaming op (a token brings (Hq + 2 Hkv) * 256 bytes in and
// about half of that out), so the design is about bytes in flight and short
// dependency chains:
//   * persistent CTAs of 8 warps stride over tokens; each token's fused QKV
//     row is staged in shared memory by one bulk copy (TMA engine), issued
//     several tokens ahead through a ring of stages with mbarrier completion
//     (every wait bounded), so the loads do not hold registers;
//   * a warp owns the head rows j == warp (mod 8) of each token and runs
//     same-kind rows (query, key or value) in batches of up to 4, so the
//     reductions (RMS, FP8 amax) of a batch interleave;
//   * lanes hold the dims so that every rotated pair sits in one lane (dims
//     2l, 2l+1, 64+2l, 65+2l for the halves layout; 4l..4l+3 interleaved):
//     the rotation needs no shuffles;
//   * RoPE angles come from an fp64 frequency table (given by the caller or
//     built per CTA); per token the angle pos * freq is formed in fp32 as an
//     exact product plus its rounding error and reduced modulo 2 pi with a
//     two-constant split of 2 pi (the Cody-Waite method), so positions up to
//     2^24 keep an angle error of a few 1e-7 rad;
//   * the angle table and the token's cache slot for the next token are
//     computed while the current token is processed (double-buffered), one
//     __syncthreads per token.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace hpc {
namespace {

#ifndef HPC_RN_MIN_CTAS
#define HPC_RN_MIN_CTAS 3  // resident CTAs per SM the register budget must allow
#endif

constexpr int kRnWarps = 8;
constexpr int kRnThreads = 32 * kRnWarps;
constexpr int kMaxStages = 8;
constexpr int kStageBudget = 40 * 1024;  // QKV bytes a CTA keeps in flight (at least 2 stages)
constexpr int kRowBytes = kHeadDim * 2;  // one BF16 head row
constexpr int kMaxPosition = 1 << 24;    // positions are exact in fp32 below this
constexpr float kTwoPiHi = 6.2831854820251465f;     // fp32(2 pi)
constexpr float kTwoPiLo = -1.7484555314695172e-7f;  // 2 pi - fp32(2 pi)
constexpr float kInvTwoPi = 0.159154937f;
constexpr float kInvPi = 0.318309873f;

enum RowKind { kQ = 0, kK = 1, kV = 2 };

struct RopeNormArgs {
    const uint16_t *qkv;
    int64_t stride;  // elements between token rows
    const uint16_t *q_w;
    const uint16_t *k_w;
    const int32_t *positions;
    const int32_t *token_req;
    const int32_t *block_table;
    const double *freq;  // [64] or nullptr: built per CTA from base
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
    int stages;
    int norm_first;
};

// ------------------------------------------------------------ lane layout
// A head row is handled by one half-warp (16 lanes, 8 dims each), so a warp
// instruction covers two rows and a row reduction takes four shuffles.
// Sub-lane s = lane & 15 holds, and pairs under the rotation:
//   halves:      dims 4s..4s+3 and 64+4s..67+4s; pairs (x[k], x[4+k])
//   interleaved: dims 8s..8s+7;                  pairs (x[2k], x[2k+1])
// In both layouts pair k of sub-lane s has frequency 4s + k.

__device__ __forceinline__ void unpack2(uint32_t w, float &lo, float &hi) {
    lo = bf16lo_to_f32(w);
    hi = bf16hi_to_f32(w);
}

template <int LAYOUT>
__device__ __forceinline__ uint4 load_words(const char *row, int s) {
    if (LAYOUT == HPC_ROPE_HALVES) {
        const uint2 lo = *reinterpret_cast<const uint2 *>(row + 8 * s);
        const uint2 hi = *reinterpret_cast<const uint2 *>(row + 128 + 8 * s);
        return make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    return *reinterpret_cast<const uint4 *>(row + 16 * s);
}

template <int LAYOUT>
__device__ __forceinline__ void store_words(char *row, int s, uint4 v) {
    if (LAYOUT == HPC_ROPE_HALVES) {
        *reinterpret_cast<uint2 *>(row + 8 * s) = make_uint2(v.x, v.y);
        *reinterpret_cast<uint2 *>(row + 128 + 8 * s) = make_uint2(v.z, v.w);
    } else {
        *reinterpret_cast<uint4 *>(row + 16 * s) = v;
    }
}

__device__ __forceinline__ void unpack8(uint4 v, float (&x)[8]) {
    unpack2(v.x, x[0], x[1]);
    unpack2(v.y, x[2], x[3]);
    unpack2(v.z, x[4], x[5]);
    unpack2(v.w, x[6], x[7]);
}

// E4M3 (round to nearest even, saturating) of four values, y[0] in the low byte.
__device__ __forceinline__ uint32_t e4m3x4(float y0, float y1, float y2, float y3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(y1), "f"(y0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(y3), "f"(y2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

template <int LAYOUT>
__device__ __forceinline__ void store_e4m3(char *row, int s, const float (&y)[8]) {
    const uint32_t a = e4m3x4(y[0], y[1], y[2], y[3]), b = e4m3x4(y[4], y[5], y[6], y[7]);
    if (LAYOUT == HPC_ROPE_HALVES) {
        *reinterpret_cast<uint32_t *>(row + 4 * s) = a;
        *reinterpret_cast<uint32_t *>(row + 64 + 4 * s) = b;
    } else {
        *reinterpret_cast<uint2 *>(row + 8 * s) = make_uint2(a, b);
    }
}

template <int LAYOUT>
__device__ __forceinline__ void store_bf16(char *row, int s, const float (&y)[8]) {
    store_words<LAYOUT>(row, s,
                        make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                   pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7])));
}

// The rotation of this sub-lane's four pairs: c, sn = cos, sin of its four
// frequencies, nsn = -sin.  In the halves layout pairs k and k + 1 sit in
// consecutive registers, so two pairs take one paired FP32 instruction
// (each lane of which rounds like the scalar one).
template <int LAYOUT>
__device__ __forceinline__ void rotate(float (&x)[8], const float (&c)[4], const float (&sn)[4],
                                       const float (&nsn)[4]) {
    if constexpr (LAYOUT == HPC_ROPE_HALVES) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float2 p = make_float2(x[2 * h], x[2 * h + 1]);
            const float2 q = make_float2(x[4 + 2 * h], x[5 + 2 * h]);
            const float2 cc = make_float2(c[2 * h], c[2 * h + 1]);
            const float2 p2 = __ffma2_rn(p, cc, __fmul2_rn(q, make_float2(nsn[2 * h], nsn[2 * h + 1])));
            const float2 q2 = __ffma2_rn(q, cc, __fmul2_rn(p, make_float2(sn[2 * h], sn[2 * h + 1])));
            x[2 * h] = p2.x, x[2 * h + 1] = p2.y;
            x[4 + 2 * h] = q2.x, x[5 + 2 * h] = q2.y;
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float p = x[2 * k], q = x[2 * k + 1];
            x[2 * k] = fmaf(p, c[k], q * nsn[k]);
            x[2 * k + 1] = fmaf(q, c[k], p * sn[k]);
        }
    }
}

// x[k] *= m[k] for the 8 values, two per instruction.
__device__ __forceinline__ void mul8(float (&x)[8], const float (&m)[8]) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float2 v = __fmul2_rn(make_float2(x[2 * h], x[2 * h + 1]),
                                    make_float2(m[2 * h], m[2 * h + 1]));
        x[2 * h] = v.x, x[2 * h + 1] = v.y;
    }
}

// x[k] *= m for the 8 values, two per instruction.
__device__ __forceinline__ void scale8(float (&x)[8], float m) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float2 v = __fmul2_rn(make_float2(x[2 * h], x[2 * h + 1]), make_float2(m, m));
        x[2 * h] = v.x, x[2 * h + 1] = v.y;
    }
}

// Sum of squares of the 8 values (two partial sums, paired).
__device__ __forceinline__ float sumsq8(const float (&x)[8]) {
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float2 v = make_float2(x[2 * h], x[2 * h + 1]);
        acc = __ffma2_rn(v, v, acc);
    }
    return acc.x + acc.y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float absmax8(const float (&x)[8]) {
    return fmax3(fmax3(fabsf(x[0]), fabsf(x[1]), fabsf(x[2])),
                 fmax3(fabsf(x[3]), fabsf(x[4]), fabsf(x[5])), fmaxf(fabsf(x[6]), fabsf(x[7])));
}

// x[k] / s correctly rounded to FP32 for the 8 values, from y = RN(1/s):
// q = RN(x y) is within an ulp of x / s, r = x - s q is exact (one FMA), and
// RN(q + r y) is the correctly rounded quotient (Markstein's theorem on
// division with a fused multiply-add); two values per instruction.
__device__ __forceinline__ void div8(float (&x)[8], float s, float y) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float2 v = make_float2(x[2 * h], x[2 * h + 1]);
        const float2 q = __fmul2_rn(v, make_float2(y, y));
        const float2 r = __ffma2_rn(make_float2(-s, -s), q, v);
        const float2 o = __ffma2_rn(r, make_float2(y, y), q);
        x[2 * h] = o.x, x[2 * h + 1] = o.y;
    }
}

// ------------------------------------------------------------ one batch of rows
// NP row pairs of one kind.  Pair i of the batch is rows row0 + 16 i and
// row0 + 16 i + 1; this half-warp takes the one at offset `half`.  Rows at or
// past `end` (the odd last row of a kind) are computed on a stand-in row and
// not stored.
template <bool FP8, int LAYOUT, bool NF, int KIND, int NP>
__device__ __forceinline__ void rows_batch(const RopeNormArgs &a, const char *stage, int t,
                                           int row0, int end, int half, int s,
                                           const float (&c)[4], const float (&sn)[4],
                                           const float (&nsn)[4], long long slot,
                                           const float (&w)[8], float kv_scale) {
    constexpr int kElem = FP8 ? 1 : 2;
    if (KIND != kQ && slot < 0) return;  // no cache slot for this token (uniform per CTA)
    int row[NP];
    bool valid[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        row[i] = row0 + 16 * i + half;
        valid[i] = row[i] < end;
        if (!valid[i]) row[i] = end - 1;
    }
    if constexpr (KIND == kV && !FP8) {  // BF16 value rows: copied word for word
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const uint4 v = load_words<LAYOUT>(stage + (size_t)row[i] * kRowBytes, s);
            if (valid[i])
                store_words<LAYOUT>(static_cast<char *>(a.v_cache) +
                                        (slot * a.Hkv + (row[i] - a.Hq - a.Hkv)) *
                                            (kHeadDim * kElem), s, v);
        }
        return;
    } else {
        float x[NP][8];
#pragma unroll
        for (int i = 0; i < NP; ++i)
            unpack8(load_words<LAYOUT>(stage + (size_t)row[i] * kRowBytes, s), x[i]);
        if constexpr (KIND == kV) {  // FP8 value rows: the correctly rounded quotient by
            // the cache scale (BF16 inputs over the scale often land exactly
            // on an E4M3 midpoint, where only the exact quotient rounds to even)
            const float y = __frcp_rn(kv_scale);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                div8(x[i], kv_scale, y);
                if (valid[i])
                    store_e4m3<LAYOUT>(static_cast<char *>(a.v_cache) +
                                           (slot * a.Hkv + (row[i] - a.Hq - a.Hkv)) * kHeadDim,
                                       s, x[i]);
            }
            return;
        } else {
            // RMS of the row (the rotation keeps it), then v = the rotated,
            // weighted row before the norm factor: the output is inv * v
            float inv[NP];
#pragma unroll
            for (int i = 0; i < NP; ++i) inv[i] = sumsq8(x[i]);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
#pragma unroll
                for (int i = 0; i < NP; ++i) inv[i] += __shfl_xor_sync(0xffffffffu, inv[i], o);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                inv[i] = rsqrtf(fmaf(inv[i], 1.0f / kHeadDim, a.eps));
                if constexpr (NF) {
                    mul8(x[i], w);
                    rotate<LAYOUT>(x[i], c, sn, nsn);
                } else {
                    rotate<LAYOUT>(x[i], c, sn, nsn);
                    mul8(x[i], w);
                }
            }
            if constexpr (KIND == kQ) {
                if (FP8) {
                    // codes = v * 448 / amax(v): the norm factor cancels; the
                    // scale is amax(inv * v) / 448
                    float amax[NP];
#pragma unroll
                    for (int i = 0; i < NP; ++i) amax[i] = absmax8(x[i]);
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1)
#pragma unroll
                        for (int i = 0; i < NP; ++i)
                            amax[i] = fmaxf(amax[i], __shfl_xor_sync(0xffffffffu, amax[i], o));
#pragma unroll
                    for (int i = 0; i < NP; ++i) {
                        const float ymax = amax[i] * inv[i];
                        const bool live = ymax > 0.f;
                        const float mul = live ? __fdividef(448.0f, amax[i]) : 0.f;
                        scale8(x[i], mul);
                        if (valid[i]) {
                            const size_t qrow = (size_t)t * a.Hq + row[i];
                            store_e4m3<LAYOUT>(static_cast<char *>(a.q_out) + qrow * kHeadDim, s,
                                               x[i]);
                            if (s == 0) a.q_scale_out[qrow] = live ? ymax * (1.0f / 448.0f) : 1.f;
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < NP; ++i) {
                        scale8(x[i], inv[i]);
                        if (valid[i])
                            store_bf16<LAYOUT>(static_cast<char *>(a.q_out) +
                                                   ((size_t)t * a.Hq + row[i]) * (kHeadDim * 2),
                                               s, x[i]);
                    }
                }
            } else {  // key rows: into the cache slot
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    const float m = FP8 ? inv[i] * __frcp_rn(kv_scale) : inv[i];
                    scale8(x[i], m);
                    if (!valid[i]) continue;
                    char *dst = static_cast<char *>(a.k_cache) +
                                (slot * a.Hkv + (row[i] - a.Hq)) * (kHeadDim * kElem);
                    if (FP8) store_e4m3<LAYOUT>(dst, s, x[i]);
                    else store_bf16<LAYOUT>(dst, s, x[i]);
                }
            }
        }
    }
}

// Rows [begin, end) of one kind form pairs (begin + 2p, begin + 2p + 1); pair
// p has the global number pair0 + p, and warp w takes the pairs numbered
// w (mod 8), so consecutive kinds continue the rotation over the warps.
template <bool FP8, int LAYOUT, bool NF, int KIND>
__device__ __forceinline__ void rows_of_kind(const RopeNormArgs &a, const char *stage, int t,
                                             int begin, int end, int pair0, int warp, int half,
                                             int s, const float (&c)[4], const float (&sn)[4],
                                             const float (&nsn)[4], long long slot,
                                             const float (&w)[8], float kv_scale) {
    const int npairs = (end - begin + 1) / 2;
    int p = ((warp - pair0) % kRnWarps + kRnWarps) % kRnWarps;  // first pair of this warp
    int count = p < npairs ? (npairs - 1 - p) / kRnWarps + 1 : 0;
    for (; count >= 2; count -= 2, p += 2 * kRnWarps)
        rows_batch<FP8, LAYOUT, NF, KIND, 2>(a, stage, t, begin + 2 * p, end, half, s, c, sn, nsn,
                                             slot, w, kv_scale);
    if (count) rows_batch<FP8, LAYOUT, NF, KIND, 1>(a, stage, t, begin + 2 * p, end, half, s, c,
                                                    sn, nsn, slot, w, kv_scale);
}

// cos/sin of pos * freq_i, freq_i = hi + lo (two floats), reduced modulo 2 pi.
__device__ __forceinline__ float2 rope_angle(int pos, float hi, float lo) {
    const float p = (float)pos;                 // exact: |pos| < 2^24 for valid tokens
    const float prod = p * hi;
    const float err = fmaf(p, hi, -prod);       // exact rounding error of the product
    const float k = rintf(prod * kInvTwoPi);
    float r = fmaf(-k, kTwoPiHi, prod);
    r = fmaf(-k, kTwoPiLo, r);
    r += fmaf(p, lo, err);                      // the small terms, |.| < 1.5
    const float k2 = rintf(r * kInvTwoPi);      // back into [-pi, pi]
    r = fmaf(-k2, kTwoPiHi, r);
    r = fmaf(-k2, kTwoPiLo, r);
    float s, c;
    sincospif(r * kInvPi, &s, &c);
    return make_float2(c, s);
}

// (cos, sin) of frequency i into a buffer of the angle table.
__device__ __forceinline__ void store_angle(float *tab, int i, float2 cs) {
    tab[(i >> 2) * 8 + (i & 3)] = cs.x;
    tab[(i >> 2) * 8 + 4 + (i & 3)] = cs.y;
}

// The token's cache slot (page * 64 + offset), or -1 with a flag raised.
__device__ __forceinline__ long long token_slot(const RopeNormArgs &a, int t, int pos, int req) {
    if (req < 0 || req >= a.B || pos < 0 || pos >= a.max_pages * kTile) {
        if (a.flags) atomicOr(a.flags, (int)HPC_FLAG_BAD_SEQLEN);
        return -1;
    }
    const int page = a.block_table[(size_t)req * a.max_pages + pos / kTile];
    if (page < 0 || page >= a.num_pages) {
        if (a.flags) atomicOr(a.flags, (int)HPC_FLAG_BAD_PAGE);
        return -1;
    }
    return (long long)page * kTile + (pos % kTile);
}

// Bounded wait on an mbarrier phase, uniform across the warp: every lane
// polls (and so observes the phase itself); the lanes agree on the outcome.
__device__ __forceinline__ bool warp_wait_phase(uint64_t *bar, uint32_t parity,
                                                volatile int *abort) {
    return mbar_wait_warp(bar, parity, abort);
}

template <bool FP8, int LAYOUT, bool NF>
__global__ void __launch_bounds__(kRnThreads, HPC_RN_MIN_CTAS) rope_norm_kernel(const RopeNormArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int row_bytes = a.R * kRowBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.stages * row_bytes);
    // [2][128]: per buffer and group g of frequencies 4g .. 4g + 3, their
    // four cosines then their four sines
    float *s_ang = reinterpret_cast<float *>(full + kMaxStages);
    float *s_fhi = s_ang + 2 * 128;
    float *s_flo = s_fhi + 64;
    long long *s_slot = reinterpret_cast<long long *>(s_flo + 64);  // [2]
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_slot + 2);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grid = gridDim.x;
    const int n_it = (a.N - (int)blockIdx.x + grid - 1) / grid;  // >= 1: the grid is <= N

    auto issue = [&](int it) {  // bulk copy of iteration it's token row into its stage
        const int t = blockIdx.x + it * grid;
        const int s = it % a.stages;
        mbar_arrive_expect_tx(&full[s], row_bytes);
        bulk_load(smem + (size_t)s * row_bytes, a.qkv + (size_t)t * a.stride, row_bytes,
                  &full[s]);
    };

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) mbar_init(&full[s], 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    // Everything this grid reads may come from the kernel before it.
    grid_dependency_wait();
    int issued = 0;  // (thread 0) iterations whose copy has been issued
    if (tid == 0)
        for (; issued < min(a.stages, n_it); ++issued) issue(issued);
    // the first token's position (and request), in flight with the table below
    int pos0 = 0, req0 = 0;
    if (tid <= 64) {
        pos0 = a.positions[blockIdx.x];
        req0 = a.token_req ? a.token_req[blockIdx.x] : (int)blockIdx.x;
    }
    if (tid < 64) {
        const double f = a.freq ? a.freq[tid] : pow(a.base, -(double)tid / 64.0);
        const float hi = (float)f;
        s_fhi[tid] = hi;
        s_flo[tid] = (float)(f - (double)hi);
    }
    const int half = lane >> 4, sub = lane & 15;
    float wq[8], wk[8];
    unpack8(load_words<LAYOUT>(reinterpret_cast<const char *>(a.q_w), sub), wq);
    unpack8(load_words<LAYOUT>(reinterpret_cast<const char *>(a.k_w), sub), wk);
    __syncthreads();  // barriers initialised, frequency table ready

    // angles and cache slot of the first token
    if (tid < 64) store_angle(s_ang, tid, rope_angle(pos0, s_fhi[tid], s_flo[tid]));
    else if (tid == 64) s_slot[0] = token_slot(a, blockIdx.x, pos0, req0);

    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
        const int t = blockIdx.x + it * grid;
        const int buf = it & 1;
        const int stage = it % a.stages;
        __syncthreads();  // this token's angles and slot are ready; the previous stage is free
        if (tid == 0 && it >= 1 && it - 1 + a.stages < n_it && !*s_abort)
            issue(issued++);  // == it - 1 + stages, into the stage freed by iteration it - 1
        // the next token's position and request, loaded while this one is processed
        int pos_n = 0, req_n = 0;
        const bool has_next = it + 1 < n_it;
        if (tid <= 64 && has_next) {
            pos_n = a.positions[t + grid];
            req_n = a.token_req ? a.token_req[t + grid] : t + grid;
        }
        if (ok) ok = warp_wait_phase(&full[stage], (uint32_t)(it / a.stages) & 1u, s_abort);
        if (ok) {
            const char *st = reinterpret_cast<const char *>(smem) + (size_t)stage * row_bytes;
            float c[4], sn[4], nsn[4];
            {
                const float4 *a4 = reinterpret_cast<const float4 *>(s_ang + buf * 128 + 8 * sub);
                const float4 c4 = a4[0], s4 = a4[1];
                c[0] = c4.x, c[1] = c4.y, c[2] = c4.z, c[3] = c4.w;
                sn[0] = s4.x, sn[1] = s4.y, sn[2] = s4.z, sn[3] = s4.w;
#pragma unroll
                for (int k = 0; k < 4; ++k) nsn[k] = -sn[k];
            }
            const long long slot = s_slot[buf];
            const int pq = (a.Hq + 1) / 2, pk = (a.Hkv + 1) / 2;  // pairs of each kind
            rows_of_kind<FP8, LAYOUT, NF, kQ>(a, st, t, 0, a.Hq, 0, warp, half, sub, c, sn, nsn, slot, wq,
                                          1.f);
            rows_of_kind<FP8, LAYOUT, NF, kK>(a, st, t, a.Hq, a.Hq + a.Hkv, pq, warp, half, sub, c, sn, nsn,
                                          slot, wk, a.k_scale);
            rows_of_kind<FP8, LAYOUT, NF, kV>(a, st, t, a.Hq + a.Hkv, a.R, pq + pk, warp, half, sub,
                                          c, sn, nsn, slot, wk, a.v_scale);
        }
        if (has_next) {
            if (tid < 64) store_angle(s_ang + (buf ^ 1) * 128, tid, rope_angle(pos_n, s_fhi[tid], s_flo[tid]));
            else if (tid == 64) s_slot[buf ^ 1] = token_slot(a, t + grid, pos_n, req_n);
        }
    }
    if (*s_abort) {
        // a copy never completed: report it, and let no copy land after exit
        // (a stage holds at most one copy at a time: wait for the last one issued
        // into each stage, again with a time limit)
        if (tid == 0) {
            if (a.flags) atomicOr(a.flags, (int)HPC_FLAG_TIMEOUT);
            for (int it = max(0, issued - a.stages); it < issued; ++it) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&full[it % a.stages], (uint32_t)(it / a.stages) & 1u) &&
                       globaltimer_ns() - t0 < 1000000000ull) {
                }
            }
        }
        __syncthreads();
    }
}

__global__ void rope_frequencies_kernel(double base, double *freq) {
    const int i = threadIdx.x;
    if (i < kHeadDim / 2) freq[i] = pow(base, -(double)(2 * i) / kHeadDim);
}

// ------------------------------------------------------------ host side
using KernelFn = void (*)(const RopeNormArgs);

template <bool FP8, int LAYOUT>
KernelFn kernel_for_order(bool norm_first) {
    return norm_first ? rope_norm_kernel<FP8, LAYOUT, true> : rope_norm_kernel<FP8, LAYOUT, false>;
}

KernelFn kernel_for(bool fp8, int layout, bool norm_first) {
    if (fp8) return layout == HPC_ROPE_HALVES
                        ? kernel_for_order<true, HPC_ROPE_HALVES>(norm_first)
                        : kernel_for_order<true, HPC_ROPE_INTERLEAVED>(norm_first);
    return layout == HPC_ROPE_HALVES ? kernel_for_order<false, HPC_ROPE_HALVES>(norm_first)
                                     : kernel_for_order<false, HPC_ROPE_INTERLEAVED>(norm_first);
}

size_t smem_bytes(int R, int stages) {
    return (size_t)stages * R * kRowBytes + kMaxStages * 8 + 2 * 64 * 8 + 2 * 64 * 4 + 2 * 8 + 16;
}

// Per device and kernel variant: the dynamic shared memory already allowed,
// and the last occupancy query (for one shared-memory size).
struct VariantCache {
    int smem_allowed = 0;
    int smem_queried = -1;
    int cap = 0;
};
constexpr int kMaxDevices = 64;
VariantCache g_cache[kMaxDevices][8];
std::mutex g_cache_mutex;

cudaError_t launch(const RopeNormArgs &a, bool fp8, int layout, cudaStream_t s) {
    const bool nf = a.norm_first != 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const KernelFn fn = kernel_for(fp8, layout, nf);
    const int smem = (int)smem_bytes(a.R, a.stages);
    int cap = 0;
    {
        std::lock_guard<std::mutex> lock(g_cache_mutex);
        VariantCache &vc = g_cache[dev][(fp8 ? 4 : 0) + 2 * layout + (nf ? 1 : 0)];
        if (smem > vc.smem_allowed) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            vc.smem_allowed = smem;
        }
        if (vc.smem_queried != smem) {
            int sms = 0, per_sm = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kRnThreads, smem);
            if (e != cudaSuccess) return e;
            if (per_sm < 1) return cudaErrorInvalidConfiguration;
            vc.smem_queried = smem;
            vc.cap = sms * per_sm;
        }
        cap = vc.cap;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(a.N, cap));
    cfg.blockDim = dim3(kRnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, a);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite_positive(float x) { return std::isfinite(x) && x > 0.f; }

}  // namespace
}  // namespace hpc

extern "C" hpc_status hpc_rope_frequencies(float rope_base, double *d_freq, hpc_stream_t stream) {
    using namespace hpc;
    if (!finite_positive(rope_base) || !d_freq || !aligned16(d_freq)) return HPC_ERR_ARG;
    rope_frequencies_kernel<<<1, kHeadDim / 2, 0, static_cast<cudaStream_t>(stream)>>>(
        (double)rope_base, d_freq);
    return cudaGetLastError() == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}

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
    const int R = Hq + 2 * Hkv;
    int stages = std::min(kMaxStages, std::max(2, kStageBudget / (R * kRowBytes)));
    if (smem_bytes(R, stages) > 200 * 1024) return HPC_ERR_UNSUPPORTED;  // > ~390 head rows
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_ARG;
    const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
    if (!std::isfinite(params->eps) || params->eps < 0.f || !finite_positive(params->rope_base))
        return HPC_ERR_ARG;
    if (params->rope_layout != HPC_ROPE_HALVES && params->rope_layout != HPC_ROPE_INTERLEAVED)
        return HPC_ERR_ARG;
    if (params->norm_first != 0 && params->norm_first != 1) return HPC_ERR_ARG;
    if (params->freq && !aligned16(params->freq)) return HPC_ERR_ARG;
    if (fp8 && (!finite_positive(k_scale) || !finite_positive(v_scale))) return HPC_ERR_ARG;
    if ((int64_t)B * max_pages_per_req >= (int64_t)1 << 31) return HPC_ERR_UNSUPPORTED;
    // cache positions must stay exact in fp32 (the RoPE angle is formed there)
    if ((int64_t)max_pages_per_req * kTile > kMaxPosition) return HPC_ERR_UNSUPPORTED;
    if (num_tokens == 0) return HPC_OK;
    if (!d_qkv || !d_q_norm_w || !d_k_norm_w || !d_positions || !d_block_table || !d_k_cache ||
        !d_v_cache || !d_q_out || (fp8 && !d_q_scale_out))
        return HPC_ERR_ARG;
    if (qkv_row_stride < (int64_t)R * HPC_HEAD_DIM || qkv_row_stride % 8 != 0) return HPC_ERR_ARG;
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
    a.freq = params->freq;
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
    a.R = R;
    a.B = B;
    a.max_pages = max_pages_per_req;
    a.num_pages = num_pages;
    a.stages = stages;
    a.norm_first = params->norm_first;
    const cudaError_t e = launch(a, fp8, params->rope_layout, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}
