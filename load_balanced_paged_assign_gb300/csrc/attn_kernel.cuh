// Persistent load-balanced paged GQA decode attention (HPC-Ops vLLM post,
// "Compute and combine" bullet; SGLang post, 围绕Live KV Work的调度,
// execution paragraph): CTA c drains bin c of the task map.  For every
// descriptor (h, r, tb, te) it streams KV pages block_table[r][tb .. te) of
// KV head h and writes, for the GQA group of h, the normalised partial
// output and its log-sum-exp into split-buffer slot = descriptor index.
//
// GB300 design (the pages' Hopper kernel is not followed):
//  * warp 0 is a producer: one lane walks the whole bin as a flat stream of
//    tiles and issues one TMA tile load per 64-token page of K and of V into
//    a STAGES-deep ring of shared-memory stages (mbarrier full/empty pairs),
//    so loads keep flowing across descriptor boundaries.  Q (and the FP8
//    q-scales) ride in the stage holding a descriptor's first tile.  After
//    the last tile it posts a terminator stage.
//  * warps 1..4 are consumers; warp w owns tokens 16w .. 16w + 15 of every
//    tile and keeps its own online-softmax state; the four states are merged
//    through shared memory at the end of each descriptor.
//  * the contractions run on mma.sync with the operands swapped so the
//    GQA group is the N = 8 side:  S^T[tok, head] = K[tok, :] . Q^T and
//    O^T[dim, head] += V^T[dim, tok] . P^T[tok, head].  P^T's B fragment is
//    the S^T accumulator transposed in registers with movmatrix, so no
//    shared-memory round trip and no padding of the 8-head group to M = 16.
//  * BF16: K via ldmatrix, V via ldmatrix.trans, bf16 MMAs.
//    FP8: Q.K^T on e4m3 MMAs (m16n8k32) straight from the FP8 Q and cache;
//    V is widened exactly to f16 in registers (byte permutes + cvt) with the
//    output dims permuted so each lane needs one 16-byte row segment per
//    token; P stays f16 (never quantised).
//  * tiles land with the 128-byte swizzle; every ldmatrix / 16-byte read
//    below touches 8 distinct 16-byte bank groups.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace hpc {

struct StageInfo {
    int kv_head, req, tile, flags;
    int seqlen, desc_idx, pad0, pad1;
    float qscale[kMaxGroup];
};
static_assert(sizeof(StageInfo) == 64, "StageInfo layout");

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kFullMask = 0xffffffffu;

// Warp-uniform bounded wait: lane 0 polls (so all lanes agree on the
// outcome), then every lane re-observes the completed phase for its own
// acquire of the data the phase guards.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
    ok = __shfl_sync(kFullMask, ok, 0);
    if (ok) mbar_try_wait(bar, parity);
    return ok != 0;
}

template <bool FP8, int STAGES>
struct AttnTraits {
    static constexpr int kElem = FP8 ? 1 : 2;
    static constexpr int kTileBytes = kTile * kHeadDim * kElem;   // one K or V page of one head
    static constexpr int kHalfBytes = kTile * 64 * 2;             // BF16: one 64-dim half
    static constexpr int kQBytes = kMaxGroup * kHeadDim * kElem;  // Q slot per stage
    static constexpr int kCombStride = kHeadDim + 4;              // floats per head row
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + STAGES * kTileBytes;
    static constexpr int kOffQ = kOffV + STAGES * kTileBytes;
    static constexpr int kOffInfo = kOffQ + STAGES * kQBytes;
    static constexpr int kOffBar = kOffInfo + STAGES * (int)sizeof(StageInfo);
    static constexpr int kOffAbort = kOffBar + (2 * STAGES + 2) * 8;  // + epilogue pair
    static constexpr int kOffComb = (kOffAbort + 16 + 15) / 16 * 16;
    static constexpr int kOffStat = kOffComb + kConsumerWarps * kMaxGroup * kCombStride * 4;
    static constexpr int kBytes = kOffStat + 2 * kConsumerWarps * kMaxGroup * 4;
    static constexpr int kSmemBytes = kBytes + 1024;  // slack to align the base to 1024 B
};

template <bool FP8, int STAGES>
__device__ __forceinline__ void attn_producer(const CUtensorMap *tmap_k, const CUtensorMap *tmap_v,
                                              const AttnParams &p, uint8_t *smem, int d_begin,
                                              int d_end, volatile int *abort) {
    using Tr = AttnTraits<FP8, STAGES>;
    const int lane = threadIdx.x & 31;
    StageInfo *info = reinterpret_cast<StageInfo *>(smem + Tr::kOffInfo);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Tr::kOffBar);
    uint64_t *empty = full + STAGES;
    const uint64_t policy = policy_evict_first();
    const uint32_t q_bytes = (uint32_t)(p.G * kHeadDim * Tr::kElem);
    uint32_t it = 0;
    bool ok = true;

    for (int d = d_begin; d < d_end && ok; ++d) {
        const int4 ds = p.desc[d];
        const int h = ds.x, r = ds.y, tb = ds.z, te = ds.w;
        if (tb >= te) continue;  // empty split of the static schedule
        const int L = p.seqlens[r];
        float qs = 1.f;
        if (FP8 && lane < p.G) qs = p.q_scale[(size_t)r * p.Hq + h * p.G + lane];
        float qsg[kMaxGroup];
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) qsg[g] = __shfl_sync(kFullMask, qs, g);
        const int32_t *bt_row = p.block_table + (size_t)r * p.max_pages;
        const uint8_t *q_src = static_cast<const uint8_t *>(p.q) +
                               ((size_t)r * p.Hq + (size_t)h * p.G) * kHeadDim * Tr::kElem;

        for (int t0 = tb; t0 < te && ok; t0 += 32) {
            const int nt = min(32, te - t0);
            int page = 0;
            if (lane < nt) {
                page = bt_row[t0 + lane];
                if (page < 0 || page >= p.num_pages) {
                    atomicOr(p.meta + 3, (int)HPC_FLAG_BAD_PAGE);
                    page = 0;  // stay inside the cache; the result is flagged as invalid
                }
            }
            for (int k = 0; k < nt; ++k) {
                const int pg = __shfl_sync(kFullMask, page, k);
                const int stage = it % STAGES;
                const uint32_t phase = (it / STAGES) & 1u;
                if (!warp_wait(&empty[stage], phase ^ 1u, abort)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int t = t0 + k;
                    const bool first = t == tb;
                    StageInfo &si = info[stage];
                    si.kv_head = h;
                    si.req = r;
                    si.tile = t;
                    si.flags = (first ? kFirst : 0) | (t == te - 1 ? kLast : 0);
                    si.seqlen = L;
                    si.desc_idx = d;
#pragma unroll
                    for (int g = 0; g < kMaxGroup; ++g) si.qscale[g] = qsg[g];
                    mbar_arrive_expect_tx(&full[stage],
                                          2u * Tr::kTileBytes + (first ? q_bytes : 0u));
                    uint8_t *sk = smem + Tr::kOffK + stage * Tr::kTileBytes;
                    uint8_t *sv = smem + Tr::kOffV + stage * Tr::kTileBytes;
                    if (FP8) {
                        tma_load_4d(sk, tmap_k, &full[stage], 0, h, 0, pg, policy);
                        tma_load_4d(sv, tmap_v, &full[stage], 0, h, 0, pg, policy);
                    } else {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            tma_load_5d(sk + half * Tr::kHalfBytes, tmap_k, &full[stage], 0, half,
                                        h, 0, pg, policy);
                            tma_load_5d(sv + half * Tr::kHalfBytes, tmap_v, &full[stage], 0, half,
                                        h, 0, pg, policy);
                        }
                    }
                    if (first)
                        bulk_load(smem + Tr::kOffQ + stage * Tr::kQBytes, q_src, q_bytes,
                                  &full[stage]);
                }
                __syncwarp();
                ++it;
            }
        }
    }
    if (ok) {  // terminator
        const int stage = it % STAGES;
        if (warp_wait(&empty[stage], ((it / STAGES) & 1u) ^ 1u, abort)) {
            if (lane == 0) {
                info[stage].flags = kEnd;
                mbar_arrive(&full[stage]);
            }
            ++it;
        } else {
            ok = false;
        }
    }
    if (!ok && lane == 0) atomicOr(p.meta + 3, (int)HPC_FLAG_TIMEOUT);
    // Before leaving, make sure no copy this warp issued is still in flight
    // (bounded as well): the last phase issued on every stage must complete.
    if (lane == 0) {
        volatile int no_abort = 0;
        const uint32_t from = it > (uint32_t)STAGES ? it - STAGES : 0u;
        for (uint32_t j = from; j < it; ++j)
            mbar_wait(&full[j % STAGES], (j / STAGES) & 1u, &no_abort);
    }
    __syncwarp();
}

// Merge of the four consumer warps' softmax states at the end of a
// descriptor, then the partial output (normalised, times v_scale) and its
// natural-log LSE are written to split-buffer slot `desc_idx`.
template <bool FP8, int STAGES>
__device__ __forceinline__ bool attn_epilogue(const AttnParams &p, uint8_t *smem,
                                              const float (&o)[8][4], float m0, float m1,
                                              float l0, float l1, int desc_idx, uint32_t parity,
                                              volatile int *abort) {
    using Tr = AttnTraits<FP8, STAGES>;
    constexpr int S = Tr::kCombStride;
    const int lane = threadIdx.x & 31, cw = (threadIdx.x >> 5) - 1;
    const int g = lane >> 2, t4 = lane & 3;
    float *comb = reinterpret_cast<float *>(smem + Tr::kOffComb);
    float *stat_m = reinterpret_cast<float *>(smem + Tr::kOffStat);
    float *stat_l = stat_m + kConsumerWarps * kMaxGroup;
    // the four consumer warps meet twice (states written / states consumed)
    // on an mbarrier pair with bounded waits
    uint64_t *comb_full = reinterpret_cast<uint64_t *>(smem + Tr::kOffBar) + 2 * STAGES;
    uint64_t *comb_done = comb_full + 1;

#pragma unroll
    for (int o_ = 4; o_ <= 16; o_ <<= 1) {
        l0 += __shfl_xor_sync(kFullMask, l0, o_);
        l1 += __shfl_xor_sync(kFullMask, l1, o_);
    }
    float *mine = comb + cw * kMaxGroup * S;
    float *row0 = mine + (2 * t4) * S, *row1 = mine + (2 * t4 + 1) * S;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (FP8) {  // m-tile j, row g <-> dim 16g + 2j, row g + 8 <-> 16g + 2j + 1
            const int dd = 16 * g + 2 * j;
            *reinterpret_cast<float2 *>(row0 + dd) = make_float2(o[j][0], o[j][2]);
            *reinterpret_cast<float2 *>(row1 + dd) = make_float2(o[j][1], o[j][3]);
        } else {  // m-tile j, row g <-> dim 16j + g, row g + 8 <-> 16j + g + 8
            const int dd = 16 * j + g;
            row0[dd] = o[j][0];
            row1[dd] = o[j][1];
            row0[dd + 8] = o[j][2];
            row1[dd + 8] = o[j][3];
        }
    }
    if (g == 0) {
        stat_m[cw * kMaxGroup + 2 * t4] = m0;
        stat_m[cw * kMaxGroup + 2 * t4 + 1] = m1;
        stat_l[cw * kMaxGroup + 2 * t4] = l0;
        stat_l[cw * kMaxGroup + 2 * t4 + 1] = l1;
    }
    mbar_arrive(comb_full);  // every lane releases its own writes
    if (!warp_wait(comb_full, parity, abort)) return false;

    const int ct = cw * 32 + lane;
    const int head = ct >> 4, part = ct & 15;
    if (head < p.G) {
        float mw[kConsumerWarps], M = kNegInf;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            mw[w] = stat_m[w * kMaxGroup + head];
            M = fmaxf(M, mw[w]);
        }
        const float Ms = M == kNegInf ? 0.f : M;
        float wsum = 0.f, wt[kConsumerWarps];
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            wt[w] = ex2(mw[w] - Ms);
            wsum += wt[w] * stat_l[w * kMaxGroup + head];
        }
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float *src = comb + (w * kMaxGroup + head) * S;
            const float4 x = *reinterpret_cast<const float4 *>(src + 4 * part);
            const float4 y = *reinterpret_cast<const float4 *>(src + 64 + 4 * part);
            a.x += wt[w] * x.x; a.y += wt[w] * x.y; a.z += wt[w] * x.z; a.w += wt[w] * x.w;
            b.x += wt[w] * y.x; b.y += wt[w] * y.y; b.z += wt[w] * y.z; b.w += wt[w] * y.w;
        }
        const float inv = p.v_scale / wsum;
        float *dst = p.part_o + ((size_t)desc_idx * p.G + head) * kHeadDim;
        *reinterpret_cast<float4 *>(dst + 4 * part) =
            make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
        *reinterpret_cast<float4 *>(dst + 64 + 4 * part) =
            make_float4(b.x * inv, b.y * inv, b.z * inv, b.w * inv);
        if (part == 0) p.part_lse[(size_t)desc_idx * p.G + head] = (Ms + lg2(wsum)) * kLn2;
    }
    mbar_arrive(comb_done);
    return warp_wait(comb_done, parity, abort);  // the buffer may be rewritten after this
}

template <bool FP8, int STAGES>
__device__ __forceinline__ void attn_consumer(const AttnParams &p, uint8_t *smem,
                                              volatile int *abort) {
    using Tr = AttnTraits<FP8, STAGES>;
    const int lane = threadIdx.x & 31, cw = (threadIdx.x >> 5) - 1;
    const int g = lane >> 2, t4 = lane & 3;
    const StageInfo *info = reinterpret_cast<const StageInfo *>(smem + Tr::kOffInfo);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Tr::kOffBar);
    uint64_t *empty = full + STAGES;
    const uint32_t sK0 = smem_u32(smem + Tr::kOffK), sV0 = smem_u32(smem + Tr::kOffV);

    // Lane-constant parts of the shared-memory addresses.  ldmatrix: lane
    // supplies row (lane & 7) of matrix (lane >> 3).
    const int mi = lane >> 3;
    const int tok_k = 16 * cw + (lane & 7) + (mi & 1) * 8;  // K: matrices 1, 3 = rows 8..15
    const int tok_v = 16 * cw + (lane & 7) + (mi >> 1) * 8;  // V^T: matrices 2, 3 = toks 8..15

    float o[8][4];
    float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f, sc0 = 0.f, sc1 = 0.f;
    uint32_t qf[8][2];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        qf[j][0] = qf[j][1] = 0u;
    }

    uint32_t epilogues = 0;
    for (uint32_t it = 0;; ++it) {
        const int stage = it % STAGES;
        if (!warp_wait(&full[stage], (it / STAGES) & 1u, abort)) {
            if (lane == 0) atomicOr(p.meta + 3, (int)HPC_FLAG_TIMEOUT);
            break;
        }
        const int flags = info[stage].flags;
        if (flags & kEnd) break;
        const int tile = info[stage].tile, L = info[stage].seqlen;
        const int desc_idx = info[stage].desc_idx;
        const uint32_t sK = sK0 + stage * Tr::kTileBytes, sV = sV0 + stage * Tr::kTileBytes;

        if (flags & kFirst) {  // new descriptor: load Q^T fragments, reset the state
            // B fragment of Q^T (k = dim, n = head): lane holds head g, dims
            // 2t4.. (bf16) or 4t4.. (e4m3) of each k-step, and +8 / +16 beyond.
            const uint8_t *q = smem + Tr::kOffQ + stage * Tr::kQBytes + g * kHeadDim * Tr::kElem;
            const bool live = g < p.G;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                if (FP8 && s >= 4) break;
                const int off = FP8 ? 32 * s + 4 * t4 : 2 * (16 * s + 2 * t4);
                qf[s][0] = live ? *reinterpret_cast<const uint32_t *>(q + off) : 0u;
                qf[s][1] = live ? *reinterpret_cast<const uint32_t *>(q + off + 16) : 0u;
            }
            sc0 = p.score_scale * info[stage].qscale[2 * t4];
            sc1 = p.score_scale * info[stage].qscale[2 * t4 + 1];
            m0 = m1 = kNegInf;
            l0 = l1 = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        }

        // ---- S^T = K . Q^T for this warp's 16 tokens x 8 heads
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        if (FP8) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int chunk = 2 * s + (mi >> 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(sK + tok_k * 128 + ((chunk ^ (tok_k & 7)) << 4), a0, a1, a2, a3);
                mma_e4m3_16832(s4, a0, a1, a2, a3, qf[s][0], qf[s][1]);
            }
        } else {
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int chunk = (2 * s + (mi >> 1)) & 7;
                const uint32_t addr =
                    sK + (s >> 2) * Tr::kHalfBytes + tok_k * 128 + ((chunk ^ (tok_k & 7)) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(addr, a0, a1, a2, a3);
                mma_bf16_16816(s4, a0, a1, a2, a3, qf[s][0], qf[s][1]);
            }
        }

        // ---- online softmax (log2 domain); tokens at or past L are masked
        const int tok0 = tile * kTile + 16 * cw;  // first token of this warp's slice
        const bool va = tok0 + g < L, vb = tok0 + g + 8 < L;
        const float x0 = va ? s4[0] * sc0 : kNegInf, x1 = va ? s4[1] * sc1 : kNegInf;
        const float x2 = vb ? s4[2] * sc0 : kNegInf, x3 = vb ? s4[3] * sc1 : kNegInf;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int o_ = 4; o_ <= 16; o_ <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, o_));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, o_));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ms0 = mn0 == kNegInf ? 0.f : mn0, ms1 = mn1 == kNegInf ? 0.f : mn1;
        const float al0 = ex2(m0 - ms0), al1 = ex2(m1 - ms1);
        m0 = mn0;
        m1 = mn1;
        const float p0 = ex2(x0 - ms0), p1 = ex2(x1 - ms1);
        const float p2 = ex2(x2 - ms0), p3 = ex2(x3 - ms1);
        uint32_t pk01, pk23;
        if (FP8) {
            pk01 = pack_f16x2(p0, p1);
            pk23 = pack_f16x2(p2, p3);
            const float2 r01 = f16x2_to_f32x2(pk01), r23 = f16x2_to_f32x2(pk23);
            l0 = l0 * al0 + r01.x + r23.x;
            l1 = l1 * al1 + r01.y + r23.y;
        } else {
            pk01 = pack_bf16x2(p0, p1);
            pk23 = pack_bf16x2(p2, p3);
            l0 = l0 * al0 + bf16lo_to_f32(pk01) + bf16lo_to_f32(pk23);
            l1 = l1 * al1 + bf16hi_to_f32(pk01) + bf16hi_to_f32(pk23);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            o[j][0] *= al0;
            o[j][1] *= al1;
            o[j][2] *= al0;
            o[j][3] *= al1;
        }
        // P^T fragments (k = token, n = head): transpose the 8x8 halves
        const uint32_t b0 = movmatrix_trans(pk01), b1 = movmatrix_trans(pk23);

        // ---- O^T += V^T . P^T
        if (FP8) {
            // rows 2t4, 2t4+1, 2t4+8, 2t4+9 of the slice; dims 16g .. 16g+15
            uint4 R[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int tok = 16 * cw + 2 * t4 + (q & 1) + (q >> 1) * 8;
                R[q] = lds128(sV + tok * 128 + ((g ^ (tok & 7)) << 4));
                if (tile * kTile + tok >= L) R[q] = make_uint4(0u, 0u, 0u, 0u);
            }
            const uint32_t wA[4] = {R[0].x, R[0].y, R[0].z, R[0].w};
            const uint32_t wB[4] = {R[1].x, R[1].y, R[1].z, R[1].w};
            const uint32_t wC[4] = {R[2].x, R[2].y, R[2].z, R[2].w};
            const uint32_t wD[4] = {R[3].x, R[3].y, R[3].z, R[3].w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t sel = (j & 1) ? 0x7362u : 0x5140u;
                const uint32_t x01 = __byte_perm(wA[j >> 1], wB[j >> 1], sel);
                const uint32_t x23 = __byte_perm(wC[j >> 1], wD[j >> 1], sel);
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(x01, a0, a1);
                e4m3x4_to_f16x2x2(x23, a2, a3);
                mma_f16_16816(o[j], a0, a1, a2, a3, b0, b1);
            }
        } else {
            const int tv = tok0 + 2 * t4;  // tokens of a0/a1 halves; +8 for a2/a3
            const uint32_t mk01 = (tv < L ? 0x0000ffffu : 0u) | (tv + 1 < L ? 0xffff0000u : 0u);
            const uint32_t mk23 =
                (tv + 8 < L ? 0x0000ffffu : 0u) | (tv + 9 < L ? 0xffff0000u : 0u);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int chunk = (2 * j + (mi & 1)) & 7;
                const uint32_t addr =
                    sV + (j >> 2) * Tr::kHalfBytes + tok_v * 128 + ((chunk ^ (tok_v & 7)) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(addr, a0, a1, a2, a3);
                mma_bf16_16816(o[j], a0 & mk01, a1 & mk01, a2 & mk23, a3 & mk23, b0, b1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);  // stage may now be refilled

        if (flags & kLast) {
            if (!attn_epilogue<FP8, STAGES>(p, smem, o, m0, m1, l0, l1, desc_idx,
                                            epilogues & 1u, abort)) {
                if (lane == 0) atomicOr(p.meta + 3, (int)HPC_FLAG_TIMEOUT);
                break;
            }
            ++epilogues;
        }
    }
}

template <bool FP8, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
    using Tr = AttnTraits<FP8, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Tr::kOffBar);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Tr::kOffAbort);
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);                        // producer arrive + TMA bytes
            mbar_init(&full[STAGES + s], kConsumerWarps);  // one arrive per consumer warp
        }
        mbar_init(&full[2 * STAGES], 32 * kConsumerWarps);      // epilogue: states written
        mbar_init(&full[2 * STAGES + 1], 32 * kConsumerWarps);  // epilogue: states consumed
        *abort = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    __syncthreads();
    const int d_begin = p.bin_ptr[blockIdx.x], d_end = p.bin_ptr[blockIdx.x + 1];
    if (threadIdx.x < 32)
        attn_producer<FP8, STAGES>(&tmap_k, &tmap_v, p, smem, d_begin, d_end, abort);
    else
        attn_consumer<FP8, STAGES>(p, smem, abort);
}

}  // namespace hpc
