// Extend / prefill attention over the paged BF16 KV cache on the fifth-
// generation tensor cores: the "prefill" and "extend" rows of the vLLM
// post's attention comparison (Table 4, "Attention: HPC-Ops vs
// FlashAttention / Triton / FlashInfer").  Request r holds L_r live tokens in
// its pages; the last q_len of them are the new query tokens, and query token
// i (position L_r - q_len + i) attends every token at a position up to its
// own (causal).  A prefill is the case L_r = q_len; an extend has a cached
// prefix before the new tokens.
//
// GB300 design (tcgen05 + TMEM + TMA), one CTA per (request, query head,
// pair of 128-token query tiles), heaviest (last) pairs first:
//   * warp 8 loads the CTA's two Q tiles once and then streams 128-token K
//     and V tiles (two 64-token pages each, gathered through the block table)
//     into two-stage rings with TMA (128-byte swizzle);
//   * one thread of warp 9 issues tcgen05.mma.  Per KV tile j and Q tile x:
//     S_x = Q_x K_j^T (both operands in shared memory) into x's TMEM score
//     columns, and once the softmax has turned them into P_x, O_x += P_x V_j
//     with P_x read straight from TMEM and V from its cache layout (an
//     MN-major shared-memory operand).  The two Q tiles share every K/V tile
//     and alternate on the tensor cores: x's next scores are issued right
//     behind x's PV product, while the other tile's softmax runs;
//   * warps 0-3 run the online softmax of Q tile 0 and warps 4-7 that of Q
//     tile 1, one thread per query row (warp w reads TMEM lanes 32 (w mod 4)
//     ..): tcgen05.ld of the row's 128 scores, the causal mask on the
//     diagonal, P = exp2(S * scale * log2 e - m) packed to BF16 and written
//     over the scores with tcgen05.st.  The running maximum m moves only when
//     a tile's maximum exceeds it by more than 8 (log2 units), so P stays <=
//     256 and the accumulator is rescaled (tcgen05.ld, multiply, tcgen05.st)
//     only on those rare tiles; the result is the same softmax, since O and
//     the row sum always share the reference m;
//   * the epilogue divides O by the row sum and writes BF16.
// A tcgen05.commit covers every MMA its thread issued before it, so when x's
// scores for tile j are complete, x's product with tile j - 1 is complete
// too: the softmax may read and rescale O_x without a further wait.
// Every mbarrier wait is bounded; on a timeout the CTA raises the error flag,
// waits (bounded) for its copies and MMAs in flight, frees TMEM and leaves.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>

#include "internal.h"
#include "tcgen05.cuh"

namespace hpc {
namespace {

constexpr int kQB = 128;                 // query rows per Q tile (UMMA M)
constexpr int kQT = 2;                   // Q tiles per CTA
constexpr int kKB = 128;                 // KV tokens per tile: two pages
constexpr int kHalf = 128 * 128;         // 128 rows x 64 BF16: one 128-byte column block
constexpr int kTileBytes = 2 * kHalf;    // a 128 x 128 BF16 tile (Q, K or V)
constexpr int kKStages = 2;              // K ring depth
constexpr int kVStages = 2;              // V ring depth
constexpr int kSoftmaxWarps = 4 * kQT;
constexpr int kProducerWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr uint32_t kTmemCols = 512;      // S_x / P_x at 128 x; O_x at 256 + 128 x
constexpr int kOCol = 256;
constexpr float kRescaleLog2 = 8.f;      // P <= 2^8 between reference moves

// Shared-memory layout (offsets from the 1024-byte aligned base).
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQT * kTileBytes;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffBar = kOffV + kVStages * kTileBytes;
// barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2],
// p_full[2], o_done[2], mma_done, v_tail
constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 3 * kQT + 2;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort word
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory over the per-CTA limit");

struct PrefillArgs {
    const int32_t *seqlens;
    const int32_t *block_table;
    __nv_bfloat16 *out;
    int32_t *flags;
    int B, Hq, Hkv, G, q_len, max_pages, num_pages, n_qp;
    float score_scale;  // sm_scale * log2(e)
};

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Lane 0 waits (bounded); the verdict is broadcast and every lane then
// observes the completed phase itself (acquire).  Warp-uniform result.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar, parity);
    return ok != 0;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// The causal extent of a Q tile: its first query row, the KV tiles its rows
// read, and the last token its first row sees.
struct QTile {
    int first, tiles, lim_first;
};

__device__ __forceinline__ QTile qtile(int i0, int L, int q_len) {
    QTile t;
    t.first = i0;
    t.lim_first = min(L - q_len + i0, L - 1);
    t.tiles = 0;
    if (i0 < q_len) {
        const int lim_last = min(L - q_len + min(i0 + kQB - 1, q_len - 1), L - 1);
        t.tiles = lim_last >= 0 ? lim_last / kKB + 1 : 0;
    }
    return t;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tq,
                        const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *q_full = bars;
    uint64_t *k_full = bars + 1, *k_empty = k_full + kKStages;
    uint64_t *v_full = k_empty + kKStages, *v_empty = v_full + kVStages;
    uint64_t *s_full = v_empty + kVStages;  // [x]: S_x complete (and every MMA before it)
    uint64_t *p_full = s_full + kQT;       // [x]: P_x written (four warps)
    uint64_t *o_done = p_full + kQT;       // [x]: O_x += P_x V complete
    uint64_t *mma_done = o_done + kQT;
    uint64_t *v_tail = mma_done + 1;       // the last V tile with its free slots zeroed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // heaviest query tiles (the last ones: the longest causal prefix) first
    const int per_qp = a.B * a.Hq;
    const int qp = a.n_qp - 1 - (int)(blockIdx.x / per_qp);
    const int rem = (int)(blockIdx.x % per_qp);
    const int r = rem / a.Hq, hq = rem % a.Hq, hkv = hq / a.G;
    const int i0 = qp * kQT * kQB;

    if (threadIdx.x == 0) {
        // one arrival (an expect-tx arrival or a tcgen05.commit) per phase,
        // except that all four warps of a Q tile publish its P
        for (int b = 0; b < kNumBars; ++b) {
            const bool per_warp = &bars[b] >= p_full && &bars[b] < o_done;
            mbar_init(&bars[b], per_warp ? 4 : 1);
        }
        *abort = 0;
        fence_barrier_init();
        prefetch_tensormap(&tq);
        prefetch_tensormap(&tk);
        prefetch_tensormap(&tv);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dependency_wait();  // Q, the caches and the lengths may come from the previous kernel

    int L = __ldg(a.seqlens + r);
    if (L < 0 || L > a.max_pages * kTile) {
        if (threadIdx.x == 0 && a.flags && hq == 0 && qp == a.n_qp - 1)
            atomicOr(a.flags, (int)HPC_FLAG_BAD_SEQLEN);
        L = min(max(L, 0), a.max_pages * kTile);
    }
    QTile qt[kQT];
#pragma unroll
    for (int x = 0; x < kQT; ++x) qt[x] = qtile(i0 + x * kQB, L, a.q_len);
    int n = 0;  // KV tiles the CTA reads
#pragma unroll
    for (int x = 0; x < kQT; ++x) n = max(n, qt[x].tiles);
    const int np = (L + kTile - 1) / kTile;  // pages of the request
    const bool tail = n > 0 && n * kKB > L;   // the last tile holds slots past L_r

    bool ok = true;
    int q_issued = 0, k_issued[kKStages] = {}, v_issued[kVStages] = {};

    if (warp == kProducerWarp) {
        const uint64_t pol = policy_evict_normal();
        if (lane == 0 && n > 0) {
            uint32_t bytes = 0;
#pragma unroll
            for (int x = 0; x < kQT; ++x) bytes += qt[x].tiles > 0 ? kTileBytes : 0;
            mbar_arrive_expect_tx(q_full, bytes);
#pragma unroll
            for (int x = 0; x < kQT; ++x)
                if (qt[x].tiles > 0)
                    for (int h = 0; h < 2; ++h)
                        tma_load_4d(smem + kOffQ + x * kTileBytes + h * kHalf, &tq, q_full, 0, h,
                                    hq, r * a.q_len + qt[x].first, pol);
            q_issued = 1;
        }
        const int32_t *bt = a.block_table + (size_t)r * a.max_pages;
        int pg = -1;
        for (int j = 0; j < n; ++j) {
            if ((j & 15) == 0) {  // the page numbers of 16 tiles, one per lane
                const int idx = 2 * j + lane;
                pg = idx < np ? __ldg(bt + idx) : -1;
            }
            const int p0 = __shfl_sync(0xffffffffu, pg, (2 * j) & 31);
            const int p1 = __shfl_sync(0xffffffffu, pg, (2 * j + 1) & 31);
            int good = 1;
            if (lane == 0) {
                const bool has1 = 2 * j + 1 < np;
                const bool l0 = p0 >= 0 && p0 < a.num_pages;
                const bool l1 = has1 && p1 >= 0 && p1 < a.num_pages;
                if ((!l0 || (has1 && !l1)) && a.flags) atomicOr(a.flags, (int)HPC_FLAG_BAD_PAGE);
                const uint32_t bytes = (uint32_t)((l0 ? 1 : 0) + (l1 ? 1 : 0)) * 2 * kTile * 128;
                for (int kv = 0; kv < 2 && good; ++kv) {
                    const int st = kv == 0 ? kKStages : kVStages, s = j % st;
                    const uint32_t par = ((j / st) & 1u) ^ 1u;
                    uint64_t *full = kv == 0 ? &k_full[s] : &v_full[s];
                    if (!mbar_wait(kv == 0 ? &k_empty[s] : &v_empty[s], par, abort)) {
                        good = 0;
                        break;
                    }
                    if (bytes == 0) {
                        mbar_arrive(full);
                    } else {
                        mbar_arrive_expect_tx(full, bytes);
                        const CUtensorMap *map = kv == 0 ? &tk : &tv;
                        uint8_t *dst = smem + (kv == 0 ? kOffK : kOffV) + s * kTileBytes;
                        for (int h = 0; h < 2; ++h) {
                            if (l0) tma_load_5d(dst + h * kHalf, map, full, 0, h, hkv, 0, p0, pol);
                            if (l1)
                                tma_load_5d(dst + h * kHalf + kTile * 128, map, full, 0, h, hkv, 0,
                                            p1, pol);
                        }
                    }
                    ++(kv == 0 ? k_issued[s] : v_issued[s]);
                }
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
                ok = false;
                break;
            }
        }
        if (ok && tail) {
            // tokens past L_r (the last page's free slots, or a page the
            // request does not have) must not reach P V: once the last V
            // tile has landed, zero those rows of both column blocks
            const int jl = n - 1, s = jl % kVStages;
            if (!warp_wait(&v_full[s], (jl / kVStages) & 1u, abort)) {
                ok = false;
            } else {
                uint8_t *vs = smem + kOffV + s * kTileBytes;
                const int z0 = L - jl * kKB;
                for (int h = 0; h < 2; ++h)
                    for (int e = z0 * 8 + lane; e < kKB * 8; e += 32)
                        sts128(smem_u32(vs + h * kHalf + e * 16), 0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(v_tail);
            }
        }
    } else if (warp == kMmaWarp) {
        const uint32_t idesc_s = idesc_bf16_f32(kQB, kKB);
        const uint32_t idesc_o = idesc_bf16_f32_bmn(kQB, kHeadDim);
        // descriptor bases: the K-step offsets below are compile-time
        // additions to the start-address field (addresses stay < 256 KB)
        const uint64_t dq0 = smem_desc_k128(smem_u32(smem + kOffQ));
        const uint64_t dk0 = smem_desc_k128(smem_u32(smem + kOffK));
        const uint64_t dv0 = smem_desc_mn128(smem_u32(smem + kOffV), kHalf);
        // S_x = Q_x K^T into x's score columns (K tile in stage s)
        auto issue_s = [&](int x, int s) {
            const uint64_t dq = dq0 + (uint64_t)((x * kTileBytes) >> 4);
            const uint64_t dk = dk0 + (uint64_t)((s * kTileBytes) >> 4);
#pragma unroll
            for (int k = 0; k < kHeadDim / 16; ++k) {
                const uint32_t off = ((k >> 2) * kHalf + (k & 3) * 32) >> 4;
                umma_bf16(tmem + 128 * x, dq + off, dk + off, idesc_s, k > 0);
            }
            umma_commit(&s_full[x]);
        };
        // O_x += P_x V (V tile in stage s), P_x from TMEM
        auto issue_pv = [&](int x, int s, bool acc) {
            const uint64_t dv = dv0 + (uint64_t)((s * kTileBytes) >> 4);
#pragma unroll
            for (int k = 0; k < kKB / 16; ++k)
                umma_bf16_ts(tmem + kOCol + 128 * x, tmem + 128 * x + 8 * k,
                             dv + (uint64_t)((k * 16 * 128) >> 4), idesc_o, acc || k > 0);
            umma_commit(&o_done[x]);
        };
        // one thread issues everything; every wait is its own (bounded)
        if (lane == 0) {
            if (n > 0) {
                ok = mbar_wait(q_full, 0, abort) && mbar_wait(&k_full[0], 0, abort);
                if (ok) {
                    tc_fence_after();
                    for (int x = 0; x < kQT; ++x)
                        if (qt[x].tiles > 0) issue_s(x, 0);
                    umma_commit(&k_empty[0]);
                }
            }
            for (int j = 0; ok && j < n; ++j) {
                const int s = j % kVStages, s1 = (j + 1) % kKStages;
                const bool next = j + 1 < n;
                ok = (j == n - 1 && tail) ? mbar_wait(v_tail, 0, abort)
                                          : mbar_wait(&v_full[s], (j / kVStages) & 1u, abort);
                if (ok && next) ok = mbar_wait(&k_full[s1], ((j + 1) / kKStages) & 1u, abort);
                for (int x = 0; x < kQT && ok; ++x) {
                    if (j >= qt[x].tiles) continue;
                    ok = mbar_wait(&p_full[x], j & 1u, abort);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(x, s, j > 0);
                    if (j + 1 < qt[x].tiles) issue_s(x, s1);
                }
                if (!ok) break;
                umma_commit(&v_empty[s]);             // after both Q tiles' products with V_j
                if (next) umma_commit(&k_empty[s1]);  // after both Q tiles' scores with K_j+1
            }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        // arrives once every MMA issued has completed (TMEM is freed after it)
        if (lane == 0) umma_commit(mma_done);
    } else {
        // softmax of Q tile x: thread = one query row, warp w reads TMEM
        // lanes 32 (w mod 4) ..
        const int x = warp >> 2, q4 = warp & 3;
        const QTile t = qt[x];
        const int rho = 32 * q4 + lane, i = t.first + rho;
        const int lim = min(L - a.q_len + i, L - 1);
        const uint32_t row = tmem + ((uint32_t)(32 * q4) << 16);
        const uint32_t scol = row + 128 * x, ocol = row + kOCol + 128 * x;
        const float sc = a.score_scale;
        float m_ref = -INFINITY, l = 0.f;
        for (int j = 0; j < t.tiles; ++j) {
            if (!warp_wait(&s_full[x], j & 1u, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // the row's 128 scores in two halves: the second half loads while
            // the first is masked and reduced
            uint32_t ra[32], rb[32], rc[32], rd[32];
            tmem_ld32_nowait(scol, ra);
            tmem_ld32_nowait(scol + 32, rb);
            tmem_wait_ld32x2(ra, rb);
            tmem_ld32_nowait(scol + 64, rc);
            tmem_ld32_nowait(scol + 96, rd);
            float s[128];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                s[c] = __uint_as_float(ra[c]);
                s[32 + c] = __uint_as_float(rb[c]);
            }
            const bool diag = j * kKB + kKB - 1 > t.lim_first;  // the causal diagonal or the end
            if (diag) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (j * kKB + c > lim) s[c] = -INFINITY;
            }
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 32; ++c) mx4[c & 3] = fmax3(mx4[c & 3], s[2 * c], s[2 * c + 1]);
            tmem_wait_ld32x2(rc, rd);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                s[64 + c] = __uint_as_float(rc[c]);
                s[96 + c] = __uint_as_float(rd[c]);
            }
            if (diag) {
#pragma unroll
                for (int c = 64; c < 128; ++c)
                    if (j * kKB + c > lim) s[c] = -INFINITY;
            }
#pragma unroll
            for (int c = 32; c < 64; ++c) mx4[c & 3] = fmax3(mx4[c & 3], s[2 * c], s[2 * c + 1]);
            const float mx = fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
            const float m_tile = mx * sc;
            const bool need = m_tile > m_ref + kRescaleLog2;
            const float new_ref = need ? m_tile : m_ref;
            const float factor = need ? ex2(m_ref - new_ref) : 1.f;
            const float base = new_ref == -INFINITY ? 0.f : new_ref;
            // P as packed BF16 pairs, written over the first 64 score columns
            // in two stores: the first is in flight while the second half is
            // computed
            uint32_t pa[32], pb[32];
            float2 ps[4] = {};
            const float2 sc2 = make_float2(sc, sc), nb2 = make_float2(-base, -base);
#pragma unroll
            for (int c = 0; c < 32; ++c) {  // paired FP32 arithmetic: two columns per instruction
                const float2 e = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), sc2, nb2);
                const float p0 = ex2(e.x), p1 = ex2(e.y);
                ps[c & 3] = __fadd2_rn(ps[c & 3], make_float2(p0, p1));
                pa[c] = pack_bf16x2(p0, p1);
            }
            tmem_st32_nowait(scol, pa);
#pragma unroll
            for (int c = 32; c < 64; ++c) {
                const float2 e = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), sc2, nb2);
                const float p0 = ex2(e.x), p1 = ex2(e.y);
                ps[c & 3] = __fadd2_rn(ps[c & 3], make_float2(p0, p1));
                pb[c - 32] = pack_bf16x2(p0, p1);
            }
            const float2 pq = __fadd2_rn(__fadd2_rn(ps[0], ps[1]), __fadd2_rn(ps[2], ps[3]));
            l = l * factor + (pq.x + pq.y);
            // O_x is settled: its product with the previous tile completed
            // before these scores did
            if (j >= 1 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float o[64];
                    tmem_ld32x2(ocol + 64 * hf, ocol + 64 * hf + 32, o);
#pragma unroll
                    for (int c = 0; c < 64; ++c) o[c] *= factor;
                    tmem_st32x2(ocol + 64 * hf, ocol + 64 * hf + 32, o);
                }
            }
            tmem_st32_nowait(scol + 32, pb);
            tmem_wait_st32x2(pa, pb);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
            m_ref = new_ref;
        }
        // epilogue: O / l as BF16
        bool have = ok && t.tiles > 0;
        if (have) {
            if (!warp_wait(&o_done[x], (t.tiles - 1) & 1u, abort))
                ok = have = false;
            else
                tc_fence_after();
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const bool store = ok && i < a.q_len;
        uint4 *dst = reinterpret_cast<uint4 *>(
            a.out + ((size_t)(r * a.q_len + min(i, a.q_len - 1)) * a.Hq + hq) * kHeadDim);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float o[64];
            if (have) {
                tmem_ld32x2(ocol + 64 * hf, ocol + 64 * hf + 32, o);
#pragma unroll
                for (int c = 0; c < 64; ++c) o[c] *= inv;
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) o[c] = 0.f;
            }
            if (store && !*abort) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    dst[8 * hf + u] = make_uint4(pack_bf16x2(o[8 * u], o[8 * u + 1]),
                                                 pack_bf16x2(o[8 * u + 2], o[8 * u + 3]),
                                                 pack_bf16x2(o[8 * u + 4], o[8 * u + 5]),
                                                 pack_bf16x2(o[8 * u + 6], o[8 * u + 7]));
            }
        }
    }

    if (!ok || *abort) {
        if (a.flags && lane == 0) atomicOr(a.flags, (int)HPC_FLAG_TIMEOUT);
        // no copy may land after the CTA has left: wait (bounded) for the last
        // copy issued into each buffer
        if (warp == kProducerWarp && lane == 0) {
            auto drain = [](uint64_t *bar, int issued) {
                if (issued == 0) return;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar, (uint32_t)(issued - 1) & 1u) &&
                       globaltimer_ns() - t0 < 1000000000ull) {
                }
            };
            drain(q_full, q_issued);
            for (int s = 0; s < kKStages; ++s) drain(&k_full[s], k_issued[s]);
            for (int s = 0; s < kVStages; ++s) drain(&v_full[s], v_issued[s]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        // no MMA may still write TMEM when it is freed (bounded, like every wait)
        if (lane == 0) {
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, &no_abort);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

std::atomic<unsigned> g_prefill_attr_done{0};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor map over Q [B * q_len, Hq, 128] BF16 as {64 dims, 2 halves, Hq,
// tokens}, box {64, 1, 1, 128}: one 64-dim half of 128 consecutive query
// tokens of one head, rows of 128 bytes (the swizzle span).
hpc_status make_q_map(CUtensorMap *m, const void *q, int64_t tokens, int32_t Hq) {
    auto encode = tensor_map_encoder();
    if (!encode) return HPC_ERR_CUDA;
    std::memset(m, 0, sizeof(*m));
    cuuint64_t dims[4] = {64, 2, (cuuint64_t)Hq, (cuuint64_t)tokens};
    cuuint64_t strides[3] = {128, 256, (cuuint64_t)Hq * 256};
    cuuint32_t box[4] = {64, 1, 1, kQB};
    cuuint32_t elem[4] = {1, 1, 1, 1};
    CUresult res = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(q), dims,
                          strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? HPC_OK : HPC_ERR_CUDA;
}

}  // namespace
}  // namespace hpc

using namespace hpc;

extern "C" hpc_status hpc_prefill_attn(const void *d_q, const void *d_k_cache,
                                       const void *d_v_cache, int32_t num_pages,
                                       const int32_t *d_block_table, int32_t max_pages_per_req,
                                       const int32_t *d_seqlens, int32_t B, int32_t Hq,
                                       int32_t Hkv, int32_t head_dim, int32_t q_len,
                                       float sm_scale, void *d_out, int32_t *d_flags,
                                       hpc_stream_t stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || max_pages_per_req <= 0 || q_len < 1 || num_pages <= 0)
        return HPC_ERR_ARG;
    if (head_dim != HPC_HEAD_DIM || Hq % Hkv != 0) return HPC_ERR_UNSUPPORTED;
    if (!std::isfinite(sm_scale)) return HPC_ERR_ARG;
    if (B == 0) return HPC_OK;
    if (!d_q || !d_k_cache || !d_v_cache || !d_block_table || !d_seqlens || !d_out)
        return HPC_ERR_ARG;
    if (!aligned16(d_q) || !aligned16(d_k_cache) || !aligned16(d_v_cache) || !aligned16(d_out))
        return HPC_ERR_ARG;
    const int64_t n_qp = (q_len + kQT * kQB - 1) / (kQT * kQB);
    const int64_t grid = n_qp * B * Hq;
    if (grid >= ((int64_t)1 << 31) || (int64_t)B * q_len >= ((int64_t)1 << 31) ||
        (int64_t)max_pages_per_req * HPC_PAGE_SIZE >= ((int64_t)1 << 30))
        return HPC_ERR_UNSUPPORTED;

    CUtensorMap tq, tk, tv;
    hpc_status st = make_q_map(&tq, d_q, (int64_t)B * q_len, Hq);
    if (st == HPC_OK) st = cache_tensor_map(&tk, d_k_cache, num_pages, Hkv, false);
    if (st == HPC_OK) st = cache_tensor_map(&tv, d_v_cache, num_pages, Hkv, false);
    if (st != HPC_OK) return st;

    PrefillArgs a;
    a.seqlens = d_seqlens;
    a.block_table = d_block_table;
    a.out = static_cast<__nv_bfloat16 *>(d_out);
    a.flags = d_flags;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.q_len = q_len;
    a.max_pages = max_pages_per_req;
    a.num_pages = num_pages;
    a.n_qp = (int)n_qp;
    a.score_scale = sm_scale * 1.4426950408889634f;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HPC_ERR_CUDA;
    const unsigned bit = 1u << (dev & 31);
    if (!(g_prefill_attr_done.load() & bit)) {
        if (cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess)
            return HPC_ERR_CUDA;
        g_prefill_attr_done.fetch_or(bit);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_attn_kernel, tq, tk, tv, a);
    return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}
