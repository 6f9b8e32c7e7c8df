// Persistent load-balanced paged GQA decode attention (HPC-Ops vLLM post,
// "Compute and combine" bullet; SGLang post, 围绕Live KV Work的调度,
// execution paragraph): the persistent CTAs drain the bins of the task map.
// For every descriptor (h, r, tb, te) a CTA streams KV pages
// block_table[r][tb .. te) of KV head h and produces, for the GQA group of
// h, the normalised partial output and its log-sum-exp (split-buffer slot =
// descriptor index).  In the fused mode it also performs the combine step: a
// unit with one chunk writes its BF16 output directly, and for a split unit
// the CTA that counts the unit's last chunk merges all of its partials.
//
// GB300 design (the pages' Hopper kernel is not followed):
//  * warp 0 is a producer: one lane walks the CTA's bins as a flat stream of
//    tiles and issues TMA tile loads (one per 64-token page of K and of V)
//    into a STAGES-deep ring of shared-memory stages guarded by full/empty
//    mbarriers, so loads keep flowing across descriptor boundaries.  A stage
//    holds TPS tiles of one descriptor.  Q (and the FP8 q-scales) ride in the
//    stage holding a descriptor's first tile.  After the last tile the
//    producer posts a terminator stage.
//  * 4 * TPS consumer warps (warps 2 ..): warp w owns tokens 16 (w % 4) ..
//    + 15 of tile w / 4 of every stage and keeps its own online-softmax
//    state.  At a descriptor's end each consumer hands its state to a
//    shared-memory slot (double-buffered where the layout fits) and goes
//    straight on with the next stage; it never waits for the merge.
//  * warp 1 is a combiner: it merges the consumers' states of each finished
//    descriptor, writes the BF16 output or the partial and its LSE, and counts
//    the chunks of split units at once, so no consumer ever waits on that
//    bookkeeping.  The merges of split units whose last chunk this CTA counts
//    run at the end, spread over all warps.
//  * contractions run on mma.sync with the operands swapped so the GQA group
//    is the N = 8 side:  S^T[tok, head] = K[tok, :] . Q^T and
//    O^T[dim, head] += V^T[dim, tok] . P^T[tok, head].  P^T's B fragment is
//    the S^T accumulator transposed in registers with movmatrix, so there is
//    no shared-memory round trip and no padding of the 8-head group to M = 16.
//  * BF16: K via ldmatrix, V via ldmatrix.trans, bf16 MMAs.
//    FP8: Q.K^T on e4m3 MMAs (m16n8k32) straight from the FP8 Q and cache;
//    V is widened exactly to f16 in registers (byte permutes + cvt) with the
//    output dims permuted so each lane needs one 16-byte row segment per
//    token; P stays f16 (never quantised).
//  * tiles land with the 128-byte swizzle; every ldmatrix / 16-byte read
//    touches 8 distinct 16-byte bank groups, and the state hand-off is
//    lane-major, so it is conflict-free too.
//  * multi-query decode (q_len > 1, the speculative / MTP layer): a
//    descriptor serves R = q_len * G query rows (rho = i * G + g) of its KV
//    head; NB = ceil(R / 8) blocks of 8 rows are the N side of the MMAs, so
//    every K/V fragment feeds NB MMAs and each KV tile is read once for all
//    rows.  Query token i sees tokens below L - q_len + 1 + i (per-column
//    limits in the softmax); NB = 1, q_len = 1 is plain decode.
//  * the kernel is launched as a programmatic dependent of the assign kernel:
//    it sets up its barriers, prefetches the block table into L2, derives its
//    first descriptor from the sequence lengths and starts streaming while
//    the assign kernel may still be running; only the producer waits for the
//    task map, when it first needs it.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace hpc {

struct StageInfo {
    int kv_head, req, tile0, ntiles;  // tiles tile0 .. tile0 + ntiles - 1 of request req
    int flags, seqlen, desc_idx, count;  // count: chunks of the unit
    int chunk_off, pad0, pad1, pad2;
    int pad3[4];
    float qscale[kMaxRows];  // FP8: scale of query row rho
};
static_assert(sizeof(StageInfo) == 128, "StageInfo layout");

// The fields of a descriptor the combine step needs.
struct DescInfo {
    int req, kv_head, desc_idx, count, chunk_off;
};

struct SlotInfo {  // what a consumer hand-off slot holds besides the states
    DescInfo di;
    int flags, pad0, pad1;
};
static_assert(sizeof(SlotInfo) == 32, "SlotInfo layout");

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kStateRegs = 36;  // per lane and row block: 32 accumulators, m0, m1, l0, l1
constexpr int kMaxLast = 16;    // split units whose merge this CTA owes, held at once
constexpr int kStageStride = kHeadDim + 4;  // floats per head row of the combiner's staging
constexpr int kFlyMaxBatch = 1024;  // largest batch whose first descriptor is derived in-kernel
constexpr int kWalkMaxBatch = 64;   // largest batch whose first bin is walked in-kernel
constexpr int kWalkTiles = 8;       // tiles streamed on derived descriptors before the map is read

// Warp-uniform bounded wait: every lane polls the phase (so each lane
// acquires the data the phase guards) and the lanes agree on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return mbar_wait_warp(bar, parity, abort);
}

template <bool FP8, int STAGES, int TPS, int NB>
struct AttnTraits {
    static constexpr int kConsumers = kConsumerWarps * TPS;          // consumer warps
    static constexpr int kThreads = 32 * (2 + kConsumers);           // + producer, combiner
    static constexpr int kElem = FP8 ? 1 : 2;
    static constexpr int kTileBytes = kTile * kHeadDim * kElem;     // one K or V page, one head
    static constexpr int kHalfBytes = kTile * 64 * 2;               // BF16: one 64-dim half
    static constexpr int kStageKV = TPS * kTileBytes;               // K (or V) bytes per stage
    static constexpr int kRows = 8 * NB;                             // query rows held per stage
    static constexpr int kQBytes = kRows * kHeadDim * kElem;        // Q slot per stage
    static constexpr int kState = kStateRegs * NB;                   // state floats per lane
    static constexpr int kSlotFloats = kConsumers * kState * 32;     // one hand-off slot
    // Shared memory of the layout below with `slots` hand-off slots.
    static constexpr int bytes_with(int slots) {
        return 2 * STAGES * kStageKV + STAGES * kQBytes + STAGES * (int)sizeof(StageInfo) +
               slots * kSlotFloats * 4 + kRows * kStageStride * 4 +
               slots * (int)sizeof(SlotInfo) + (kMaxLast + 1) * (int)sizeof(SlotInfo) +
               (2 * STAGES + 2 * slots + 1) * 8 + 16 + 1024;
    }
    // consumer -> combiner hand-off slots: double-buffered when that fits
    // (two row blocks double the state a slot holds)
    static constexpr int kSlots = bytes_with(2) <= 227 * 1024 ? 2 : 1;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + STAGES * kStageKV;
    static constexpr int kOffQ = kOffV + STAGES * kStageKV;
    static constexpr int kOffInfo = kOffQ + STAGES * kQBytes;
    static constexpr int kOffComb = kOffInfo + STAGES * (int)sizeof(StageInfo);
    static constexpr int kOffStage = kOffComb + kSlots * kSlotFloats * 4;
    static constexpr int kOffSlotInfo = kOffStage + kRows * kStageStride * 4;
    static constexpr int kOffLast = kOffSlotInfo + kSlots * (int)sizeof(SlotInfo);
    static constexpr int kOffBar = kOffLast + (kMaxLast + 1) * (int)sizeof(SlotInfo);
    // full[STAGES], empty[STAGES], slot full[2], slot empty[2], end rendezvous
    static constexpr int kNumBars = 2 * STAGES + 2 * kSlots + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // abort word
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kSmemBytes = kBytes + 1024;  // slack to align the base to 1024 B
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// ------------------------------------------------------------------ producer
// Shared state of the producer warp.
struct ProducerState {
    uint32_t it;          // stages issued so far
    bool waited;          // grid_dependency_wait done: the task map may be read
    unsigned late_flags;  // device error bits, OR-ed into meta[3] after the wait
};

__device__ __forceinline__ void wait_for_map(ProducerState &ps) {
    if (!ps.waited) {
        grid_dependency_wait();
        ps.waited = true;
    }
}

// First descriptor of bin c, from the sequence lengths alone (the closed form
// of the assign kernel: n_r = ceil(L_r / 64) with the same clamping, T =
// Hkv * sum n_r, budget = max(ceil(T / bins), floor, 1), bin c = global tiles
// [c * budget, ...), units head-major).  Returns false when the batch is too
// large to scan here; te == tb means the bin is empty.
__device__ __forceinline__ bool first_descriptor(const AttnParams &p, int c, int &h, int &r,
                                                 int &tb, int &te) {
    if (p.B > kFlyMaxBatch) return false;
    const int lane = threadIdx.x & 31, cap = p.max_pages * kTile;
    int N = 0;
    for (int base = 0; base < p.B; base += 32) {
        const int rr = base + lane;
        int L = rr < p.B ? p.seqlens[rr] : 0;
        L = L < 0 ? 0 : min(L, cap);
        N += __reduce_add_sync(kFullMask, (L + kTile - 1) / kTile);
    }
    const long long T = (long long)p.Hkv * N;
    const int budget = (int)max((T + p.num_bins - 1) / p.num_bins, (long long)max(p.min_tiles, 1));
    const long long t = (long long)c * budget;
    h = r = tb = te = 0;
    if (t >= T) return true;  // an empty bin
    h = (int)(t / N);
    const int tl = (int)(t - (long long)h * N);
    int carry = 0;
    for (int base = 0; base < p.B; base += 32) {
        const int rr = base + lane;
        int L = rr < p.B ? p.seqlens[rr] : 0;
        L = L < 0 ? 0 : min(L, cap);
        const int n = (L + kTile - 1) / kTile;
        int incl = n;  // inclusive prefix of n over this chunk
#pragma unroll
        for (int o_ = 1; o_ < 32; o_ <<= 1) {
            const int y = __shfl_up_sync(kFullMask, incl, o_);
            if (lane >= o_) incl += y;
        }
        const unsigned hit = __ballot_sync(kFullMask, rr < p.B && carry + incl > tl);
        if (hit) {  // the request holding global tile t
            const int l = __ffs(hit) - 1;
            const int start = carry + __shfl_sync(kFullMask, incl - n, l);
            const int nr = __shfl_sync(kFullMask, n, l);
            r = base + l;
            tb = tl - start;
            te = tb + (int)min((long long)(nr - tb), T - t < budget ? T - t : (long long)budget);
            return true;
        }
        carry += __shfl_sync(kFullMask, incl, 31);
    }
    return true;  // unreachable for a consistent batch
}

// The descriptors of bin c from the sequence lengths alone, for batches of up
// to 64 requests (tile counts held in two registers per lane): the closed form
// of the assign kernel walked unit by unit.  Used by CTAs whose first
// descriptors are short, so that they need not wait for the assign kernel's
// map before streaming (its writes become visible to this grid only a few
// microseconds after that kernel ends).
struct FlyWalk {
    int n0, n1;      // tiles of requests lane and lane + 32
    int N, budget;   // tiles per KV head, tiles per bin
    long long end;   // global tile where bin c ends
    int c, k;        // the bin; descriptors produced so far
    int base;        // index of the bin's first descriptor in the map (-1 until needed)
    int h, r, pre;   // current unit, tiles of the requests before r
    long long t;     // global tile at the current descriptor's start
    int tb, te;      // the current descriptor: tiles [tb, te) of unit (h, r); te == tb: done
};

__device__ __forceinline__ int walk_tiles(const FlyWalk &w, int r) {
    return __shfl_sync(kFullMask, r < 32 ? w.n0 : w.n1, r & 31);
}

// Index in the map of bin c's first descriptor: every bin before c holds one
// descriptor plus one per unit with tiles starting strictly inside it.
__device__ __forceinline__ void walk_base(const AttnParams &p, FlyWalk &w) {
    const int lane = threadIdx.x & 31;
    int i0 = w.n0, i1 = w.n1;
#pragma unroll
    for (int o_ = 1; o_ < 32; o_ <<= 1) {
        const int y0 = __shfl_up_sync(kFullMask, i0, o_), y1 = __shfl_up_sync(kFullMask, i1, o_);
        if (lane >= o_) i0 += y0, i1 += y1;
    }
    i1 += __shfl_sync(kFullMask, i0, 31);
    const int e0 = i0 - w.n0, e1 = i1 - w.n1;  // exclusive prefixes
    const bool a0 = lane < p.B && w.n0 > 0, a1 = lane + 32 < p.B && w.n1 > 0;
    const long long X = (long long)w.c * w.budget;  // < T: at most Hkv heads below
    int inner = 0;
    if (X <= 0x7FFFFFFFll) {
        // the starts h N + e of each head, their residues mod budget
        // carried from head to head (one add and compare each): few
        // instructions, as this runs before the CTA's first copy
        const unsigned Xu = (unsigned)X, b = (unsigned)w.budget, N = (unsigned)w.N;
        const unsigned Nm = N % b;
        unsigned m0 = (unsigned)e0 % b, m1 = (unsigned)e1 % b;
        int cnt = 0;
        for (unsigned hN = 0; hN < Xu; hN += N) {
            cnt += (a0 && hN + e0 < Xu && m0 != 0) + (a1 && hN + e1 < Xu && m1 != 0);
            m0 += Nm;
            m0 -= m0 >= b ? b : 0u;
            m1 += Nm;
            m1 -= m1 >= b ? b : 0u;
        }
        inner = __reduce_add_sync(kFullMask, cnt);
    } else {
        for (long long hN = 0; hN < X; hN += w.N) {
            const long long s0 = hN + e0, s1 = hN + e1;
            inner += __popc(__ballot_sync(kFullMask, a0 && s0 < X && s0 % w.budget != 0)) +
                     __popc(__ballot_sync(kFullMask, a1 && s1 < X && s1 % w.budget != 0));
        }
    }
    w.base = w.c + inner;
}

__device__ __forceinline__ void walk_init(const AttnParams &p, int c, FlyWalk &w) {
    const int lane = threadIdx.x & 31, cap = p.max_pages * kTile;
    int L0 = lane < p.B ? p.seqlens[lane] : 0;
    int L1 = lane + 32 < p.B ? p.seqlens[lane + 32] : 0;
    L0 = L0 < 0 ? 0 : min(L0, cap);
    L1 = L1 < 0 ? 0 : min(L1, cap);
    w.n0 = (L0 + kTile - 1) / kTile;
    w.n1 = (L1 + kTile - 1) / kTile;
    w.N = __reduce_add_sync(kFullMask, w.n0 + w.n1);
    const long long T = (long long)p.Hkv * w.N;
    w.budget = (int)max((T + p.num_bins - 1) / p.num_bins, (long long)max(p.min_tiles, 1));
    w.c = c;
    w.k = 0;
    w.base = -1;
    w.t = (long long)c * w.budget;
    w.end = min(w.t + w.budget, T);
    w.h = w.r = w.pre = w.tb = w.te = 0;
    if (w.t >= T) return;  // an empty bin
    w.h = (int)(w.t / w.N);
    const int tl = (int)(w.t - (long long)w.h * w.N);
    // the request holding tile tl of head h: inclusive prefix over both halves
    int i0 = w.n0, i1 = w.n1;
#pragma unroll
    for (int o_ = 1; o_ < 32; o_ <<= 1) {
        const int y0 = __shfl_up_sync(kFullMask, i0, o_), y1 = __shfl_up_sync(kFullMask, i1, o_);
        if (lane >= o_) i0 += y0, i1 += y1;
    }
    i1 += __shfl_sync(kFullMask, i0, 31);
    const unsigned h0 = __ballot_sync(kFullMask, lane < p.B && i0 > tl);
    const unsigned h1 = __ballot_sync(kFullMask, lane + 32 < p.B && i1 > tl);
    const int l = h0 ? __ffs(h0) - 1 : 32 + __ffs(h1) - 1;
    w.r = l;
    const int incl = __shfl_sync(kFullMask, l < 32 ? i0 : i1, l & 31);
    const int n = walk_tiles(w, l);
    w.pre = incl - n;
    w.tb = tl - w.pre;
    w.te = w.tb + (int)min((long long)(n - w.tb), w.end - w.t);
    if (w.te - w.tb < kWalkTiles) walk_base(p, w);  // its layout is derived: index the bin now
}

// The next descriptor of the bin (te == tb once the bin is done).
__device__ __forceinline__ void walk_next(const AttnParams &p, FlyWalk &w) {
    w.t += w.te - w.tb;
    ++w.k;
    if (w.t >= w.end) {
        w.tb = w.te = 0;
        return;
    }
    int n = walk_tiles(w, w.r);
    do {  // the next unit with tiles (one exists: the bin has tiles left)
        w.pre += n;
        if (++w.r == p.B) w.r = 0, w.pre = 0, ++w.h;
        n = walk_tiles(w, w.r);
    } while (n == 0);
    w.tb = 0;
    w.te = (int)min((long long)n, w.end - w.t);
}

// The chunk layout of the current descriptor.  Every bin before c holds one
// descriptor plus one per unit with tiles starting strictly inside it, so the
// bin's first descriptor has index c + #{such unit starts before tile c *
// budget}; a unit spans bins first .. last (its chunks, consecutive in the
// map), and its descriptor in bin c is chunk c - first.
__device__ __forceinline__ void walk_chunk(const AttnParams &p, FlyWalk &w, int &idx, int &count,
                                           int &off) {
    if (w.base < 0) walk_base(p, w);
    const long long s = (long long)w.h * w.N + w.pre;
    const int n = walk_tiles(w, w.r);
    int first, last;
    if (s + n <= 0x7FFFFFFFll) {
        first = (int)((unsigned)s / (unsigned)w.budget);
        last = (int)((unsigned)(s + n - 1) / (unsigned)w.budget);
    } else {
        first = (int)(s / w.budget);
        last = (int)((s + n - 1) / w.budget);
    }
    idx = w.base + w.k;
    count = last - first + 1;
    off = idx - (w.c - first);
}

// Streams one descriptor (h, r, tb, te) through the stage ring.  desc_idx is
// its index in the task map, or -1 when it was derived before the map could
// be read, as the k-th descriptor of bin `bin`: its chunk layout then comes
// from `walk` (non-null: derived, a few instructions) or from the map, in
// which case its last stage's copies are issued before the map is waited for
// (the stage is released once the layout is written), so the wait overlaps
// the stage's transfer.  Returns false after a timeout.
template <bool FP8, int STAGES, int TPS, int NB>
__device__ __forceinline__ bool stream_desc(const CUtensorMap *tmap_k, const CUtensorMap *tmap_v,
                                            const AttnParams &p, uint8_t *smem, int h, int r,
                                            int tb, int te, int desc_idx, int bin,
                                            FlyWalk *walk, int bin_pos, ProducerState &ps,
                                            uint64_t policy, volatile int *abort) {
    using Tr = AttnTraits<FP8, STAGES, TPS, NB>;
    const int lane = threadIdx.x & 31;
    StageInfo *info = reinterpret_cast<StageInfo *>(smem + Tr::kOffInfo);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Tr::kOffBar);
    uint64_t *empty = full + STAGES;
    // Q: the G heads of KV head h for each of the q_len query tokens, stacked
    // as rows rho = i * G + g (one bulk copy per query token)
    const uint32_t q_group = (uint32_t)(p.G * kHeadDim * Tr::kElem);
    const uint32_t q_bytes = q_group * (uint32_t)p.q_len;
    const size_t q_token_stride = (size_t)p.Hq * kHeadDim * Tr::kElem;
    if (tb >= te) return true;  // empty split of the static schedule
    const int L = p.seqlens[r];
    const int u = h * p.B + r;
    float qs = 1.f;
    if (FP8 && lane < p.R) {
        const int i = lane / p.G;
        qs = p.q_scale[((size_t)r * p.q_len + i) * p.Hq + h * p.G + (lane - i * p.G)];
    }
    const int32_t *bt_row = p.block_table + (size_t)r * p.max_pages;
    const uint8_t *q_src = static_cast<const uint8_t *>(p.q) +
                           ((size_t)r * p.q_len * p.Hq + (size_t)h * p.G) * kHeadDim * Tr::kElem;
    // the first 32 block-table entries are requested with the q-scales, so
    // the two loads share one round trip; the q-scales (FP8) are broadcast
    // only after the first stage's copies are issued: the consumers need
    // them once the stage has landed, so their load (from DRAM after a
    // flush, where the block table is warm in L2) does not hold up the copies
    int page0 = 0;
    if (lane < min(32, te - tb)) page0 = bt_row[tb + lane];
    float qsg[Tr::kRows];
#pragma unroll
    for (int g = 0; g < Tr::kRows; ++g) qsg[g] = 1.f;
    bool late_q = FP8;  // the q-scales are not broadcast yet

    for (int t0 = tb; t0 < te; t0 += 32) {  // 32 block-table entries at a time
        const int nt = min(32, te - t0);
        int page = 0;
        if (lane < nt) {
            page = t0 == tb ? page0 : bt_row[t0 + lane];
            if (page < 0 || page >= p.num_pages) {
                ps.late_flags |= HPC_FLAG_BAD_PAGE;
                page = 0;  // stay inside the cache; the result is flagged as invalid
            }
        }
        for (int k = 0; k < nt; k += TPS) {
            const int ns = min(TPS, nt - k);  // tiles in this stage
            int pg[TPS];
#pragma unroll
            for (int s = 0; s < TPS; ++s) pg[s] = __shfl_sync(kFullMask, page, min(k + s, 31));
            const bool last_stage = t0 + k + ns == te;
            // the combine step needs the unit's chunk layout with the last
            // stage: read from the map ahead of the stage's wait, or (a
            // descriptor derived before the map was read) looked up once the
            // stage's copies are on their way
            const bool defer = last_stage && desc_idx < 0 && !walk && !ps.waited;
            int idx = desc_idx, count = 0, chunk_off = 0;
            if (last_stage && walk) {
                walk_chunk(p, *walk, idx, count, chunk_off);
            } else if (last_stage && !defer) {
                wait_for_map(ps);
                if (idx < 0) idx = p.bin_ptr[bin] + bin_pos;
                if (p.chunk_count) {
                    count = p.chunk_count[u];
                    chunk_off = p.chunk_off[u];
                }
            }
            const int stage = ps.it % STAGES;
            const uint32_t phase = (ps.it / STAGES) & 1u;
            if (!warp_wait(&empty[stage], phase ^ 1u, abort)) return false;
            if (lane == 0) {
                const int t = t0 + k;
                const bool first = t == tb;
                StageInfo &si = info[stage];
                si.kv_head = h;
                si.req = r;
                si.tile0 = t;
                si.ntiles = ns;
                si.flags = (first ? kFirst : 0) | (last_stage ? kLast : 0);
                si.seqlen = L;
                si.desc_idx = idx;
                si.count = count;
                si.chunk_off = chunk_off;
                if (!late_q) {
#pragma unroll
                    for (int g = 0; g < Tr::kRows; ++g) si.qscale[g] = qsg[g];
                }
                const uint32_t bytes = 2u * ns * Tr::kTileBytes + (first ? q_bytes : 0u);
                if (defer || late_q) mbar_expect_tx(&full[stage], bytes);  // arrives below
                else mbar_arrive_expect_tx(&full[stage], bytes);
#pragma unroll
                for (int s = 0; s < TPS; ++s) {
                    if (s >= ns) break;
                    uint8_t *sk = smem + Tr::kOffK + stage * Tr::kStageKV + s * Tr::kTileBytes;
                    uint8_t *sv = smem + Tr::kOffV + stage * Tr::kStageKV + s * Tr::kTileBytes;
                    if (FP8) {
                        tma_load_4d(sk, tmap_k, &full[stage], 0, h, 0, pg[s], policy);
                        tma_load_4d(sv, tmap_v, &full[stage], 0, h, 0, pg[s], policy);
                    } else {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            tma_load_5d(sk + half * Tr::kHalfBytes, tmap_k, &full[stage], 0, half,
                                        h, 0, pg[s], policy);
                            tma_load_5d(sv + half * Tr::kHalfBytes, tmap_v, &full[stage], 0, half,
                                        h, 0, pg[s], policy);
                        }
                    }
                }
                if (first)
                    for (int i = 0; i < p.q_len; ++i)
                        bulk_load(smem + Tr::kOffQ + stage * Tr::kQBytes + i * q_group,
                                  q_src + i * q_token_stride, q_group, &full[stage]);
            }
            if (late_q) {
#pragma unroll
                for (int g = 0; g < Tr::kRows; ++g) qsg[g] = __shfl_sync(kFullMask, qs, g);
                late_q = false;
                if (lane == 0) {
#pragma unroll
                    for (int g = 0; g < Tr::kRows; ++g) info[stage].qscale[g] = qsg[g];
                    if (!defer) mbar_arrive(&full[stage]);  // releases the q-scales with it
                }
            }
            if (defer) {
                wait_for_map(ps);
                idx = p.bin_ptr[bin] + bin_pos;
                if (p.chunk_count) {
                    count = p.chunk_count[u];
                    chunk_off = p.chunk_off[u];
                }
                if (lane == 0) {
                    StageInfo &si = info[stage];
                    si.desc_idx = idx;
                    si.count = count;
                    si.chunk_off = chunk_off;
                    mbar_arrive(&full[stage]);  // releases the stage's fields with it
                }
            }
            __syncwarp();
            ++ps.it;
        }
    }
    return true;
}

template <bool FP8, int STAGES, int TPS, int NB>
__device__ __forceinline__ void attn_producer(const CUtensorMap *tmap_k, const CUtensorMap *tmap_v,
                                              const AttnParams &p, uint8_t *smem,
                                              volatile int *abort) {
    using Tr = AttnTraits<FP8, STAGES, TPS, NB>;
    const int lane = threadIdx.x & 31;
    StageInfo *info = reinterpret_cast<StageInfo *>(smem + Tr::kOffInfo);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Tr::kOffBar);
    uint64_t *empty = full + STAGES;
    const uint64_t policy = policy_evict_first();
    ProducerState ps{0u, false, 0u};
    bool ok = true;

    // The task map is read only after grid_dependency_wait (the assign kernel
    // may still be running when this grid starts).  The first descriptor of
    // the first bin needs no map: it is derived from the sequence lengths
    // (caller inputs, complete before the assign kernel passed its own wait),
    // so streaming starts at once.
    // A CTA whose first descriptors are short (the tail of a unit that began
    // in the bin before) would reach their ends, where the combine needs the
    // map, long before the map is visible: for batches of up to 64 requests it
    // walks its bin from the lengths, with the chunk layout derived too, until
    // kWalkTiles tiles are on their way; the map takes over from there.
    int skip = 0;  // descriptors of the first bin already streamed
    const bool dynamic = p.num_bins > (int)gridDim.x;
    bool walked = false;  // the whole first bin came from the walk (the map is not needed)
    if (p.fly && p.B <= kWalkMaxBatch) {
        FlyWalk w;
        walk_init(p, blockIdx.x, w);
        int streamed = 0;
        while (ok && w.te > w.tb) {
            const bool derive = streamed + (w.te - w.tb) < kWalkTiles;
            ok = stream_desc<FP8, STAGES, TPS, NB>(tmap_k, tmap_v, p, smem, w.h, w.r, w.tb, w.te,
                                               -1, blockIdx.x, derive ? &w : nullptr, w.k, ps,
                                               policy, abort);
            ++skip;
            streamed += w.te - w.tb;
            if (!derive) break;  // its end read the map
            walk_next(p, w);
        }
        walked = ok && w.te == w.tb && !ps.waited && !dynamic;
    } else if (p.fly) {
        int h, r, tb, te;
        if (first_descriptor(p, blockIdx.x, h, r, tb, te) && te > tb) {
            ok = stream_desc<FP8, STAGES, TPS, NB>(tmap_k, tmap_v, p, smem, h, r, tb, te, -1,
                                               blockIdx.x, nullptr, 0, ps, policy, abort);
            skip = 1;
        }
    }
    if (!walked) wait_for_map(ps);

    // Bins: CTA c starts with bin c; with more bins than CTAs the rest are
    // pulled in order from a device counter (the grab for the following bin
    // is issued when a bin starts, so its latency hides behind the stream).
    int bin = blockIdx.x;
    while (ok && !walked) {
        int grab = 0;
        if (dynamic && lane == 0) grab = atomicAdd(p.bin_counter, 1);
        const int d_begin = p.bin_ptr[bin] + (bin == (int)blockIdx.x ? skip : 0);
        const int d_end = p.bin_ptr[bin + 1];
        for (int d = d_begin; d < d_end && ok; ++d) {
            const int4 ds = p.desc[d];
            ok = stream_desc<FP8, STAGES, TPS, NB>(tmap_k, tmap_v, p, smem, ds.x, ds.y, ds.z, ds.w, d,
                                               bin, nullptr, 0, ps, policy, abort);
        }
        if (!dynamic) break;
        grab = __shfl_sync(kFullMask, grab, 0);
        if (grab == p.num_bins - 1 && lane == 0) *p.bin_counter = 0;  // last grab of the launch
        bin = (int)gridDim.x + grab;
        if (bin >= p.num_bins) break;
    }
    if (ok) {  // terminator
        const int stage = ps.it % STAGES;
        if (warp_wait(&empty[stage], ((ps.it / STAGES) & 1u) ^ 1u, abort)) {
            if (lane == 0) {
                info[stage].flags = kEnd;
                mbar_arrive(&full[stage]);
            }
            ++ps.it;
        } else {
            ok = false;
        }
    }
    if (!ok) ps.late_flags |= HPC_FLAG_TIMEOUT;
    const unsigned flags = __reduce_or_sync(kFullMask, ps.late_flags);
    if (flags) {
        wait_for_map(ps);  // meta[3] is written by the assign kernel
        if (lane == 0) atomicOr(p.meta + 3, (int)flags);
    }
    // Before leaving, make sure no copy this warp issued is still in flight
    // (bounded as well): the last phase issued on every stage must complete.
    // Every lane waits, so none is parked at a warp barrier meanwhile.
    {
        volatile int no_abort = 0;
        const uint32_t from = ps.it > (uint32_t)STAGES ? ps.it - STAGES : 0u;
        for (uint32_t j = from; j < ps.it; ++j)
            mbar_wait(&full[j % STAGES], (j / STAGES) & 1u, &no_abort);
    }
    __syncwarp();
}

// Merge of split unit `di` for query row rho (= i * G + g) by one warp: lane l
// owns dims 4l .. 4l + 3; LSEs are read lane-parallel and their weights
// broadcast by shuffle, with MB partial rows in flight at a time (the merge
// runs at the end of the stream, when the registers are free, so a long
// unit's chunks cost few L2 round trips; MB = 16 for one row block, 8 for two,
// whose kernels have fewer registers to spare).  A row that sees no token in
// any chunk (multi-query rows of a request shorter than q_len) is written as
// zeros.
template <int MB>
__device__ __forceinline__ void merge_unit_head(const AttnParams &p, const DescInfo &di, int rho) {
    const int lane = threadIdx.x & 31;
    const float *lse = p.part_lse + (size_t)di.chunk_off * p.R + rho;
    const float4 *po = reinterpret_cast<const float4 *>(
                           p.part_o + ((size_t)di.chunk_off * p.R + rho) * kHeadDim) + lane;
    const size_t row = (size_t)p.R * kHeadDim / 4;  // float4s between chunk rows
    float4 x[MB];
#pragma unroll
    for (int j = 0; j < MB; ++j)
        x[j] = j < di.count ? __ldcg(po + (size_t)j * row) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float lv0 = lane < di.count ? __ldcg(lse + (size_t)lane * p.R) : kNegInf;
    float m = lv0;
    for (int i = 32 + lane; i < di.count; i += 32) m = fmaxf(m, __ldcg(lse + (size_t)i * p.R));
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o_));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    for (int base = 0; base < di.count; base += 32) {
        const int cnt = min(32, di.count - base);
        float wl = 0.f;
        if (lane < cnt)
            wl = ex2(((base ? __ldcg(lse + (size_t)(base + lane) * p.R) : lv0) - m) * kLog2e);
        float ws = wl;
#pragma unroll
        for (int o_ = 16; o_ > 0; o_ >>= 1) ws += __shfl_xor_sync(kFullMask, ws, o_);
        wsum += ws;
        for (int i0 = 0; i0 < cnt; i0 += MB) {
            if (base | i0) {
#pragma unroll
                for (int j = 0; j < MB; ++j)
                    x[j] = i0 + j < cnt ? __ldcg(po + (size_t)(base + i0 + j) * row)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < MB; ++j) {
                const float w = __shfl_sync(kFullMask, wl, (i0 + j) & 31);
                acc.x += w * x[j].x; acc.y += w * x[j].y;
                acc.z += w * x[j].z; acc.w += w * x[j].w;
            }
        }
    }
    const float inv = m == kNegInf ? 0.f : 1.f / wsum;
    if (inv == 0.f) acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int qi = rho / p.G;
    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out) +
                         (((size_t)di.req * p.q_len + qi) * p.Hq + di.kv_head * p.G +
                          (rho - qi * p.G)) * kHeadDim + 4 * lane;
    *reinterpret_cast<uint2 *>(dst) =
        make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

// The same for K rows at once (rows of split units with at most 32 chunks):
// each round issues MB partial rows of every one of the K rows before any is
// consumed, so a warp merging two rows pays the L2 round trips once.
template <int MB, int K>
__device__ __forceinline__ void merge_unit_rows(const AttnParams &p, const DescInfo (&di)[K],
                                                const int (&rho)[K]) {
    const int lane = threadIdx.x & 31;
    const size_t row = (size_t)p.R * kHeadDim / 4;  // float4s between chunk rows
    const float4 *po[K];
    float wl[K], wsum[K], m[K];
    float4 acc[K];
    float4 x[K][MB];
    int maxc = 0;
    // first round: every row's LSEs and its first MB chunk rows together (the
    // rows do not depend on the weights)
#pragma unroll
    for (int k = 0; k < K; ++k) {
        po[k] = reinterpret_cast<const float4 *>(p.part_o +
                                                 ((size_t)di[k].chunk_off * p.R + rho[k]) * kHeadDim) +
                lane;
        const float *lse = p.part_lse + (size_t)di[k].chunk_off * p.R + rho[k];
        wl[k] = lane < di[k].count ? __ldcg(lse + (size_t)lane * p.R) : kNegInf;
        maxc = max(maxc, di[k].count);
        acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < MB; ++j)
            x[k][j] = j < di[k].count ? __ldcg(po[k] + (size_t)j * row)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
        m[k] = wl[k];
#pragma unroll
        for (int o_ = 16; o_ > 0; o_ >>= 1) m[k] = fmaxf(m[k], __shfl_xor_sync(kFullMask, m[k], o_));
        wl[k] = lane < di[k].count ? ex2((wl[k] - m[k]) * kLog2e) : 0.f;
        wsum[k] = wl[k];
#pragma unroll
        for (int o_ = 16; o_ > 0; o_ >>= 1) wsum[k] += __shfl_xor_sync(kFullMask, wsum[k], o_);
    }
    for (int i0 = 0; i0 < maxc; i0 += MB) {
        if (i0 > 0) {
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int j = 0; j < MB; ++j)
                    x[k][j] = i0 + j < di[k].count ? __ldcg(po[k] + (size_t)(i0 + j) * row)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int j = 0; j < MB; ++j) {
                const float w = __shfl_sync(kFullMask, wl[k], (i0 + j) & 31);
                acc[k].x += w * x[k][j].x; acc[k].y += w * x[k][j].y;
                acc[k].z += w * x[k][j].z; acc[k].w += w * x[k][j].w;
            }
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const float inv = m[k] == kNegInf ? 0.f : 1.f / wsum[k];
        const float4 a = inv == 0.f ? make_float4(0.f, 0.f, 0.f, 0.f) : acc[k];
        const int qi = rho[k] / p.G;
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out) +
                             (((size_t)di[k].req * p.q_len + qi) * p.Hq + di[k].kv_head * p.G +
                              (rho[k] - qi * p.G)) * kHeadDim + 4 * lane;
        *reinterpret_cast<uint2 *>(dst) =
            make_uint2(pack_bf16x2(a.x * inv, a.y * inv), pack_bf16x2(a.z * inv, a.w * inv));
    }
}

// ------------------------------------------------------------------ combiner
// Register r = 4 j + e of accumulator lane (g, t4) holds (dim, head):
//   head = 2 t4 + (e & 1);
//   BF16: dim = 16 j + g + 8 (e >> 1)   (m-tile j, rows g and g + 8)
//   FP8:  dim = 16 g + 2 j + (e >> 1)   (permuted rows, see the consumer)
template <bool FP8>
__device__ __forceinline__ int state_dim(int r, int g) {
    const int j = r >> 2, e = r & 3;
    return FP8 ? 16 * g + 2 * j + (e >> 1) : 16 * j + g + 8 * (e >> 1);
}

// Column of `dim` in a staging row: the float4 group is XOR-ed with
// (dim / 16) % 8, which spreads the combiner's scalar writes over more
// banks (FP8 lanes own 16 consecutive dims) while keeping float4 reads of
// dims 4q .. 4q + 3 contiguous.
__device__ __forceinline__ int stage_col(int dim) { return dim ^ (((dim >> 4) & 7) << 2); }

// Merges the consumers' states of each finished descriptor and writes the
// result; counts chunks of split units.  Returns false after a timeout.
template <bool FP8, int STAGES, int TPS, int NB>
__device__ __forceinline__ bool attn_combiner(const AttnParams &p, uint8_t *smem,
                                              volatile int *abort) {
    using Tr = AttnTraits<FP8, STAGES, TPS, NB>;
    constexpr int NC = Tr::kConsumers;
    const int lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
    const float *comb = reinterpret_cast<const float *>(smem + Tr::kOffComb);
    float *stage = reinterpret_cast<float *>(smem + Tr::kOffStage);
    const SlotInfo *slots = reinterpret_cast<const SlotInfo *>(smem + Tr::kOffSlotInfo);
    SlotInfo *last = reinterpret_cast<SlotInfo *>(smem + Tr::kOffLast);  // [0].flags = count
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Tr::kOffBar);
    uint64_t *slot_full = bars + 2 * STAGES, *slot_empty = slot_full + Tr::kSlots;
    const bool fused = p.out != nullptr;
    int nlast = 0;

    for (uint32_t n = 0;; ++n) {
        const int k = n % Tr::kSlots;
        if (!warp_wait(&slot_full[k], (n / Tr::kSlots) & 1u, abort)) return false;
        const SlotInfo si = slots[k];
        if (si.flags & kEnd) break;
        // [warp][lane][36 NB]: this lane's 9 NB float4 of every consumer warp;
        // row block nb holds rows 8 nb + (2 t4, 2 t4 + 1) of this lane
        const float4 *st = reinterpret_cast<const float4 *>(comb + k * Tr::kSlotFloats) +
                           lane * 9 * NB;
        float lse_l[NB][2];  // natural-log LSE of this lane's two rows of each block
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float4 ml[NC];
            float M0 = kNegInf, M1 = kNegInf;
#pragma unroll
            for (int w = 0; w < NC; ++w) {
                ml[w] = st[w * 32 * 9 * NB + nb * 9 + 8];  // (m0, m1, l0, l1)
                M0 = fmaxf(M0, ml[w].x);
                M1 = fmaxf(M1, ml[w].y);
            }
            const float Z0 = M0 == kNegInf ? 0.f : M0, Z1 = M1 == kNegInf ? 0.f : M1;
            float acc[32], L0 = 0.f, L1 = 0.f;
#pragma unroll
            for (int r = 0; r < 32; ++r) acc[r] = 0.f;
#pragma unroll
            for (int w = 0; w < NC; ++w) {
                const float a0 = ex2(ml[w].x - Z0), a1 = ex2(ml[w].y - Z1);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 v = st[w * 32 * 9 * NB + nb * 9 + j];
                    acc[4 * j + 0] += v.x * a0;
                    acc[4 * j + 1] += v.y * a1;
                    acc[4 * j + 2] += v.z * a0;
                    acc[4 * j + 3] += v.w * a1;
                }
                L0 += ml[w].z * a0;
                L1 += ml[w].w * a1;
            }
            if (nb == NB - 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&slot_empty[k]);  // the consumers may refill the slot
            }
#pragma unroll
            for (int o_ = 4; o_ <= 16; o_ <<= 1) {  // per-row sums over the tokens of all lanes
                L0 += __shfl_xor_sync(kFullMask, L0, o_);
                L1 += __shfl_xor_sync(kFullMask, L1, o_);
            }
            // a row that saw no token (L = 0) is a zero row with LSE -inf
            const float inv0 = L0 > 0.f ? p.v_scale / L0 : 0.f;
            const float inv1 = L1 > 0.f ? p.v_scale / L1 : 0.f;
            lse_l[nb][0] = L0 > 0.f ? (Z0 + lg2(L0)) * kLn2 : kNegInf;
            lse_l[nb][1] = L1 > 0.f ? (Z1 + lg2(L1)) * kLn2 : kNegInf;
            // stage the normalised result as [row][dim] for coalesced stores
#pragma unroll
            for (int r = 0; r < 32; ++r)
                stage[(8 * nb + 2 * t4 + (r & 1)) * kStageStride + stage_col(state_dim<FP8>(r, g))] =
                    acc[r] * ((r & 1) ? inv1 : inv0);
        }
        __syncwarp();
        const DescInfo di = si.di;
        const bool direct = fused && di.count == 1;
        if (direct) {  // the unit's only chunk: final BF16 output
            for (int rho = 0; rho < p.R; ++rho) {
                const float4 v = *reinterpret_cast<const float4 *>(stage + rho * kStageStride +
                                                                   stage_col(4 * lane));
                const int qi = rho / p.G;
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out) +
                                     (((size_t)di.req * p.q_len + qi) * p.Hq + di.kv_head * p.G +
                                      (rho - qi * p.G)) * kHeadDim;
                reinterpret_cast<uint2 *>(dst)[lane] =
                    make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
            }
        } else {  // partial + LSE, kept in L2 for the CTA (or kernel) that merges
            const uint64_t keep = policy_evict_last();
            for (int rho = 0; rho < p.R; ++rho) {
                const float4 v = *reinterpret_cast<const float4 *>(stage + rho * kStageStride +
                                                                   stage_col(4 * lane));
                float *dst = p.part_o + ((size_t)di.desc_idx * p.R + rho) * kHeadDim;
                st_global_hint(reinterpret_cast<float4 *>(dst) + lane, v, keep);
            }
            if (g == 0) {
                float *dl = p.part_lse + (size_t)di.desc_idx * p.R;
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    const int rho = 8 * nb + 2 * t4;
                    if (rho < p.R) st_global_hint(dl + rho, lse_l[nb][0], keep);
                    if (rho + 1 < p.R) st_global_hint(dl + rho + 1, lse_l[nb][1], keep);
                }
            }
            if (fused) {  // count this chunk of a split unit
                __syncwarp();  // every lane's partial stores precede lane 0's release below
                int completes = 0;
                if (lane == 0) {
                    int *ctr = p.unit_done + di.kv_head * p.B + di.req;
                    const int prev = atom_add_acq_rel_gpu(ctr, 1);
                    if (prev == di.count - 1) {  // this CTA completes the unit
                        *ctr = 0;                 // every chunk counted: ready for the next launch
                        completes = 1;
                    }
                }
                if (__shfl_sync(kFullMask, completes, 0)) {
                    if (nlast < kMaxLast) {  // merged at the end by all warps
                        if (lane == 0) last[1 + nlast].di = di;
                        ++nlast;
                    } else {  // list full (many bins per CTA): merge here, alone
                        for (int rho = 0; rho < p.R; ++rho) merge_unit_head<NB == 1 ? 16 : 8>(p, di, rho);
                    }
                }
            }
        }
        __syncwarp();  // the staging area is rewritten by the next descriptor
    }
    if (lane == 0) last[0].flags = nlast;
    return true;
}

// ------------------------------------------------------------------ consumer
template <bool FP8, int STAGES, int TPS, int NB>
__device__ __forceinline__ bool attn_consumer(const AttnParams &p, uint8_t *smem,
                                              volatile int *abort) {
    using Tr = AttnTraits<FP8, STAGES, TPS, NB>;
    const int lane = threadIdx.x & 31, cw = (threadIdx.x >> 5) - 2;
    const int g = lane >> 2, t4 = lane & 3;
    const int slot = cw >> 2;  // which tile of the stage this warp works on
    const int sub = cw & 3;    // which 16 tokens of that tile
    const StageInfo *info = reinterpret_cast<const StageInfo *>(smem + Tr::kOffInfo);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Tr::kOffBar);
    uint64_t *empty = full + STAGES;
    uint64_t *slot_full = full + 2 * STAGES, *slot_empty = slot_full + Tr::kSlots;
    float *comb = reinterpret_cast<float *>(smem + Tr::kOffComb);
    SlotInfo *slots = reinterpret_cast<SlotInfo *>(smem + Tr::kOffSlotInfo);
    const uint32_t sK0 = smem_u32(smem + Tr::kOffK) + slot * Tr::kTileBytes;
    const uint32_t sV0 = smem_u32(smem + Tr::kOffV) + slot * Tr::kTileBytes;

    // Lane-constant parts of the shared-memory addresses.  ldmatrix: lane
    // supplies row (lane & 7) of matrix (lane >> 3).
    const int mi = lane >> 3;
    const int tok_k = 16 * sub + (lane & 7) + (mi & 1) * 8;  // K: matrices 1, 3 = rows 8..15
    const int tok_v = 16 * sub + (lane & 7) + (mi >> 1) * 8;  // V^T: matrices 2, 3 = toks 8..15

    // Row block nb holds query rows 8 nb .. 8 nb + 7; this lane owns columns
    // (rows) 8 nb + 2 t4 + c, c = 0, 1 of every block.
    float o[NB][8][4];
    float m[NB][2], l[NB][2], sc[NB][2];
    int lim[NB][2];  // tokens visible to the lane's rows: t < lim (causal for q_len > 1)
    uint32_t qf[NB][8][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            m[nb][c] = kNegInf;
            l[nb][c] = sc[nb][c] = 0.f;
            lim[nb][c] = 0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            o[nb][j][0] = o[nb][j][1] = o[nb][j][2] = o[nb][j][3] = 0.f;
            qf[nb][j][0] = qf[nb][j][1] = 0u;
        }
    }

    uint32_t handed = 0;  // descriptors handed to the combiner
    for (uint32_t it = 0;; ++it) {
        const int stage = it % STAGES;
        if (!warp_wait(&full[stage], (it / STAGES) & 1u, abort)) return false;
        const int flags = info[stage].flags;
        const int ntiles = info[stage].ntiles, tile0 = info[stage].tile0;
        const int L = info[stage].seqlen;
        DescInfo di;
        if (flags & kLast)
            di = {info[stage].req, info[stage].kv_head, info[stage].desc_idx, info[stage].count,
                  info[stage].chunk_off};

        if (!(flags & kEnd)) {
            if (flags & kFirst) {  // new descriptor: load Q^T fragments, reset the state
                // B fragment of Q^T (k = dim, n = row): lane holds row 8 nb + g, dims
                // 2t4.. (bf16) or 4t4.. (e4m3) of each k-step, and +8 / +16 beyond.
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    const int row = 8 * nb + g;
                    const uint8_t *q =
                        smem + Tr::kOffQ + stage * Tr::kQBytes + row * kHeadDim * Tr::kElem;
                    const bool live = row < p.R;
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        if (FP8 && s >= 4) break;
                        const int off = FP8 ? 32 * s + 4 * t4 : 2 * (16 * s + 2 * t4);
                        qf[nb][s][0] = live ? *reinterpret_cast<const uint32_t *>(q + off) : 0u;
                        qf[nb][s][1] = live ? *reinterpret_cast<const uint32_t *>(q + off + 16) : 0u;
                    }
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int rho = 8 * nb + 2 * t4 + c;
                        sc[nb][c] = p.score_scale * info[stage].qscale[rho];
                        // query token i = rho / G sees tokens below L - q_len + 1 + i
                        lim[nb][c] = rho < p.R ? L - p.q_len + 1 + rho / p.G : L;
                        m[nb][c] = kNegInf;
                        l[nb][c] = 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        o[nb][j][0] = o[nb][j][1] = o[nb][j][2] = o[nb][j][3] = 0.f;
                }
            }

            if (slot < ntiles) {
                const uint32_t sK = sK0 + stage * Tr::kStageKV, sV = sV0 + stage * Tr::kStageKV;
                const int tile = tile0 + slot;

                // ---- S^T = K . Q^T for this warp's 16 tokens x 8 NB rows
                float s4[NB][4];
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) s4[nb][0] = s4[nb][1] = s4[nb][2] = s4[nb][3] = 0.f;
                if (FP8) {
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const int chunk = 2 * s + (mi >> 1);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(sK + tok_k * 128 + ((chunk ^ (tok_k & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb)
                            mma_e4m3_16832(s4[nb], a0, a1, a2, a3, qf[nb][s][0], qf[nb][s][1]);
                    }
                } else {
                    float s4b[NB][4];  // two chains: even / odd k-steps
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
                        s4b[nb][0] = s4b[nb][1] = s4b[nb][2] = s4b[nb][3] = 0.f;
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const int chunk = (2 * s + (mi >> 1)) & 7;
                        const uint32_t addr = sK + (s >> 2) * Tr::kHalfBytes + tok_k * 128 +
                                              ((chunk ^ (tok_k & 7)) << 4);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb) {
                            if (s & 1)
                                mma_bf16_16816(s4b[nb], a0, a1, a2, a3, qf[nb][s][0], qf[nb][s][1]);
                            else
                                mma_bf16_16816(s4[nb], a0, a1, a2, a3, qf[nb][s][0], qf[nb][s][1]);
                        }
                    }
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                        for (int e = 0; e < 4; ++e) s4[nb][e] += s4b[nb][e];
                }

                // FP8: the V^T fragments do not depend on P, so they are loaded
                // and widened to f16 here and the conversions overlap the
                // softmax's latencies (the two-row-block kernel, bound by its
                // consumers, gains ~2%; it also no longer spills)
                uint32_t va[8][4];
                if (FP8) {
                    // rows 2t4, 2t4+1, 2t4+8, 2t4+9 of the slice; dims 16g .. 16g+15
                    uint4 Rv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int tok = 16 * sub + 2 * t4 + (q & 1) + (q >> 1) * 8;
                        Rv[q] = lds128(sV + tok * 128 + ((g ^ (tok & 7)) << 4));
                        if (tile * kTile + tok >= L) Rv[q] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    const uint32_t wA[4] = {Rv[0].x, Rv[0].y, Rv[0].z, Rv[0].w};
                    const uint32_t wB[4] = {Rv[1].x, Rv[1].y, Rv[1].z, Rv[1].w};
                    const uint32_t wC[4] = {Rv[2].x, Rv[2].y, Rv[2].z, Rv[2].w};
                    const uint32_t wD[4] = {Rv[3].x, Rv[3].y, Rv[3].z, Rv[3].w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t sel = (j & 1) ? 0x7362u : 0x5140u;
                        e4m3x4_to_f16x2x2(__byte_perm(wA[j >> 1], wB[j >> 1], sel), va[j][0], va[j][1]);
                        e4m3x4_to_f16x2x2(__byte_perm(wC[j >> 1], wD[j >> 1], sel), va[j][2], va[j][3]);
                    }
                }
                // ---- online softmax (log2 domain); a token at or past a row's
                // limit is masked for that row
                const int tok0 = tile * kTile + 16 * sub;  // first token of this warp's slice
                const int ta = tok0 + g, tb_ = tok0 + g + 8;
                float x[NB][4], mx[NB][2];
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    x[nb][0] = ta < lim[nb][0] ? s4[nb][0] * sc[nb][0] : kNegInf;
                    x[nb][1] = ta < lim[nb][1] ? s4[nb][1] * sc[nb][1] : kNegInf;
                    x[nb][2] = tb_ < lim[nb][0] ? s4[nb][2] * sc[nb][0] : kNegInf;
                    x[nb][3] = tb_ < lim[nb][1] ? s4[nb][3] * sc[nb][1] : kNegInf;
                    mx[nb][0] = fmaxf(x[nb][0], x[nb][2]);
                    mx[nb][1] = fmaxf(x[nb][1], x[nb][3]);
                }
#pragma unroll
                for (int o_ = 4; o_ <= 16; o_ <<= 1)
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        mx[nb][0] = fmaxf(mx[nb][0], __shfl_xor_sync(kFullMask, mx[nb][0], o_));
                        mx[nb][1] = fmaxf(mx[nb][1], __shfl_xor_sync(kFullMask, mx[nb][1], o_));
                    }
                float al[NB][2];
                bool rescale = false;
                uint32_t b0[NB], b1[NB];
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    float ms[2];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const float mn = fmaxf(m[nb][c], mx[nb][c]);
                        ms[c] = mn == kNegInf ? 0.f : mn;
                        al[nb][c] = ex2(m[nb][c] - ms[c]);
                        m[nb][c] = mn;
                        rescale |= al[nb][c] != 1.f;
                    }
                    const float p0 = ex2(x[nb][0] - ms[0]), p1 = ex2(x[nb][1] - ms[1]);
                    const float p2 = ex2(x[nb][2] - ms[0]), p3 = ex2(x[nb][3] - ms[1]);
                    uint32_t pk01, pk23;
                    if (FP8) {
                        pk01 = pack_f16x2(p0, p1);
                        pk23 = pack_f16x2(p2, p3);
                        const float2 r01 = f16x2_to_f32x2(pk01), r23 = f16x2_to_f32x2(pk23);
                        l[nb][0] = l[nb][0] * al[nb][0] + r01.x + r23.x;
                        l[nb][1] = l[nb][1] * al[nb][1] + r01.y + r23.y;
                    } else {
                        pk01 = pack_bf16x2(p0, p1);
                        pk23 = pack_bf16x2(p2, p3);
                        l[nb][0] = l[nb][0] * al[nb][0] + bf16lo_to_f32(pk01) + bf16lo_to_f32(pk23);
                        l[nb][1] = l[nb][1] * al[nb][1] + bf16hi_to_f32(pk01) + bf16hi_to_f32(pk23);
                    }
                    // P^T fragments (k = token, n = row): transpose the 8x8 halves
                    b0[nb] = movmatrix_trans(pk01);
                    b1[nb] = movmatrix_trans(pk23);
                }
                if (__any_sync(kFullMask, rescale)) {  // rescale only on a new max
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            o[nb][j][0] *= al[nb][0];
                            o[nb][j][1] *= al[nb][1];
                            o[nb][j][2] *= al[nb][0];
                            o[nb][j][3] *= al[nb][1];
                        }
                }

                // ---- O^T += V^T . P^T (one V fragment feeds every row block)
                if (FP8) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb)
                            mma_f16_16816(o[nb][j], va[j][0], va[j][1], va[j][2], va[j][3], b0[nb], b1[nb]);
                } else {
                    const int tv = tok0 + 2 * t4;  // tokens of a0/a1 halves; +8 for a2/a3
                    const uint32_t mk01 =
                        (tv < L ? 0x0000ffffu : 0u) | (tv + 1 < L ? 0xffff0000u : 0u);
                    const uint32_t mk23 =
                        (tv + 8 < L ? 0x0000ffffu : 0u) | (tv + 9 < L ? 0xffff0000u : 0u);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int chunk = (2 * j + (mi & 1)) & 7;
                        const uint32_t addr = sV + (j >> 2) * Tr::kHalfBytes + tok_v * 128 +
                                              ((chunk ^ (tok_v & 7)) << 4);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_trans(addr, a0, a1, a2, a3);
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb)
                            mma_bf16_16816(o[nb][j], a0 & mk01, a1 & mk01, a2 & mk23, a3 & mk23,
                                           b0[nb], b1[nb]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && !(flags & kEnd)) mbar_arrive(&empty[stage]);  // stage may be refilled

        if (flags & (kLast | kEnd)) {  // hand the state (or the end) to the combiner
            const int k = handed % Tr::kSlots;
            if (!warp_wait(&slot_empty[k], ((handed / Tr::kSlots) & 1u) ^ 1u, abort))
                return false;
            if (flags & kLast) {  // lane-major: 9 NB float4 per lane, conflict-free
                float4 *dst = reinterpret_cast<float4 *>(
                    comb + ((k * Tr::kConsumers + cw) * 32 + lane) * Tr::kState);
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[9 * nb + j] =
                            make_float4(o[nb][j][0], o[nb][j][1], o[nb][j][2], o[nb][j][3]);
                    dst[9 * nb + 8] = make_float4(m[nb][0], m[nb][1], l[nb][0], l[nb][1]);
                }
                if (cw == 0 && lane == 0) slots[k] = SlotInfo{di, 0, 0, 0};
            } else if (cw == 0 && lane == 0) {
                slots[k].flags = kEnd;
            }
            mbar_arrive(&slot_full[k]);  // every lane releases its own writes
            ++handed;
            if (flags & kEnd) return true;
        }
    }
}

// ------------------------------------------------------------------ kernel
template <bool FP8, int STAGES, int TPS, int NB>
__global__ void __launch_bounds__(AttnTraits<FP8, STAGES, TPS, NB>::kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
    using Tr = AttnTraits<FP8, STAGES, TPS, NB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Tr::kOffBar);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Tr::kOffMisc);
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars[s], 1);                          // full: producer arrive + TMA bytes
            mbar_init(&bars[STAGES + s], Tr::kConsumers);    // empty: one arrive per consumer warp
        }
        for (int k = 0; k < Tr::kSlots; ++k) {
            mbar_init(&bars[2 * STAGES + k], 32 * Tr::kConsumers);   // slot full: every consumer lane
            mbar_init(&bars[2 * STAGES + Tr::kSlots + k], 1);        // slot empty: the combiner
        }
        mbar_init(&bars[2 * STAGES + 2 * Tr::kSlots], 32 * (Tr::kConsumers + 1));  // end rendezvous
        *abort = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    // The block table and Q are caller inputs, not outputs of the assign
    // kernel: warm L2 with this CTA's share of them while the assign kernel
    // may still be running.
    {
        const size_t bt_bytes = (size_t)p.B * p.max_pages * 4;
        const size_t q_bytes = (size_t)p.B * p.q_len * p.Hq * kHeadDim * Tr::kElem;
        const char *bt = reinterpret_cast<const char *>(p.block_table);
        const char *q = static_cast<const char *>(p.q);
        for (size_t off = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 128; off < bt_bytes;
             off += (size_t)gridDim.x * blockDim.x * 128)
            prefetch_l2(bt + off);
        for (size_t off = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 128; off < q_bytes;
             off += (size_t)gridDim.x * blockDim.x * 128)
            prefetch_l2(q + off);
    }
    // No grid-wide wait here: only the producer reads the task map, and it
    // waits for the assign kernel right before it first needs the map.
    grid_launch_dependents();
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        attn_producer<FP8, STAGES, TPS, NB>(&tmap_k, &tmap_v, p, smem, abort);
        return;
    }
    // Every global write of this grid (outputs, partials, counters) comes
    // after the previous grid in the stream has finished: the combiner, idle
    // until the first hand-off, waits here; the end phase waits below.
    if (warp == 1) grid_dependency_wait();
    if (warp == 1 && p.out) {  // fused mode: requests without live tokens get zero rows
        const int row_vec = p.q_len * p.Hq * kHeadDim * 2 / 16;  // 16-byte vectors per request
        for (int r = blockIdx.x; r < p.B; r += gridDim.x) {
            if (p.seqlens[r] > 0) continue;
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) +
                                                   (size_t)r * p.q_len * p.Hq * kHeadDim);
            for (int i = lane; i < row_vec; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
        }
    }
    bool ok = warp == 1 ? attn_combiner<FP8, STAGES, TPS, NB>(p, smem, abort)
                        : attn_consumer<FP8, STAGES, TPS, NB>(p, smem, abort);
    if (!ok) {
        grid_dependency_wait();  // meta[3] is written by the assign kernel
        if (lane == 0) atomicOr(p.meta + 3, (int)HPC_FLAG_TIMEOUT);
        *abort = 1;
    }
    // End of the stream: the combiner has published the split units whose
    // merge this CTA owes; all non-producer warps merge them, one warp per
    // (unit, head).
    uint64_t *end_bar = bars + 2 * STAGES + 2 * Tr::kSlots;
    mbar_arrive(end_bar);
    if (!warp_wait(end_bar, 0, abort)) {
        grid_dependency_wait();
        if (lane == 0) atomicOr(p.meta + 3, (int)HPC_FLAG_TIMEOUT);
        return;
    }
    if (!p.out || *abort) return;
    grid_dependency_wait();  // (long complete by now) before this warp's first global writes
    const SlotInfo *last = reinterpret_cast<const SlotInfo *>(smem + Tr::kOffLast);
    const int nlast = last[0].flags;
    const int nw = 1 + Tr::kConsumers, w = warp - 1;
    const int items = nlast * p.R;
    if constexpr (!FP8) {
        // BF16: five merging warps, so a unit's eight rows (sixteen with two
        // query tokens) take two (four) passes one row at a time; two rows per
        // warp, their loads in flight together, take half as many
        for (int item = 2 * w; item < items; item += 2 * nw) {
            const DescInfo &d0 = last[1 + item / p.R].di;
            if (item + 1 < items) {
                const DescInfo &d1 = last[1 + (item + 1) / p.R].di;
                if (d0.count <= 32 && d1.count <= 32) {
                    const DescInfo dd[2] = {d0, d1};
                    const int rr[2] = {item % p.R, (item + 1) % p.R};
                    merge_unit_rows<12, 2>(p, dd, rr);
                } else {
                    merge_unit_head<NB == 1 ? 16 : 8>(p, d0, item % p.R);
                    merge_unit_head<NB == 1 ? 16 : 8>(p, d1, (item + 1) % p.R);
                }
            } else {
                merge_unit_head<NB == 1 ? 16 : 8>(p, d0, item % p.R);
            }
        }
    } else {
        for (int item = w; item < items; item += nw)
            merge_unit_head<NB == 1 ? 16 : 8>(p, last[1 + item / p.R].di, item % p.R);
    }
}

}  // namespace hpc
