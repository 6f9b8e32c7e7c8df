// Combine step: merges each (request, query head)'s per-chunk partials under
// the global softmax normalisation into the BF16 output (HPC-Ops vLLM post,
// "Compute and combine" bullet: the combine kernel reads the chunk count of
// each (head, request) pair; SGLang post, 围绕Live KV Work的调度).
//
// With q_len query tokens per request (multi-query decode) a unit's partial
// rows are rho = i * G + g (query token i, head g of the group) and the
// output is [B, q_len, Hq, 128].
//
// One warp per (request, query token, query head); lane i owns dims 4i .. 4i + 3, so every
// partial row (128 fp32) is one coalesced 512-byte read and the output row
// one 256-byte write.  Chunk LSEs are read lane-parallel and max-reduced.

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace hpc {
namespace {

constexpr int kCombineWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;

__global__ void __launch_bounds__(32 * kCombineWarps)
    combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_lse,
                   const int32_t *__restrict__ chunk_count, const int32_t *__restrict__ chunk_off,
                   int B, int Hq, int G, int q_len, __nv_bfloat16 *__restrict__ out) {
    grid_dependency_wait();  // partials of the attention grid are complete
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);  // (r * q_len + i) * Hq + hq
    if (row >= B * q_len * Hq) return;
    const int ri = row / Hq, hq = row - ri * Hq;
    const int r = ri / q_len, i = ri - r * q_len;
    const int h = hq / G;
    const int R = q_len * G, g = i * G + (hq - h * G);  // the unit's partial row
    const int u = h * B + r;
    const int n = chunk_count[u];
    const int off = chunk_off[u];

    // LSEs are read lane-parallel (lane i holds chunk base + i) and their
    // weights broadcast by shuffle, so the partial-row loads of up to four
    // chunks are in flight together instead of one dependent load per chunk.
    float m = -INFINITY;
    for (int c = lane; c < n; c += 32) m = fmaxf(m, part_lse[(size_t)(off + c) * R + g]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    for (int base = 0; base < n; base += 32) {
        const int cnt = min(32, n - base);
        const float wl =
            lane < cnt ? ex2((part_lse[(size_t)(off + base + lane) * R + g] - m) * kLog2e) : 0.f;
        float ws = wl;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
        wsum += ws;
        for (int k = 0; k < cnt; k += 4) {
            float4 x[4];
            float w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                w[j] = __shfl_sync(0xffffffffu, wl, (k + j) & 31);
                const size_t slot = (size_t)(off + base + k + j) * R + g;
                x[j] = k + j < cnt ? reinterpret_cast<const float4 *>(part_o + slot * kHeadDim)[lane]
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc.x += w[j] * x[j].x;
                acc.y += w[j] * x[j].y;
                acc.z += w[j] * x[j].z;
                acc.w += w[j] * x[j].w;
            }
        }
    }
    // no chunk, or no visible token for this query (all LSEs -inf): a zero row
    const float inv = n > 0 && m != -INFINITY ? 1.f / wsum : 0.f;
    if (inv == 0.f) acc = make_float4(0.f, 0.f, 0.f, 0.f);
    uint2 packed;
    packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2 *>(out + (size_t)row * kHeadDim)[lane] = packed;
}

}  // namespace

cudaError_t launch_combine(const float *part_o, const float *part_lse, const hpc_task_map &map,
                           int B, int Hq, int Hkv, int q_len, void *out, cudaStream_t s) {
    const int rows = B * q_len * Hq;
    if (rows == 0) return cudaSuccess;
    const int grid = (rows + kCombineWarps - 1) / kCombineWarps;
    // a programmatic dependent of the attention grid: launches during its tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * kCombineWarps);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, part_o, part_lse,
                              (const int32_t *)map.chunk_count, (const int32_t *)map.chunk_off, B,
                              Hq, Hq / Hkv, q_len, static_cast<__nv_bfloat16 *>(out));
}

}  // namespace hpc
