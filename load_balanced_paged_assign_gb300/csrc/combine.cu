// Combine step: merges each (request, query head)'s per-chunk partials under
// the global softmax normalisation into the BF16 output (HPC-Ops vLLM post,
// "Compute and combine" bullet: the combine kernel reads the chunk count of
// each (head, request) pair; SGLang post, 围绕Live KV Work的调度).
//
// One warp per (request, query head); lane i owns dims 4i .. 4i + 3, so every
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
                   int B, int Hq, int G, __nv_bfloat16 *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);  // r * Hq + hq
    if (row >= B * Hq) return;
    const int r = row / Hq, hq = row - r * Hq;
    const int h = hq / G, g = hq - h * G;
    const int u = h * B + r;
    const int n = chunk_count[u];
    const int off = chunk_off[u];

    float m = -INFINITY;
    for (int i = lane; i < n; i += 32) m = fmaxf(m, part_lse[(size_t)(off + i) * G + g]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    for (int i = 0; i < n; ++i) {
        const size_t slot = (size_t)(off + i) * G + g;
        const float w = ex2((part_lse[slot] - m) * kLog2e);
        const float4 o = reinterpret_cast<const float4 *>(part_o + slot * kHeadDim)[lane];
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
        wsum += w;
    }
    const float inv = n > 0 ? 1.f / wsum : 0.f;
    uint2 packed;
    packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2 *>(out + (size_t)row * kHeadDim)[lane] = packed;
}

}  // namespace

cudaError_t launch_combine(const float *part_o, const float *part_lse, const hpc_task_map &map,
                           int B, int Hq, int Hkv, void *out, cudaStream_t s) {
    const int rows = B * Hq;
    if (rows == 0) return cudaSuccess;
    const int grid = (rows + kCombineWarps - 1) / kCombineWarps;
    combine_kernel<<<grid, 32 * kCombineWarps, 0, s>>>(part_o, part_lse, map.chunk_count,
                                                       map.chunk_off, B, Hq, Hq / Hkv,
                                                       static_cast<__nv_bfloat16 *>(out));
    return cudaGetLastError();
}

}  // namespace hpc
