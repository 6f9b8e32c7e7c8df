// FP8-E4M3 KV cache instantiation of the persistent attention kernel.
#include "attn_kernel.cuh"

namespace hpc {

// 4 stages x 2 tiles x (8 KB K + 8 KB V), Q, two hand-off slots and the
// combiner's staging: about 210 KB, one CTA per SM; two tiles per stage give
// 8 consumer warps, which FP8 needs to hide its per-tile latency.
#ifndef HPC_FP8_STAGES
#define HPC_FP8_STAGES 4
#endif
#ifndef HPC_FP8_TPS
#define HPC_FP8_TPS 2
#endif
constexpr int kStagesFp8 = HPC_FP8_STAGES;  // pipeline depth (build-time tunable)
constexpr int kTpsFp8 = HPC_FP8_TPS;        // tiles per stage: 1 or 2
using TraitsFp8 = AttnTraits<true, kStagesFp8, kTpsFp8, 1>;
// Multi-query decode with 8 < q_len * G <= 16 query rows per KV head: twice
// the state per consumer; eight consumers (two tiles per stage) hide the
// per-tile latency as in decode, with a single hand-off slot to fit.
#ifndef HPC_FP8_STAGES_MQ
#define HPC_FP8_STAGES_MQ 4
#endif
#ifndef HPC_FP8_TPS_MQ
#define HPC_FP8_TPS_MQ 2
#endif
constexpr int kStagesFp8Mq = HPC_FP8_STAGES_MQ;
constexpr int kTpsFp8Mq = HPC_FP8_TPS_MQ;
using TraitsFp8Mq = AttnTraits<true, kStagesFp8Mq, kTpsFp8Mq, 2>;

AttnConfig attn_config_fp8(int nb) {
    if (nb == 2)
        return {reinterpret_cast<const void *>(&attn_kernel<true, kStagesFp8Mq, kTpsFp8Mq, 2>),
                TraitsFp8Mq::kSmemBytes, TraitsFp8Mq::kThreads};
    return {reinterpret_cast<const void *>(&attn_kernel<true, kStagesFp8, kTpsFp8, 1>),
            TraitsFp8::kSmemBytes, TraitsFp8::kThreads};
}

// Launched as a programmatic dependent of the previous kernel in the stream
// (the assign kernel): its prologue overlaps that kernel's tail.
cudaError_t launch_attn_fp8(int nb, const CUtensorMap &tk, const CUtensorMap &tv,
                             const AttnParams &p, int grid, cudaStream_t s) {
    const AttnConfig c = attn_config_fp8(nb);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(c.threads);
    cfg.dynamicSmemBytes = c.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (nb == 2) return cudaLaunchKernelEx(&cfg, attn_kernel<true, kStagesFp8Mq, kTpsFp8Mq, 2>, tk, tv, p);
    return cudaLaunchKernelEx(&cfg, attn_kernel<true, kStagesFp8, kTpsFp8, 1>, tk, tv, p);
}

}  // namespace hpc
