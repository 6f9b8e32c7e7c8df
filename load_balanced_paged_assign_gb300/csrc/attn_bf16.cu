// BF16 KV cache instantiation of the persistent attention kernel.
#include "attn_kernel.cuh"

namespace hpc {

// 4 stages x 1 tile x (16 KB K + 16 KB V), Q, two consumer -> combiner
// hand-off slots and the combiner's staging: about 183 KB, one CTA per SM.
#ifndef HPC_BF16_STAGES
#define HPC_BF16_STAGES 4
#endif
#ifndef HPC_BF16_TPS
#define HPC_BF16_TPS 1
#endif
constexpr int kStagesBf16 = HPC_BF16_STAGES;  // pipeline depth (build-time tunable)
constexpr int kTpsBf16 = HPC_BF16_TPS;        // tiles per stage: 1 or 2
using TraitsBf16 = AttnTraits<false, kStagesBf16, kTpsBf16, 1>;
// Multi-query decode with 8 < q_len * G <= 16 query rows per KV head: twice
// the state per consumer; one tile per stage (four consumers), four stages
// and two hand-off slots still fit (about 227 KB).
#ifndef HPC_BF16_STAGES_MQ
#define HPC_BF16_STAGES_MQ 4
#endif
#ifndef HPC_BF16_TPS_MQ
#define HPC_BF16_TPS_MQ 1
#endif
constexpr int kStagesBf16Mq = HPC_BF16_STAGES_MQ;
constexpr int kTpsBf16Mq = HPC_BF16_TPS_MQ;
using TraitsBf16Mq = AttnTraits<false, kStagesBf16Mq, kTpsBf16Mq, 2>;

AttnConfig attn_config_bf16(int nb) {
    if (nb == 2)
        return {reinterpret_cast<const void *>(&attn_kernel<false, kStagesBf16Mq, kTpsBf16Mq, 2>),
                TraitsBf16Mq::kSmemBytes, TraitsBf16Mq::kThreads};
    return {reinterpret_cast<const void *>(&attn_kernel<false, kStagesBf16, kTpsBf16, 1>),
            TraitsBf16::kSmemBytes, TraitsBf16::kThreads};
}

// Launched as a programmatic dependent of the previous kernel in the stream
// (the assign kernel): its prologue overlaps that kernel's tail.
cudaError_t launch_attn_bf16(int nb, const CUtensorMap &tk, const CUtensorMap &tv,
                             const AttnParams &p, int grid, cudaStream_t s) {
    const AttnConfig c = attn_config_bf16(nb);
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
    if (nb == 2) return cudaLaunchKernelEx(&cfg, attn_kernel<false, kStagesBf16Mq, kTpsBf16Mq, 2>, tk, tv, p);
    return cudaLaunchKernelEx(&cfg, attn_kernel<false, kStagesBf16, kTpsBf16, 1>, tk, tv, p);
}

}  // namespace hpc
