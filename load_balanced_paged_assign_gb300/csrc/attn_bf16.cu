// BF16 KV cache instantiation of the persistent attention kernel.
#include "attn_kernel.cuh"

namespace hpc {

// 4 stages x 1 tile x (16 KB K + 16 KB V) + Q: about 155 KB, one CTA per SM.
#ifndef HPC_BF16_STAGES
#define HPC_BF16_STAGES 4
#endif
#ifndef HPC_BF16_TPS
#define HPC_BF16_TPS 1
#endif
constexpr int kStagesBf16 = HPC_BF16_STAGES;  // pipeline depth (build-time tunable)
constexpr int kTpsBf16 = HPC_BF16_TPS;        // tiles per stage: 1 or 2
using TraitsBf16 = AttnTraits<false, kStagesBf16, kTpsBf16>;

AttnConfig attn_config_bf16() {
    return {reinterpret_cast<const void *>(&attn_kernel<false, kStagesBf16, kTpsBf16>),
            TraitsBf16::kSmemBytes, TraitsBf16::kThreads};
}

// Launched as a programmatic dependent of the previous kernel in the stream
// (the assign kernel): its prologue overlaps that kernel's tail.
cudaError_t launch_attn_bf16(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &p,
                             int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(TraitsBf16::kThreads);
    cfg.dynamicSmemBytes = TraitsBf16::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_kernel<false, kStagesBf16, kTpsBf16>, tk, tv, p);
}

}  // namespace hpc
