// BF16 KV cache instantiation of the persistent attention kernel.
#include "attn_kernel.cuh"

namespace hpc {

// 4 stages x (16 KB K + 16 KB V + 2 KB Q): about 155 KB, one CTA per SM.
constexpr int kStagesBf16 = 4;

AttnConfig attn_config_bf16() {
    return {reinterpret_cast<const void *>(&attn_kernel<false, kStagesBf16>),
            AttnTraits<false, kStagesBf16>::kSmemBytes, kStagesBf16};
}

cudaError_t launch_attn_bf16(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &p,
                             int grid, cudaStream_t s) {
    constexpr int smem = AttnTraits<false, kStagesBf16>::kSmemBytes;
    attn_kernel<false, kStagesBf16><<<grid, kThreads, smem, s>>>(tk, tv, p);
    return cudaGetLastError();
}

}  // namespace hpc
