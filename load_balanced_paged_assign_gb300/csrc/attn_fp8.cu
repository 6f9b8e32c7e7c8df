// FP8-E4M3 KV cache instantiation of the persistent attention kernel.
#include "attn_kernel.cuh"

namespace hpc {

// 8 stages x (8 KB K + 8 KB V + 1 KB Q): about 155 KB, one CTA per SM.
constexpr int kStagesFp8 = 8;

AttnConfig attn_config_fp8() {
    return {reinterpret_cast<const void *>(&attn_kernel<true, kStagesFp8>),
            AttnTraits<true, kStagesFp8>::kSmemBytes, kStagesFp8};
}

cudaError_t launch_attn_fp8(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &p,
                            int grid, cudaStream_t s) {
    constexpr int smem = AttnTraits<true, kStagesFp8>::kSmemBytes;
    attn_kernel<true, kStagesFp8><<<grid, kThreads, smem, s>>>(tk, tv, p);
    return cudaGetLastError();
}

}  // namespace hpc
