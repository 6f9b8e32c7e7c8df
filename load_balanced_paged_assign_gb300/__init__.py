"""GB300-native load-balanced paged GQA decode attention.

CUDA kernels behind a C ABI (include/hpc_decode.h, libhpcdecode.so): the
fused prologue (QK-Norm, RoPE, paged KV write, FP8 query) produces the
attention inputs; the assign kernel builds a per-step task map of balanced
tile bins, the persistent attention kernel drains the bins into split
partials, and the combine kernel merges them into BF16 output.  Beside the
decode path: extend / prefill attention on tcgen05 tensor cores and the
router GEMM with a BF16 hi/lo split of FP32 weights.  This package
holds the build step, the ctypes binding and the seeded workload generators.
"""

from .binding import (EXPORTS, HPC_KV_BF16, HPC_KV_FP8_E4M3, HPC_ROPE_HALVES,
                      HPC_ROPE_INTERLEAVED, HpcError, TaskMap, Workspace, hpc_decode_attn,
                      hpc_decode_attn_combine, hpc_decode_attn_combine_mq, hpc_decode_attn_mq,
                      hpc_decode_combine, hpc_decode_combine_mq, hpc_decode_desc_capacity,
                      hpc_decode_num_ctas, hpc_decode_plan, hpc_decode_plan_static,
                      hpc_decode_read_meta, hpc_decode_static_capacity, hpc_decode_step,
                      hpc_decode_step_mq,
                      hpc_decode_packed_layout, hpc_decode_step_host,
                      hpc_decode_step_host_packed, hpc_decode_version, hpc_prefill_attn,
                      hpc_rope_frequencies, hpc_rope_norm, hpc_router_gemm, hpc_router_plan, hpc_router_split, hpc_router_workspace_bytes,
                      hpc_selftest_wait_timeout,
                      kv_dtype_of, lib)

__all__ = [
    "EXPORTS", "HPC_KV_BF16", "HPC_KV_FP8_E4M3", "HPC_ROPE_HALVES", "HPC_ROPE_INTERLEAVED",
    "HpcError", "TaskMap", "Workspace", "hpc_decode_attn", "hpc_decode_attn_combine",
    "hpc_decode_attn_combine_mq", "hpc_decode_attn_mq", "hpc_decode_combine",
    "hpc_decode_combine_mq", "hpc_decode_desc_capacity", "hpc_decode_num_ctas",
    "hpc_decode_plan", "hpc_decode_plan_static", "hpc_decode_read_meta",
    "hpc_decode_packed_layout", "hpc_decode_static_capacity", "hpc_decode_step",
    "hpc_decode_step_host", "hpc_decode_step_host_packed", "hpc_decode_step_mq",
    "hpc_decode_version", "hpc_prefill_attn", "hpc_rope_frequencies", "hpc_rope_norm", "hpc_router_gemm",
    "hpc_router_plan", "hpc_router_split", "hpc_router_workspace_bytes", "hpc_selftest_wait_timeout",
    "kv_dtype_of", "lib",
]
