"""hpc_decode_step_noalloc: the decode step for callers that cannot allocate
device memory (its task map and partials live in an array built into the
library).  Called through the C ABI on two calls in a row with different
batches — the second call runs on whatever the first left in the shared
array — and checked against the fp64 oracle and, bit for bit, against
hpc_decode_step with caller-allocated scratch running the same kernels
(load-balanced plan, attention, separate combine kernel).  Kept in a file
collected last."""

import pytest
import torch

import load_balanced_paged_assign_gb300 as hd
from _gpu import assert_close, device_ctas, oracle_out, run_step
from load_balanced_paged_assign_gb300.workloads import WORKLOADS, Workload, make_batch

pytestmark = pytest.mark.gpu


def noalloc(batch, num_ctas, floor):
    w = batch.workload
    B = int(batch.seqlens.numel())
    out = torch.full((B, w.num_q_heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    meta = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    hd.binding.hpc_decode_step_noalloc(batch.q, batch.q_scale, batch.k_cache, batch.v_cache,
                                       batch.k_scale, batch.v_scale, batch.block_table,
                                       batch.seqlens, w.num_q_heads, w.num_kv_heads, w.sm_scale,
                                       num_ctas, floor, out, meta)
    torch.cuda.synchronize()
    return out, meta.tolist()


def check_against_step(batch, num_ctas, floor):
    # the allocating step on the kernels the no-alloc step runs: the combine as
    # its own kernel (no unit counters), so the outputs must agree bit for bit
    ref, ws = run_step(batch, num_ctas=num_ctas, floor=floor, fused=False)
    got, meta = noalloc(batch, num_ctas, floor)
    assert meta == ws.tmap.meta.tolist()[:4]
    assert meta[3] == 0
    assert torch.isfinite(got).all()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert_close(got, oracle_out(batch), batch.workload.kv_dtype)


def test_two_calls_in_a_row_match_the_allocating_entry_point():
    first = make_batch(WORKLOADS["hy3_tp8"], device="cuda")
    check_against_step(first, device_ctas("bf16"), 2)
    lens = [5000, 1, 64, 65, 130000, 700, 0, 4096]
    w = Workload("mixed_fp8", len(lens), 8, 1, seqlens=tuple(lens), kv_dtype="e4m3", seed=31)
    second = make_batch(w, device="cuda", poison_tail=True)
    check_against_step(second, 40, 1)


def test_sixteen_head_groups_and_large_batches():
    """Groups of 16 query heads per KV head (twice the partial rows per
    descriptor) and a batch of 1500 requests (the CTAs wait for the task map
    instead of deriving their first descriptor), both within the built-in
    scratch."""
    lens = [3000, 1, 64, 130, 20000, 0, 777]
    w = Workload("na16", len(lens), 16, 1, seqlens=tuple(lens), seed=61)
    check_against_step(make_batch(w, device="cuda", poison_tail=True), device_ctas("bf16"), 2)
    lens = [int(x) for x in torch.randint(0, 300, (1500,), generator=torch.Generator().manual_seed(5))]
    w = Workload("na1500", len(lens), 8, 1, seqlens=tuple(lens), kv_dtype="e4m3", seed=62)
    check_against_step(make_batch(w, device="cuda", poison_tail=True), device_ctas("e4m3"), 2)


def test_too_large_a_problem_is_rejected_before_launch():
    w = WORKLOADS["tiny"]
    batch = make_batch(w, device="cuda")
    B = int(batch.seqlens.numel())
    out = torch.empty((B, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(hd.HpcError) as e:
        # 100,000 persistent CTAs would need far more descriptors than fit
        hd.binding.hpc_decode_step_noalloc(batch.q, None, batch.k_cache, batch.v_cache, 1.0, 1.0,
                                           batch.block_table, batch.seqlens, 8, 1, w.sm_scale,
                                           100000, 2, out)
    assert e.value.status == hd.binding.HPC_ERR_WORKSPACE
