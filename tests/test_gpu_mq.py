"""Multi-query decode (q_len query tokens per request, causal among them)
through the C ABI against the fp64 oracle (oracle.attention_mq): small
shapes on both row-block paths (q_len * G <= 8 and <= 16), both KV dtypes,
the fused and the separate combine, short requests (L < q_len), the static
plan, q_len = 1 against the plain step, full-size MTP batches compared on
every row, and a batch of 2000 requests."""

import dataclasses

import numpy as np
import pytest
import torch

import load_balanced_paged_assign_gb300 as hd
import oracle
from _gpu import TOL, assert_close, device_ctas, run_step
from load_balanced_paged_assign_gb300.workloads import WORKLOADS, Workload, make_batch

pytestmark = pytest.mark.gpu


def run_step_mq(batch, num_ctas=None, floor=2, num_splits=0, fused=True):
    w = batch.workload
    B = int(batch.seqlens.numel())
    if num_ctas is None:
        num_ctas = device_ctas(w.kv_dtype)
    ws = hd.Workspace(B, w.num_q_heads, w.num_kv_heads, num_ctas=num_ctas, num_splits=num_splits,
                      device="cuda", q_len=w.q_len)
    ws.out.fill_(float("nan"))
    hd.hpc_decode_step_mq(batch.q, batch.q_scale, batch.k_cache, batch.v_cache, batch.k_scale,
                          batch.v_scale, batch.block_table, batch.seqlens, w.num_q_heads,
                          w.num_kv_heads, w.q_len, w.sm_scale, num_ctas, floor, num_splits,
                          ws.tmap, ws.part_o, ws.part_lse, ws.out,
                          unit_done=ws.unit_done if fused else None)
    torch.cuda.synchronize()
    if fused:
        assert int(torch.count_nonzero(ws.unit_done)) == 0
    assert ws.tmap.to_host()["flags"] == 0
    return ws.out[:B], ws


def oracle_mq(batch, rows=None):
    return oracle.attention_mq(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                               batch.seqlens, batch.workload.q_len, rows=rows,
                               **batch.oracle_kwargs())


SHAPES = [  # (Hq, Hkv, q_len): rows per KV head q_len * Hq / Hkv
    (8, 1, 2), (8, 2, 2), (4, 1, 3), (4, 4, 4), (16, 2, 2), (8, 1, 1), (2, 1, 8), (6, 2, 5),
]


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
@pytest.mark.parametrize("fused", [True, False])
def test_small_shapes_against_oracle(kv_dtype, shape, fused):
    hq, hkv, q_len = SHAPES[shape]
    lens = [q_len, 1, 63, 64, 65, 129 + q_len, 700, 2000, max(q_len - 1, 0), 3000]
    w = Workload(f"mq{shape}", len(lens), hq, hkv, seqlens=tuple(lens), kv_dtype=kv_dtype,
                 seed=300 + shape, q_len=q_len)
    batch = make_batch(w, device="cuda", poison_tail=True)
    ref = oracle_mq(batch)
    for ctas in (13, device_ctas(kv_dtype)):
        got, _ = run_step_mq(batch, num_ctas=ctas, fused=fused)
        assert_close(got.reshape(-1, 128), ref.reshape(-1, 128), kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_static_plan(kv_dtype):
    lens = [5, 300, 1000, 4097]
    w = Workload("mqs", len(lens), 8, 1, seqlens=tuple(lens), kv_dtype=kv_dtype, seed=41, q_len=2)
    batch = make_batch(w, device="cuda", poison_tail=True)
    got, _ = run_step_mq(batch, num_splits=4)
    assert_close(got.reshape(-1, 128), oracle_mq(batch).reshape(-1, 128), kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_single_query_equals_the_plain_step(kv_dtype):
    w = Workload("mq1", 6, 8, 1, seqlens=(1, 64, 65, 500, 3000, 9000), kv_dtype=kv_dtype, seed=43)
    batch = make_batch(w, device="cuda")
    got, _ = run_step_mq(batch)
    ref, _ = run_step(batch)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_rows_without_a_visible_token_are_zero():
    w = Workload("mqz", 3, 4, 1, seqlens=(1, 3, 10), seed=45, q_len=4)  # 16 rows per KV head
    batch = make_batch(w, device="cuda")
    got, _ = run_step_mq(batch)
    assert not got[0, :3].float().abs().sum() and not got[1, :1].float().abs().sum()
    assert torch.isfinite(got.float()).all()
    assert_close(got.reshape(-1, 128), oracle_mq(batch).reshape(-1, 128), "bf16")


@pytest.mark.parametrize("name", ["hy3_tp8", "fp8", "skewed"])
def test_full_size_mtp_batch(name):
    """The workload's own lengths with one draft token (q_len = 2): G = 8 gives
    16 query rows per KV head, the two-block path.  Every row against the
    oracle."""
    w = dataclasses.replace(WORKLOADS[name], q_len=2)
    batch = make_batch(w, device="cuda", poison_tail=True)
    got, _ = run_step_mq(batch)
    assert_close(got.reshape(-1, 128), oracle_mq(batch).reshape(-1, 128), w.kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_large_batch_mtp(kv_dtype):
    """2000 requests with two query tokens each (above 1024 the CTAs wait for
    the task map instead of deriving their first descriptor), short mixed
    lengths with some shorter than q_len and a few long ones."""
    rng = np.random.default_rng(77)
    lens = [int(x) for x in rng.integers(0, 600, 2000)]
    for i in rng.choice(2000, 3, replace=False):
        lens[int(i)] = int(rng.integers(5000, 20000))
    w = Workload("mqbig", len(lens), 8, 1, seqlens=tuple(lens), kv_dtype=kv_dtype, seed=4600,
                 q_len=2)
    batch = make_batch(w, device="cuda", poison_tail=True)
    ref = oracle_mq(batch)
    for fused in (True, False):
        got, _ = run_step_mq(batch, fused=fused)
        assert_close(got.reshape(-1, 128), ref.reshape(-1, 128), kv_dtype)


def test_repeated_launches_are_bitwise_identical():
    w = dataclasses.replace(WORKLOADS["hy3_tp8"], q_len=2)
    batch = make_batch(w, device="cuda")
    a, _ = run_step_mq(batch)
    b, _ = run_step_mq(batch)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
