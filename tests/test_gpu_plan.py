"""GPU assign kernel and static plan vs the task-map oracle, bit for bit."""

import random

import pytest
import torch

import load_balanced_paged_assign_gb300 as hd
import oracle
from load_balanced_paged_assign_gb300.workloads import WORKLOADS, draw_seqlens

pytestmark = pytest.mark.gpu


def plan(seqlens, Hkv, num_ctas, floor, max_pages=None):
    lens = torch.tensor(list(seqlens), dtype=torch.int32, device="cuda")
    B = len(seqlens)
    if max_pages is None:
        max_pages = max([(L + 63) // 64 for L in seqlens] + [1])
    tm = hd.TaskMap.dynamic(B, Hkv, num_ctas)
    tm.bin_ptr.fill_(-7)
    tm.desc.fill_(-7)
    hd.hpc_decode_plan(lens, Hkv, max_pages, num_ctas, floor, tm)
    torch.cuda.synchronize()
    return tm.to_host()


def check(seqlens, Hkv, num_ctas, floor):
    got = plan(seqlens, Hkv, num_ctas, floor)
    ref = oracle.assign_closed_form(list(seqlens), Hkv, num_ctas, floor)
    assert got["flags"] == 0
    assert (got["total_tiles"], got["budget"], got["num_desc"]) == \
        (ref.total_tiles, ref.budget, ref.num_desc)
    assert got["desc"] == ref.desc
    assert got["bin_ptr"] == ref.bin_ptr
    assert got["chunk_count"] == ref.chunk_count
    assert got["chunk_off"] == ref.chunk_off


def test_worked_example():
    got = plan([64, 200, 1000, 2048], 1, 132, 2)
    assert got["num_desc"] == 30 and got["budget"] == 2 and got["total_tiles"] == 53
    assert got["chunk_count"] == [1, 3, 9, 17]
    assert got["desc"][:5] == [(0, 0, 0, 1), (0, 1, 0, 1), (0, 1, 1, 3), (0, 1, 3, 4),
                               (0, 2, 0, 1)]
    assert got["desc"][-1] == (0, 3, 31, 32)
    assert got["bin_ptr"][27:] == [30] * 106
    check([64, 200, 1000, 2048], 1, 132, 2)


@pytest.mark.parametrize("seqlens,hkv,ctas,floor", [
    ([1], 1, 4, 1), ([64], 1, 4, 1), ([65], 1, 4, 1),
    ([1, 63, 64, 65, 128, 129], 2, 5, 1),
    ([0, 5, 0, 300], 2, 3, 2),
    ([0, 0, 0], 4, 8, 2),
    ([4096] * 8, 8, 16, 2),
    ([131072] + [4096] * 31, 1, 152, 2),
    ([100] * 3, 1, 1000, 2),
    ([8192] * 16, 8, 1, 2),
    ([10, 20000, 30, 70000, 5], 3, 7, 50),
    ([], 1, 152, 2),
])
def test_edge_cases(seqlens, hkv, ctas, floor):
    check(seqlens, hkv, ctas, floor)


def test_random_maps():
    rng = random.Random(1234)
    for _ in range(200):
        B = rng.randint(1, 40)
        hkv = rng.choice([1, 2, 4, 8])
        ctas = rng.choice([1, 2, 17, 132, 152, 304, 1000])
        floor = rng.choice([0, 1, 2, 3, 8, 64])
        lens = [rng.choice([0, 1, 63, 64, 65, rng.randint(1, 5000), int(2 ** rng.uniform(0, 17))])
                for _ in range(B)]
        check(lens, hkv, ctas, floor)


def test_large_batch_multi_chunk_scans():
    rng = random.Random(99)
    lens = [rng.randint(0, 700) for _ in range(5000)]
    check(lens, 2, 152, 2)
    check(lens, 3, 2000, 1)


@pytest.mark.parametrize("name", ["tiny", "hy3_tp8", "skewed", "uniform", "fp8",
                                  "t3_1x128k_31x4k"])
def test_workload_maps(name):
    w = WORKLOADS[name]
    lens = draw_seqlens(w, torch.Generator().manual_seed(w.seed))
    for ctas in sorted({w.num_ctas or 152, 132, 152, 304}):
        check(lens, w.num_kv_heads, ctas, w.min_tiles)


def test_bad_seqlen_is_clamped_and_flagged():
    lens = torch.tensor([100, 5000, -3], dtype=torch.int32, device="cuda")
    tm = hd.TaskMap.dynamic(3, 1, 8)
    hd.hpc_decode_plan(lens, 1, 4, 8, 1, tm)  # 4 pages hold at most 256 tokens
    got = tm.to_host()
    assert got["flags"] & hd.binding.HPC_FLAG_BAD_SEQLEN
    ref = oracle.assign_closed_form([100, 256, 0], 1, 8, 1)
    assert got["desc"] == ref.desc and got["bin_ptr"] == ref.bin_ptr


@pytest.mark.parametrize("S", [1, 2, 3, 8, 32])
def test_static_plan(S):
    rng = random.Random(S)
    for _ in range(20):
        B = rng.randint(1, 20)
        hkv = rng.choice([1, 2, 8])
        lens = [rng.choice([0, 1, 64, 65, 700, 4096, rng.randint(1, 40000)]) for _ in range(B)]
        t = torch.tensor(lens, dtype=torch.int32, device="cuda")
        tm = hd.TaskMap.static(B, hkv, S)
        hd.hpc_decode_plan_static(t, hkv, max((L + 63) // 64 for L in lens + [1]), S, tm)
        got = tm.to_host()
        ref = oracle.static_plan(lens, hkv, S)
        assert got["flags"] == 0
        assert got["desc"] == ref.desc
        assert got["bin_ptr"] == ref.bin_ptr
        assert got["chunk_count"] == ref.chunk_count
        assert got["chunk_off"] == ref.chunk_off
