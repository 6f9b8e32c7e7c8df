"""GPU decode attention (plan + persistent attention + combine, through the
C ABI) against the fp64 oracle.

Small cases are compared element by element; the full-size workloads run in
the launch configuration the benchmark times (persistent CTAs = what the
device holds, floor 2) and are compared with the oracle on every row."""

import numpy as np
import pytest
import torch

import load_balanced_paged_assign_gb300 as hd
from _gpu import TOL, assert_close, assert_map_matches, device_ctas, oracle_out, run_step
from load_balanced_paged_assign_gb300.workloads import WORKLOADS, Workload, make_batch

pytestmark = pytest.mark.gpu

BOUNDARY_LENS = [1, 63, 64, 65, 127, 128, 129, 300, 1000, 4097]


def small(B, hq, hkv, kv_dtype="bf16", floor=2, ctas=0):
    return Workload("small", B, hq, hkv, seqlens=tuple([1] * B), kv_dtype=kv_dtype, seed=77,
                    min_tiles=floor, num_ctas=ctas)


def test_tiny_workload_full_parity():
    w = WORKLOADS["tiny"]
    batch = make_batch(w, device="cuda", poison_tail=True)
    out, ws = run_step(batch)
    assert_map_matches(ws, batch.seqlens.tolist(), w.num_kv_heads, w.num_ctas, w.min_tiles)
    assert_close(out, oracle_out(batch), "bf16")


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("hq,hkv", [(8, 1), (8, 2), (16, 2), (4, 1), (1, 1), (64, 8), (6, 3),
                                    (16, 1), (12, 1), (32, 2), (10, 1)])
@pytest.mark.parametrize("ctas", [1, 7, 0])
@pytest.mark.parametrize("fused", [True, False])
def test_small_shapes(kv_dtype, hq, hkv, ctas, fused):
    w = small(len(BOUNDARY_LENS), hq, hkv, kv_dtype, ctas=ctas)
    batch = make_batch(w, device="cuda", seqlens=BOUNDARY_LENS, poison_tail=True,
                       seed=100 + hq + hkv)
    out, _ = run_step(batch, fused=fused)
    assert_close(out, oracle_out(batch), kv_dtype)


WALK_CASES = [  # (B, Hkv, persistent CTAs, floor): up to 64 requests the first bin is walked
    (64, 1, 152, 1), (65, 1, 152, 1), (64, 4, 97, 2), (40, 2, 37, 1), (17, 8, 152, 3), (3, 1, 152, 1)]


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("case", range(len(WALK_CASES)))
def test_first_bins_derived_from_the_lengths(kv_dtype, case):
    """Mixed lengths with empty requests and a few long ones, so that many
    bins open with the short tail of a unit that began in the bin before:
    the CTAs stream their first bins before the task map is visible (walked
    from the lengths for up to 64 requests, the first descriptor only above).
    The map and the output match the oracles, the unit counters return to 0."""
    B, hkv, ctas, floor = WALK_CASES[case]
    rng = np.random.default_rng(3100 + case)
    lens = [int(x) for x in rng.integers(1, 1500, B)]
    for i in rng.choice(B, max(1, B // 8), replace=False):
        lens[int(i)] = 0
    for i in rng.choice(B, max(1, B // 16), replace=False):
        lens[int(i)] = int(rng.integers(8000, 40000))
    w = Workload(f"walk{case}", B, 8 * hkv, hkv, seqlens=tuple(lens), kv_dtype=kv_dtype,
                 seed=3200 + case, min_tiles=floor, num_ctas=ctas)
    batch = make_batch(w, device="cuda", poison_tail=True)
    out, ws = run_step(batch)
    assert_map_matches(ws, batch.seqlens.tolist(), hkv, ctas, floor)
    assert_close(out, oracle_out(batch), kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_fused_and_separate_combine_agree(kv_dtype):
    lens = [9000, 3, 64, 700, 129, 20000, 0, 65]
    w = small(len(lens), 8, 2, kv_dtype)
    batch = make_batch(w, device="cuda", seqlens=lens, seed=17)
    for ctas in (5, 33, 152):
        a, _ = run_step(batch, num_ctas=ctas, fused=True)
        b, _ = run_step(batch, num_ctas=ctas, fused=False)
        assert (a.float() - b.float()).abs().max().item() <= 2 ** -8


def test_fused_counters_survive_repeated_launches():
    # the map is reused by several launches (layers); counters reset themselves
    lens = [30000, 100, 5000, 64]
    w = small(len(lens), 8, 1)
    batch = make_batch(w, device="cuda", seqlens=lens, seed=23)
    ws = hd.Workspace(4, 8, 1, num_ctas=40)
    hd.hpc_decode_plan(batch.seqlens, 1, batch.max_pages, 40, 2, ws.tmap)
    outs = []
    for _ in range(3):
        ws.out.fill_(float("nan"))
        hd.hpc_decode_attn_combine(batch.q, None, batch.k_cache, batch.v_cache, 1.0, 1.0,
                                   batch.block_table, batch.seqlens, 8, 1, w.sm_scale, ws.tmap,
                                   ws.part_o, ws.part_lse, ws.unit_done, ws.out)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws.unit_done)) == 0
        outs.append(ws.out.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert_close(outs[0], oracle_out(batch), "bf16")


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("bins_per_cta", [2, 4])
def test_dynamic_bins_parity_and_counter_reset(kv_dtype, bins_per_cta):
    # more bins than resident CTAs: the persistent grid pulls the extra bins
    lens = [20000, 5, 3000, 64, 129, 70000, 0, 640, 1]
    w = small(len(lens), 8, 2, kv_dtype)
    batch = make_batch(w, device="cuda", seqlens=lens, poison_tail=True, seed=41)
    bins = bins_per_cta * device_ctas(kv_dtype) + 3
    ws = hd.Workspace(len(lens), 8, 2, num_ctas=bins)
    hd.hpc_decode_plan(batch.seqlens, 2, batch.max_pages, bins, 1, ws.tmap)
    ref = oracle_out(batch)
    outs = []
    for _ in range(3):  # the map is reused; the bin counter must come back to zero
        ws.out.fill_(float("nan"))
        hd.hpc_decode_attn_combine(batch.q, batch.q_scale, batch.k_cache, batch.v_cache,
                                   batch.k_scale, batch.v_scale, batch.block_table, batch.seqlens,
                                   8, 2, w.sm_scale, ws.tmap, ws.part_o, ws.part_lse, ws.unit_done,
                                   ws.out)
        torch.cuda.synchronize()
        meta = ws.tmap.meta.tolist()
        assert meta[3] == 0 and meta[4] == 0
        assert int(torch.count_nonzero(ws.unit_done)) == 0
        outs.append(ws.out[:len(lens)].clone())
    for o in outs:
        assert_close(o, ref, kv_dtype)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    unfused, _ = run_step(batch, num_ctas=bins, floor=1, fused=False)
    assert_close(unfused, ref, kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_more_owed_merges_than_the_end_list_holds(kv_dtype):
    """~54 one-tile bins per CTA over 4096 two-chunk units: a CTA completes
    ~27 split units, more than its end-of-stream list holds (16), so the
    combiner merges the rest at once.  Every row against the oracle, the
    output run to run bit for bit, the counters back at zero."""
    B, hkv = 2048, 2
    lens = [128] * B
    w = Workload("owed", B, 8 * hkv, hkv, seqlens=tuple(lens), kv_dtype=kv_dtype, seed=5200)
    batch = make_batch(w, device="cuda", poison_tail=True)
    bins = B * hkv * 2  # budget 1: every unit's two tiles land in two bins
    ws = hd.Workspace(B, 8 * hkv, hkv, num_ctas=bins)
    hd.hpc_decode_plan(batch.seqlens, hkv, batch.max_pages, bins, 1, ws.tmap)
    ref = oracle_out(batch)
    outs = []
    for _ in range(2):
        ws.out.fill_(float("nan"))
        hd.hpc_decode_attn_combine(batch.q, batch.q_scale, batch.k_cache, batch.v_cache,
                                   batch.k_scale, batch.v_scale, batch.block_table, batch.seqlens,
                                   8 * hkv, hkv, w.sm_scale, ws.tmap, ws.part_o, ws.part_lse,
                                   ws.unit_done, ws.out)
        torch.cuda.synchronize()
        meta = ws.tmap.meta.tolist()
        assert meta[1] == 1 and meta[3] == 0 and meta[4] == 0
        assert int(torch.count_nonzero(ws.unit_done)) == 0
        outs.append(ws.out[:B].clone())
    assert_close(outs[0], ref, kv_dtype)
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("floor", [0, 1, 4, 1000])
def test_floor_values(kv_dtype, floor):
    lens = [3000, 17, 64, 9000, 1]
    w = small(len(lens), 8, 1, kv_dtype, floor=floor)
    batch = make_batch(w, device="cuda", seqlens=lens, seed=5)
    out, ws = run_step(batch, num_ctas=40)
    assert_map_matches(ws, lens, 1, 40, floor)
    assert_close(out, oracle_out(batch), kv_dtype)


def test_length_one_returns_v_row_bitwise():
    w = small(3, 8, 1)
    batch = make_batch(w, device="cuda", seqlens=[1, 1, 1], seed=9)
    out, _ = run_step(batch)
    for r in range(3):
        page = int(batch.block_table[r, 0])
        v0 = batch.v_cache[page, 0, 0]
        for hq in range(8):
            assert torch.equal(out[r, hq], v0)


@pytest.mark.parametrize("fused", [True, False])
def test_constant_v_returns_that_row(fused):
    """Softmax weights sum to one, so a value row shared by every token comes
    back as that row: the kernel's fp32 sums differ from it by a few fp32
    ulps, far below half a BF16 ulp, so the BF16 output is the row itself."""
    w = small(4, 8, 2)
    batch = make_batch(w, device="cuda", seqlens=[77, 300, 4096, 1], seed=3)
    row = torch.linspace(-3, 3, 128, device="cuda").to(torch.bfloat16)
    batch.v_cache[:] = row
    out, _ = run_step(batch, num_ctas=16, fused=fused)
    err = (out.float() - row.float()).abs().max().item()
    assert err <= 1e-2
    assert torch.equal(out, row.expand_as(out))


@pytest.mark.parametrize("fused", [True, False])
def test_zero_length_requests_give_zero_rows(fused):
    lens = [0, 100, 0, 5000]
    w = small(4, 8, 1)
    batch = make_batch(w, device="cuda", seqlens=lens, seed=4)
    out, _ = run_step(batch, num_ctas=9, fused=fused)
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
    assert_close(out, oracle_out(batch), "bf16")


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_deterministic_and_page_permutation_invariant(kv_dtype):
    lens = [5000, 70, 1300, 64]
    w = small(4, 8, 2, kv_dtype)
    batch = make_batch(w, device="cuda", seqlens=lens, seed=6)
    a, _ = run_step(batch, num_ctas=20)
    b, _ = run_step(batch, num_ctas=20)
    assert torch.equal(a, b)
    P = batch.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(2)).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P, device="cuda")
    batch.k_cache = batch.k_cache[perm].contiguous()
    batch.v_cache = batch.v_cache[perm].contiguous()
    bt = batch.block_table.clone()
    live = bt >= 0
    bt[live] = inv[bt[live].long()].to(torch.int32)
    batch.block_table = bt
    c, _ = run_step(batch, num_ctas=20)
    assert torch.equal(a, c)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("S", [1, 3, 8])
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("hq", [16, 32])
def test_static_schedule_parity(kv_dtype, S, fused, hq):
    w = small(len(BOUNDARY_LENS), hq, 2, kv_dtype)
    batch = make_batch(w, device="cuda", seqlens=BOUNDARY_LENS, poison_tail=True, seed=11)
    out, ws = run_step(batch, num_splits=S, fused=fused)
    assert ws.tmap.to_host()["flags"] == 0
    assert_close(out, oracle_out(batch), kv_dtype)


def test_bad_page_is_flagged_not_read_out_of_bounds():
    w = small(2, 8, 1)
    batch = make_batch(w, device="cuda", seqlens=[200, 100], seed=8)
    batch.block_table[0, 1] = batch.num_pages + 5
    out, ws = run_step(batch, num_ctas=4)
    flags = hd.hpc_decode_read_meta(ws.tmap)[3]
    assert flags & hd.binding.HPC_FLAG_BAD_PAGE
    ref = oracle_out(make_batch(w, device="cuda", seqlens=[200, 100], seed=8))
    assert_close(out[1:], ref[1:], "bf16")  # the other request is unaffected


def _host_copy(t, pinned, shift):
    """A host copy of t: pinned or pageable; shift = 1 places it 4 bytes past a
    16-byte boundary (int32 / float32 arrays only)."""
    c = t.cpu().contiguous()
    if not shift:
        return c.pin_memory() if pinned else c.clone()
    flat = torch.empty(c.numel() + 4, dtype=c.dtype)
    if pinned:
        flat = flat.pin_memory()
    v = flat[1:1 + c.numel()].view(c.shape)
    v.copy_(c)
    return v


HOST_STEP_CASES = [("tiny", True, 0), ("tiny", False, 0), ("tiny", True, 1), ("fp8", True, 0),
                   ("fp8", True, 1), ("fp8", False, 0)]


@pytest.mark.parametrize("name,pinned,shift", HOST_STEP_CASES)
def test_host_buffer_step_matches_device_step(name, pinned, shift):
    """hpc_decode_step_host: pinned inputs are brought in by one copy kernel
    through their device aliases (16-byte vectors, or bytes where an address
    is not 16-byte aligned: shift moves the host lengths, block table and FP8
    scales 4 bytes off), pageable ones by the copy engine; the output is
    bit-identical to the device-buffer step."""
    w = WORKLOADS[name]
    batch = make_batch(w, device="cuda")
    ctas = w.num_ctas or device_ctas(w.kv_dtype)
    dev_out, _ = run_step(batch, num_ctas=ctas, fused=False)
    B, Hq, Hkv = w.batch, w.num_q_heads, w.num_kv_heads
    fp8 = w.kv_dtype == "e4m3"
    h_q = _host_copy(batch.q, pinned, 0)
    h_qs = _host_copy(batch.q_scale, pinned, shift) if fp8 else None
    h_sl = _host_copy(batch.seqlens, pinned, shift)
    h_bt = _host_copy(batch.block_table, pinned, shift)
    assert h_q.is_pinned() == pinned and h_bt.is_pinned() == pinned
    h_out = torch.empty((B, Hq, 128), dtype=torch.bfloat16).pin_memory()
    d_q, d_sl, d_bt = torch.empty_like(batch.q), torch.empty_like(batch.seqlens), \
        torch.empty_like(batch.block_table)
    d_qs = torch.empty_like(batch.q_scale) if fp8 else None
    ws = hd.Workspace(B, Hq, Hkv, num_ctas=ctas)
    hd.hpc_decode_step_host(h_q, h_qs, h_sl, h_bt, h_out, d_q, d_qs, d_sl, d_bt, ws.out,
                            batch.k_cache, batch.v_cache, batch.k_scale, batch.v_scale, Hq, Hkv,
                            w.sm_scale, ctas, w.min_tiles, 0, ws.tmap, ws.part_o, ws.part_lse)
    torch.cuda.synchronize()
    assert torch.equal(h_out.view(torch.int16), dev_out.cpu().view(torch.int16))
    assert torch.equal(d_bt.cpu(), batch.block_table.cpu())
    assert torch.equal(d_sl.cpu(), batch.seqlens.cpu())
    if fp8:
        assert torch.equal(d_qs.cpu(), batch.q_scale.cpu())


def full_size_parity(name, static_splits=()):
    """A full-size workload in the bench's launch configuration: the task map
    bit-exact, every output row against the oracle (dynamic schedule, and the
    static split-KV schedule for each S given)."""
    w = WORKLOADS[name]
    batch = make_batch(w, device="cuda", poison_tail=True)
    out, ws = run_step(batch)
    assert_map_matches(ws, batch.seqlens.tolist(), w.num_kv_heads,
                       w.num_ctas or device_ctas(w.kv_dtype), w.min_tiles)
    ref = oracle_out(batch)
    assert_close(out, ref, w.kv_dtype)
    for S in static_splits:
        static, _ = run_step(batch, num_splits=S)
        assert_close(static, ref, w.kv_dtype)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["hy3_tp8", "skewed", "uniform", "fp8"])
def test_full_size_workload_parity(name):
    full_size_parity(name)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["t3_64x0.5k", "t3_64x4k", "t3_32x0.125k_32x4k",
                                  "t3_2x32k_30x4k", "t3_1x64k_15x4k", "t3_1x128k_31x4k"])
def test_table3_mixes_parity(name):
    full_size_parity(name, static_splits=(4,))


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("B,hkv", [(1024, 1), (1025, 1), (2048, 1), (2048, 2), (3000, 1)])
def test_large_batches_through_the_step(kv_dtype, B, hkv):
    """Batches above 1024 requests: the attention CTAs no longer derive their
    first descriptor from the lengths and wait for the task map instead.  Short
    mixed lengths with empty requests and a few long ones; map bit-exact,
    every row against the oracle, fused and separate combine."""
    rng = np.random.default_rng(B + 7 * hkv)
    lens = [int(x) for x in rng.integers(1, 700, B)]
    for i in rng.choice(B, B // 10, replace=False):
        lens[int(i)] = 0
    for i in rng.choice(B, 4, replace=False):
        lens[int(i)] = int(rng.integers(5000, 30000))
    w = Workload(f"large{B}", B, 8 * hkv, hkv, seqlens=tuple(lens), kv_dtype=kv_dtype,
                 seed=4400 + B + hkv)
    batch = make_batch(w, device="cuda", poison_tail=True)
    ref = oracle_out(batch)
    for fused in (True, False):
        out, ws = run_step(batch, fused=fused)
        assert_map_matches(ws, lens, hkv, device_ctas(kv_dtype), w.min_tiles)
        assert_close(out, ref, kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("hq", [8, 16])
def test_unit_split_over_many_bins(kv_dtype, hq):
    """One 128K-token request beside two short ones, one KV head: the long
    unit is cut into ~147 chunks (more than 64, so the merges take every LSE
    round and every group of 32 chunks; with 16 query heads the two-row-block
    merge), fused and separate combine, every row against the oracle."""
    lens = [131072, 64, 3000]
    w = Workload(f"longunit{hq}", len(lens), hq, 1, seqlens=tuple(lens), kv_dtype=kv_dtype,
                 seed=5100 + hq)
    batch = make_batch(w, device="cuda", poison_tail=True)
    ref = oracle_out(batch)
    for fused in (True, False):
        out, ws = run_step(batch, fused=fused)
        assert_map_matches(ws, lens, 1, device_ctas(kv_dtype), w.min_tiles)
        assert max(ws.tmap.chunk_count[:len(lens)].tolist()) > 64
        assert_close(out, ref, kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("hq", [16, 12])
@pytest.mark.parametrize("fused", [True, False])
def test_group_of_up_to_sixteen_heads_full_size(kv_dtype, hq, fused):
    """GQA groups of 9 to 16 query heads per KV head (one descriptor serves the
    whole group, two blocks of eight query rows): the hy3_tp8 lengths, every
    row against the oracle."""
    base = WORKLOADS["hy3_tp8"]
    lens = make_batch(base, device="cpu").seqlens.tolist()
    w = Workload(f"g{hq}", len(lens), hq, 1, seqlens=tuple(lens), kv_dtype=kv_dtype,
                 seed=4500 + hq)
    batch = make_batch(w, device="cuda", poison_tail=True)
    out, ws = run_step(batch, fused=fused)
    assert_map_matches(ws, lens, 1, device_ctas(kv_dtype), w.min_tiles)
    assert_close(out, oracle_out(batch), kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_step_replays_from_a_cuda_graph(kv_dtype):
    # the step's launches (incl. the programmatic dependent ones) can be captured
    lens = [9000, 3, 640, 70000, 0, 129]
    w = small(len(lens), 8, 2, kv_dtype)
    batch = make_batch(w, device="cuda", seqlens=lens, seed=51)
    eager, _ = run_step(batch, num_ctas=40, floor=2)
    ws = hd.Workspace(len(lens), 8, 2, num_ctas=40)

    def step():
        hd.hpc_decode_step(batch.q, batch.q_scale, batch.k_cache, batch.v_cache, batch.k_scale,
                           batch.v_scale, batch.block_table, batch.seqlens, 8, 2, w.sm_scale, 40,
                           2, 0, ws.tmap, ws.part_o, ws.part_lse, ws.out, unit_done=ws.unit_done)

    step()  # one-time set-up outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(2):
        ws.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(ws.out[:len(lens)], eager)
        assert int(torch.count_nonzero(ws.unit_done)) == 0


def test_randomized_stress_against_oracle():
    # random shapes, lengths, floors and bin counts; fused and separate combine;
    # every case is checked against the oracle and re-run for bitwise equality
    rng = np.random.default_rng(2026)
    for case in range(30):
        kv_dtype = "e4m3" if rng.random() < 0.5 else "bf16"
        hkv = int(rng.choice([1, 2, 4]))
        hq = hkv * int(rng.choice([1, 2, 4, 8]))
        B = int(rng.integers(1, 24))
        lens = []
        for _ in range(B):
            kind = rng.random()
            lens.append(int(rng.integers(0, 3)) if kind < 0.1 else
                        int(rng.integers(1, 300)) if kind < 0.5 else
                        int(2 ** rng.uniform(8, 15)))
        floor = int(rng.choice([0, 1, 2, 8]))
        ctas = int(rng.choice([1, 13, 100, device_ctas(kv_dtype), 3 * device_ctas(kv_dtype) + 1]))
        fused = bool(rng.random() < 0.7)
        w = small(B, hq, hkv, kv_dtype, floor=floor)
        batch = make_batch(w, device="cuda", seqlens=lens, poison_tail=True, seed=500 + case)
        a, ws = run_step(batch, num_ctas=ctas, floor=floor, fused=fused)
        assert ws.tmap.to_host()["flags"] == 0
        b, _ = run_step(batch, num_ctas=ctas, floor=floor, fused=fused)
        assert torch.equal(a, b), f"case {case} not deterministic"
        assert_close(a, oracle_out(batch), kv_dtype)


@pytest.mark.parametrize("name", ["t4_8q1s1k", "t4_16q1s2k", "t4_32q1s1k", "t4_64q1s4k"])
def test_table4_decode_rows(name):
    """The decode rows of the vLLM comparison's Table 4 (Hq = 64, Hkv = 8):
    the task map bit-exact against the oracle, every output row, the dynamic
    and the static schedule."""
    full_size_parity(name, static_splits=(4,))


@pytest.mark.parametrize("name", ["hy3_tp8", "fp8"])
def test_packed_host_step_equals_the_device_step(name):
    """hpc_decode_step_host_packed: one input buffer brought in (a pinned one
    by a copy kernel through its device alias, a pageable one by the copy
    engine); the output, in a device buffer copied out or stored straight into
    pinned host memory, is bit-identical to the device-buffer step."""
    w = WORKLOADS[name]
    batch = make_batch(w, device="cuda")
    ref, _ = run_step(batch)
    fp8 = w.kv_dtype == "e4m3"
    B, Hq, Hkv, mp = w.batch, w.num_q_heads, w.num_kv_heads, batch.max_pages
    kvd = hd.HPC_KV_FP8_E4M3 if fp8 else hd.HPC_KV_BF16
    total, off = hd.hpc_decode_packed_layout(B, Hq, mp, kvd)
    h_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    h_in[off[0]:off[0] + batch.q.numel() * batch.q.element_size()] = \
        batch.q.cpu().contiguous().view(torch.uint8).reshape(-1)
    if fp8:
        h_in[off[1]:off[1] + B * Hq * 4] = batch.q_scale.cpu().contiguous().view(torch.uint8).reshape(-1)
    h_in[off[2]:off[2] + B * 4] = batch.seqlens.cpu().view(torch.uint8)
    h_in[off[3]:off[3] + B * mp * 4] = batch.block_table.cpu().contiguous().view(torch.uint8).reshape(-1)
    d_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    ctas = device_ctas(w.kv_dtype)
    ws = hd.Workspace(B, Hq, Hkv, num_ctas=ctas, device="cuda", kv_dtype=kvd)
    h_out = torch.empty((B, Hq, 128), dtype=torch.bfloat16).pin_memory()
    hd.hpc_decode_step_host_packed(h_in, d_in, h_out, ws.out, batch.k_cache, batch.v_cache,
                                   batch.k_scale, batch.v_scale, B, Hq, Hkv, mp, w.sm_scale, ctas,
                                   w.min_tiles, 0, ws.tmap, ws.part_o, ws.part_lse,
                                   unit_done=ws.unit_done)
    torch.cuda.synchronize()
    assert torch.equal(h_out.view(torch.int16), ref.cpu().view(torch.int16))
    # no device output: the kernels store straight into the pinned host buffer
    h_out2 = torch.full((B, Hq, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
    hd.hpc_decode_step_host_packed(h_in, d_in, h_out2, None, batch.k_cache, batch.v_cache,
                                   batch.k_scale, batch.v_scale, B, Hq, Hkv, mp, w.sm_scale, ctas,
                                   w.min_tiles, 0, ws.tmap, ws.part_o, ws.part_lse,
                                   unit_done=ws.unit_done)
    torch.cuda.synchronize()
    assert torch.equal(h_out2.view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(d_in.cpu(), h_in)  # every byte of the pinned input arrived
    # a pageable input buffer goes through the copy engine: the same output
    h_pageable = torch.empty(total, dtype=torch.uint8)
    h_pageable.copy_(h_in)
    assert not h_pageable.is_pinned()
    d_in.zero_()
    h_out3 = torch.full((B, Hq, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
    hd.hpc_decode_step_host_packed(h_pageable, d_in, h_out3, None, batch.k_cache, batch.v_cache,
                                   batch.k_scale, batch.v_scale, B, Hq, Hkv, mp, w.sm_scale, ctas,
                                   w.min_tiles, 0, ws.tmap, ws.part_o, ws.part_lse,
                                   unit_done=ws.unit_done)
    torch.cuda.synchronize()
    assert torch.equal(h_out3.view(torch.int16), ref.cpu().view(torch.int16))
    # a pageable output buffer has no device alias: refused, nothing launched
    with pytest.raises(hd.HpcError):
        hd.hpc_decode_step_host_packed(h_in, d_in, torch.empty((B, Hq, 128), dtype=torch.bfloat16),
                                       None, batch.k_cache, batch.v_cache, batch.k_scale,
                                       batch.v_scale, B, Hq, Hkv, mp, w.sm_scale, ctas, w.min_tiles,
                                       0, ws.tmap, ws.part_o, ws.part_lse, unit_done=ws.unit_done)
