"""Pins for the fp64 attention oracle (CPU only).

What the oracle computes is decode attention of each new token over its
request's whole live KV cache (vLLM post, "The challenge: mixed-length decode
in every batch"), reading K/V in place through the block table (SGLang post,
"From HPC-Ops kernel to SGLang"), and the split-plus-combine identity behind
the persistent kernel (vLLM post, "Compute and combine").  Each pin below is
something other than the oracle itself: a library routine (torch's float8 and
bf16 casts, torch's scaled-dot-product attention in fp64 on contiguously
gathered K/V), a closed form, or an invariance of softmax attention.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from load_balanced_paged_assign_gb300.workloads import WORKLOADS, Workload, make_batch


def small_workload(B, hq, hkv, kv_dtype="bf16"):
    return Workload("t", B, hq, hkv, seqlens=tuple([1] * B), kv_dtype=kv_dtype, seed=5)


def run_oracle(batch, **extra):
    return oracle.attention(batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.seqlens,
                            **batch.oracle_kwargs(), **extra)


def dequant(t, scale=None):
    x = t.to(torch.float64)
    return x if scale is None else x * scale


def sdpa_reference(batch):
    """torch SDPA (fp64, CPU) on K/V gathered contiguously by torch indexing."""
    w = batch.workload
    G = w.group
    fp8 = w.kv_dtype == "e4m3"
    q = dequant(batch.q, batch.q_scale.to(torch.float64)[..., None] if fp8 else None)
    k_all = dequant(batch.k_cache, batch.k_scale if fp8 else None)
    v_all = dequant(batch.v_cache, batch.v_scale if fp8 else None)
    out = torch.zeros((len(batch.seqlens), w.num_q_heads, 128), dtype=torch.float64)
    for r, L in enumerate(batch.seqlens.tolist()):
        if L == 0:
            continue
        idx = torch.arange(L)
        pages = batch.block_table[r].long()[idx // 64]
        k = k_all[pages, idx % 64]  # [L, Hkv, D]
        v = v_all[pages, idx % 64]
        k = k.repeat_interleave(G, dim=1).transpose(0, 1)  # [Hq, L, D]
        v = v.repeat_interleave(G, dim=1).transpose(0, 1)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[r][:, None, :], k, v, scale=w.sm_scale)
        out[r] = o[:, 0, :]
    return out.numpy()


def test_e4m3_decoder_matches_torch_on_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(mine))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], mine[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


def test_bf16_decoder_matches_torch():
    bits = torch.randint(-32768, 32767, (5000,), generator=torch.Generator().manual_seed(3),
                         dtype=torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    mine = np.array([oracle.bf16_to_double(int(b) & 0xFFFF) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(ref[fin], mine[fin])
    assert np.array_equal(np.isnan(ref), np.isnan(mine))


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("hq,hkv", [(8, 1), (8, 2), (4, 4), (16, 1), (12, 1), (32, 2)])
def test_matches_library_sdpa(kv_dtype, hq, hkv):
    lens = [1, 63, 64, 65, 128, 129, 300, 0]
    w = small_workload(len(lens), hq, hkv, kv_dtype)
    batch = make_batch(w, seqlens=lens, seed=21 + hq + hkv)
    got = run_oracle(batch)
    ref = sdpa_reference(batch)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_length_one_returns_v0_exactly():
    w = small_workload(3, 8, 1)
    batch = make_batch(w, seqlens=[1, 1, 1], seed=2)
    got = run_oracle(batch)
    for r in range(3):
        page = int(batch.block_table[r, 0])
        v0 = batch.v_cache[page, 0, 0].to(torch.float64).numpy()
        for hq in range(8):
            assert np.array_equal(got[r, hq], v0)


def test_constant_v_returns_that_row():
    w = small_workload(2, 8, 2)
    batch = make_batch(w, seqlens=[77, 300], seed=4)
    row = torch.linspace(-3, 3, 128).to(torch.bfloat16)
    batch.v_cache[:] = row
    got = run_oracle(batch)
    np.testing.assert_allclose(got, np.broadcast_to(row.double().numpy(), got.shape), atol=1e-13)


def test_zero_query_gives_mean_of_v():
    w = small_workload(2, 8, 1)
    batch = make_batch(w, seqlens=[130, 64], seed=6)
    batch.q.zero_()
    got = run_oracle(batch)
    for r, L in enumerate([130, 64]):
        idx = torch.arange(L)
        pages = batch.block_table[r].long()[idx // 64]
        mean = batch.v_cache[pages, idx % 64, 0].double().mean(0).numpy()
        for hq in range(8):
            np.testing.assert_allclose(got[r, hq], mean, atol=1e-13)


def test_zero_length_request_gives_zeros():
    w = small_workload(2, 8, 1)
    batch = make_batch(w, seqlens=[0, 100], seed=8)
    got = run_oracle(batch)
    assert np.all(got[0] == 0.0)
    assert np.any(got[1] != 0.0)


def test_page_permutation_invariance():
    w = small_workload(3, 8, 2)
    batch = make_batch(w, seqlens=[200, 64, 513], seed=9)
    ref = run_oracle(batch)
    P = batch.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(1))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    batch.k_cache = batch.k_cache[perm].contiguous()  # new page i holds old page perm[i]
    batch.v_cache = batch.v_cache[perm].contiguous()
    bt = batch.block_table.clone()
    live = bt >= 0
    bt[live] = inv[bt[live].long()].to(torch.int32)
    batch.block_table = bt
    got = run_oracle(batch)
    assert np.array_equal(got, ref)


def test_shift_of_all_keys_leaves_output_unchanged():
    # adding the same vector c to every key shifts all scores of a head by
    # q.c, which softmax cancels; integer keys and c = 1 keep bf16 exact
    w = small_workload(2, 8, 1)
    batch = make_batch(w, seqlens=[150, 64], seed=10)
    kq = batch.k_cache.double().round().clamp(-8, 8)
    batch.k_cache = kq.to(torch.bfloat16)
    base = run_oracle(batch)
    batch.k_cache = (kq + 1.0).to(torch.bfloat16)
    moved = run_oracle(batch)
    np.testing.assert_allclose(moved, base, rtol=0, atol=1e-12)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_split_plus_combine_equals_unsplit(kv_dtype):
    lens = [1, 64, 65, 700, 2000, 0, 129]
    w = small_workload(len(lens), 8, 2, kv_dtype)
    batch = make_batch(w, seqlens=lens, seed=12)
    unsplit = run_oracle(batch)
    for ctas, floor in [(5, 1), (40, 2), (3, 7)]:
        tm = oracle.assign_closed_form(lens, 2, ctas, floor)
        split = oracle.split_attention(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                                       batch.seqlens, tm, **batch.oracle_kwargs())
        np.testing.assert_allclose(split, unsplit, rtol=0, atol=1e-12)
    st = oracle.static_plan(lens, 2, 4)
    split = oracle.split_attention(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                                   batch.seqlens, st, **batch.oracle_kwargs())
    np.testing.assert_allclose(split, unsplit, rtol=0, atol=1e-12)


def test_poisoned_tail_slots_are_never_read():
    w = small_workload(3, 8, 1, "e4m3")
    lens = [70, 1, 127]
    batch = make_batch(w, seqlens=lens, seed=13, poison_tail=True)
    got = run_oracle(batch)
    assert np.all(np.isfinite(got))
    clean = make_batch(w, seqlens=lens, seed=13, poison_tail=False)
    assert np.array_equal(run_oracle(clean), got)


def test_combine_of_disjoint_halves():
    # two partials of equal LSE average; a -inf partial carries no weight
    parts = np.array([[1.0] * 128, [3.0] * 128, [100.0] * 128])
    out = oracle.combine(parts, np.array([0.5, 0.5, -math.inf]))
    np.testing.assert_allclose(out, 2.0, atol=1e-15)
    out = oracle.combine(parts[:2], np.array([math.log(3.0), 0.0]))
    np.testing.assert_allclose(out, (3 * 1.0 + 1 * 3.0) / 4, atol=1e-15)


def test_sampled_rows_match_full():
    w = WORKLOADS["tiny"]
    batch = make_batch(w)
    full = run_oracle(batch)
    rows = [0, 9, 17, 31]
    got = run_oracle(batch, rows=rows)
    for i, row in enumerate(rows):
        assert np.array_equal(got[i], full.reshape(-1, 128)[row])


# ------------------------------------------------------- multi-query decode
# q_len new query tokens per request (the last q_len live tokens); query
# token i sees the live tokens j < L - q_len + 1 + i.

def mq_batch(kv_dtype, q_len, lens, hq=8, hkv=2, seed=21):
    w = Workload("mq", len(lens), hq, hkv, seqlens=tuple(lens), kv_dtype=kv_dtype, seed=seed,
                 q_len=q_len)
    return make_batch(w, poison_tail=True)


def run_mq(batch, **extra):
    return oracle.attention_mq(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                               batch.seqlens, batch.workload.q_len, **batch.oracle_kwargs(),
                               **extra)


def sdpa_causal_reference(batch):
    """torch SDPA (fp64) with an explicit mask: query i sees keys j <= L - q_len + i."""
    w = batch.workload
    G, ql = w.group, w.q_len
    fp8 = w.kv_dtype == "e4m3"
    q = dequant(batch.q, batch.q_scale.to(torch.float64)[..., None] if fp8 else None)
    k_all = dequant(batch.k_cache, batch.k_scale if fp8 else None)
    v_all = dequant(batch.v_cache, batch.v_scale if fp8 else None)
    out = np.zeros((len(batch.seqlens), ql, w.num_q_heads, 128))
    for r, L in enumerate(batch.seqlens.tolist()):
        idx = torch.arange(L)
        pages = batch.block_table[r].long()[idx // 64]
        k = k_all[pages, idx % 64].repeat_interleave(G, dim=1).transpose(0, 1)  # [Hq, L, D]
        v = v_all[pages, idx % 64].repeat_interleave(G, dim=1).transpose(0, 1)
        mask = idx[None, :] <= (L - ql + torch.arange(ql))[:, None]  # [q_len, L]
        o = torch.nn.functional.scaled_dot_product_attention(
            q[r].transpose(0, 1), k, v, attn_mask=mask, scale=w.sm_scale)  # [Hq, q_len, D]
        out[r] = o.transpose(0, 1).numpy()
    return out


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("q_len,hq,hkv", [(2, 8, 2), (3, 4, 4), (4, 4, 1), (2, 16, 2)])
def test_multi_query_matches_library_sdpa_with_causal_mask(kv_dtype, q_len, hq, hkv):
    lens = [q_len, 63 + q_len, 64, 65, 129, 200]
    batch = mq_batch(kv_dtype, q_len, lens, hq, hkv)
    got = run_mq(batch)
    ref = sdpa_causal_reference(batch)
    assert np.allclose(got, ref, atol=1e-12, rtol=1e-10)


def test_multi_query_single_token_is_plain_decode():
    w = Workload("mq1", 5, 8, 2, seqlens=(1, 64, 65, 300, 1000), seed=23)
    batch = make_batch(w)
    got = oracle.attention_mq(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                              batch.seqlens, 1, **batch.oracle_kwargs())
    assert np.array_equal(got[:, 0], run_oracle(batch))


def test_multi_query_closed_forms():
    # the first query of a request of exactly q_len tokens sees only token 0:
    # its output is v_0 of its KV head; the last query sees every token
    q_len = 3
    batch = mq_batch("bf16", q_len, [q_len, 70], hq=4, hkv=2)
    out = run_mq(batch)
    v = batch.v_cache.to(torch.float64)
    p0 = int(batch.block_table[0, 0])
    for hq in range(4):
        assert np.array_equal(out[0, 0, hq], v[p0, 0, hq // 2].numpy())
    # a request shorter than q_len: queries with no visible token give zeros
    short = mq_batch("bf16", 4, [2, 5], hq=4, hkv=1)
    out = run_mq(short)
    assert not out[0, :2].any() and out[0, 2:].any()


def test_multi_query_rows_match_full():
    batch = mq_batch("e4m3", 2, [64, 130, 7], hq=8, hkv=1)
    full = run_mq(batch).reshape(-1, 128)
    rows = [0, 5, 17, 31, 47]
    assert np.array_equal(run_mq(batch, rows=rows), full[rows])


# ------------------------------------------------------- extend / prefill
# Many query tokens per request (the vLLM post's Table 4 prefill and extend
# rows): the same rule at q_len in the hundreds, several 128-token query
# blocks, prefills (L = q_len) and extends over a cached prefix.

@pytest.mark.parametrize("q_len,lens", [(200, [200]), (130, [130, 400]), (300, [257, 300, 700])])
def test_prefill_and_extend_match_library_sdpa_with_causal_mask(q_len, lens):
    batch = mq_batch("bf16", q_len, lens, hq=4, hkv=2, seed=31)
    got = run_mq(batch, num_threads=4)
    ref = sdpa_causal_reference(batch)
    assert np.allclose(got, ref, atol=1e-12, rtol=1e-10)


def test_prefill_first_query_sees_only_the_first_token():
    q_len = 150
    batch = mq_batch("bf16", q_len, [q_len], hq=4, hkv=1, seed=33)
    out = run_mq(batch, rows=[0, 1, 2, 3])  # query 0, every head
    v0 = batch.v_cache.to(torch.float64)[int(batch.block_table[0, 0]), 0, 0].numpy()
    for h in range(4):
        assert np.array_equal(out[h], v0)
