"""Extend / prefill attention (hpc_prefill_attn, tcgen05 tensor cores) through
the C ABI against the fp64 oracle (oracle.attention_mq: query token i of
request r sees the live tokens j < L_r - q_len + 1 + i).

Small shapes are compared in full: one and several 128-token query blocks
with a ragged last block, prefills (L = q_len) at every tile-boundary length,
extends over short and long cached prefixes, rows that see no token (L <
q_len), groups G = 1 .. 16, NaN-poisoned free slots in the last pages.  The
Table-4 shapes of the vLLM post are compared on sampled rows that include the
first and last query tokens and the 128-token block edges.  Plus seeded
random batches, run-to-run determinism, page-permutation invariance and the
kernel's own flags for bad lengths and pages."""

import numpy as np
import pytest
import torch

import load_balanced_paged_assign_gb300 as hd
import oracle
from _gpu import assert_close
from load_balanced_paged_assign_gb300.workloads import WORKLOADS, Workload, make_batch

pytestmark = pytest.mark.gpu


def run_prefill(batch, flags=None):
    w = batch.workload
    B = int(batch.seqlens.numel())
    out = torch.full((B, w.q_len, w.num_q_heads, 128), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    own = flags is None
    if own:
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    hd.hpc_prefill_attn(batch.q, batch.k_cache, batch.v_cache, batch.block_table, batch.seqlens,
                        w.num_q_heads, w.num_kv_heads, w.q_len, w.sm_scale, out, flags=flags)
    torch.cuda.synchronize()
    if own:
        assert int(flags.item()) == 0
    return out


def oracle_rows(batch, rows=None):
    return oracle.attention_mq(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                               batch.seqlens, batch.workload.q_len, rows=rows,
                               **batch.oracle_kwargs())


def small(name, lens, hq, hkv, q_len, seed):
    w = Workload(name, len(lens), hq, hkv, seqlens=tuple(lens), seed=seed, q_len=q_len)
    # q must be [B, q_len, Hq, 128] even for q_len = 1
    batch = make_batch(w, device="cuda", poison_tail=True)
    if q_len == 1:
        batch.q = batch.q.reshape(len(lens), 1, hq, 128)
    return batch


PREFILL_LENS = [1, 5, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300]


@pytest.mark.parametrize("L", PREFILL_LENS)
def test_prefill_single_request(L):
    batch = small(f"pf{L}", [L], 8, 1, L, 500 + L)
    got = run_prefill(batch)
    assert_close(got.reshape(-1, 128), oracle_rows(batch).reshape(-1, 128), "bf16")


EXTEND = [  # (lens, Hq, Hkv, q_len)
    ([100, 250, 700], 8, 2, 100),
    ([130, 5000], 4, 1, 130),
    ([300, 301, 1000, 4097], 2, 2, 300),
    ([50, 10, 200], 4, 4, 100),     # L < q_len: the first rows see nothing
    ([64, 640], 16, 1, 64),
    ([1000], 16, 16, 7),
    ([2000, 129], 6, 2, 129),
]


@pytest.mark.parametrize("case", range(len(EXTEND)))
def test_extend_against_oracle(case):
    lens, hq, hkv, q_len = EXTEND[case]
    batch = small(f"ex{case}", lens, hq, hkv, q_len, 600 + case)
    got = run_prefill(batch)
    ref = oracle_rows(batch)
    assert_close(got.reshape(-1, 128), ref.reshape(-1, 128), "bf16")
    # rows that see no token are exact zeros
    for r, L in enumerate(lens):
        blind = max(0, q_len - L)
        if blind:
            assert not got[r, :blind].float().abs().sum()


def sample_rows(w, batch, n, seed):
    """Flat rows (r * q_len + i) * Hq + hq: random ones plus every head of the
    first and last query tokens and of the tokens at 128-block edges."""
    B, q, Hq = int(batch.seqlens.numel()), w.q_len, w.num_q_heads
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(B * q * Hq, n, replace=False).tolist())
    for r in range(B):
        for i in {0, 1, 127, 128, q // 2, q - 129, q - 128, q - 1}:
            if 0 <= i < q:
                rows.update(((r * q + i) * Hq + h) for h in range(0, Hq, 7))
    return sorted(rows)


@pytest.mark.parametrize("name", ["t4_q512", "t4_q1ks2k", "t4_q2k", "t4_2q1ks4k", "t4_q8k"])
def test_table4_shapes(name):
    w = WORKLOADS[name]
    batch = make_batch(w, device="cuda", poison_tail=True)
    got = run_prefill(batch)
    rows = sample_rows(w, batch, 160, 11)
    assert_close(got, oracle_rows(batch, rows=rows), "bf16", rows=rows)
    assert torch.isfinite(got.float()).all()


def test_repeated_launches_are_bitwise_identical():
    batch = make_batch(WORKLOADS["t4_q1ks2k"], device="cuda")
    a = run_prefill(batch)
    b = run_prefill(batch)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_page_permutation_invariance():
    """The same tokens on other physical pages give bit-identical output."""
    lens = [700, 1500]
    batch = small("perm", lens, 8, 2, 300, 77)
    a = run_prefill(batch)
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(batch.num_pages, generator=g).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel(), device="cuda")
    batch.k_cache = batch.k_cache[inv]
    batch.v_cache = batch.v_cache[inv]
    bt = batch.block_table.clone()
    live = bt >= 0
    bt[live] = perm[bt[live].long()].to(torch.int32)
    batch.block_table = bt
    b = run_prefill(batch)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bad_length_and_page_are_flagged():
    batch = small("flags", [200, 300], 4, 1, 100, 91)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    batch.seqlens[0] = 10 ** 6  # beyond the block table: clamped to its 4 pages
    run_prefill(batch, flags=flags)
    assert int(flags.item()) & hd.binding.HPC_FLAG_BAD_SEQLEN
    batch = small("flags2", [200, 300], 4, 1, 100, 92)
    batch.block_table[1, 2] = batch.num_pages + 5  # not read; flagged
    flags.zero_()
    got = run_prefill(batch, flags=flags)
    assert int(flags.item()) & hd.binding.HPC_FLAG_BAD_PAGE
    # the other request is unaffected
    ref = oracle_rows(batch, rows=list(range(0, 100 * 4)))
    assert_close(got[0].reshape(-1, 128), ref, "bf16")


def test_unsupported_shapes_are_refused():
    batch = small("bad", [100], 6, 4, 100, 93)  # Hq % Hkv != 0
    out = torch.empty((1, 100, 6, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(hd.HpcError):
        hd.hpc_prefill_attn(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                            batch.seqlens, 6, 4, 100, 0.088, out)


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes(seed):
    """Seeded random batches: 1-4 requests, q_len 1..300, lengths below and
    above q_len (up to 3000 tokens of prefix), G in {1, 2, 4, 8}."""
    rng = np.random.default_rng(900 + seed)
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8]))
    q_len = int(rng.integers(1, 301))
    B = int(rng.integers(1, 5))
    lens = [int(q_len + rng.integers(-min(q_len, 40), 3000)) for _ in range(B)]
    lens = [max(L, 0) for L in lens]
    batch = small(f"rand{seed}", lens, g * hkv, hkv, q_len, 950 + seed)
    got = run_prefill(batch)
    assert_close(got.reshape(-1, 128), oracle_rows(batch).reshape(-1, 128), "bf16")
