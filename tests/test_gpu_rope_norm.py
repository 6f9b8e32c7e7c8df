"""Parity of the fused attention prologue (hpc_rope_norm) with its fp64 oracle,
through the C ABI: query (BF16, or E4M3 codes with per-(token, head) scales),
the new K and V cache rows, every other cache slot untouched, error flags;
then the prologue feeding the decode step."""

import dataclasses

import numpy as np
import pytest
import torch

import load_balanced_paged_assign_gb300 as hd
import oracle
from oracle import rope_norm as rn
from _gpu import TOL, assert_close, run_step
from _prologue import check_against_oracle, run_gpu, words
from load_balanced_paged_assign_gb300.workloads import (PROLOGUES, PrologueInputs,
                                                        PrologueWorkload, Workload, draw_qkv,
                                                        make_batch, make_prologue_inputs)

pytestmark = pytest.mark.gpu


def snapshot(inp):
    return words(inp.k_cache).copy(), words(inp.v_cache).copy()


def freq_table(base):
    f = torch.empty(64, dtype=torch.float64, device="cuda")
    hd.hpc_rope_frequencies(base, f)
    return f


def run_and_check(inp, tokens=None, **overrides):
    k0, v0 = snapshot(inp)
    q, qs, flags = run_gpu(inp, **overrides)
    ov = {}
    if "rope_base" in overrides:
        ov["base"] = overrides["rope_base"]
    if "eps" in overrides:
        ov["eps"] = overrides["eps"]
    res = check_against_oracle(inp, k0, v0, q, qs, flags, tokens, **ov)
    return q, qs, flags, res


def test_frequency_table_matches_the_oracle():
    for base in (10000.0, 1e6, 500000.0, 2.5):
        got = freq_table(base).cpu().numpy()
        ref = rn.rope_frequencies(128, float(np.float32(base)))
        assert np.allclose(got, ref, rtol=1e-15, atol=0)


SHAPES = [(8, 1), (4, 2), (64, 8), (2, 2), (16, 16)]


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("layout", [hd.HPC_ROPE_HALVES, hd.HPC_ROPE_INTERLEAVED])
@pytest.mark.parametrize("norm_first", [True, False])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_prefill_shapes(kv_dtype, layout, norm_first, shape):
    Hq, Hkv = SHAPES[shape]
    pw = PrologueWorkload(f"p{shape}", Hq, Hkv, kv_dtype=kv_dtype, prefill_tokens=150 + shape,
                          rope_layout=layout, norm_first=norm_first, rope_base=10000.0,
                          seed=40 + shape)
    # every other case takes the caller's frequency table
    table = {"freq": freq_table(10000.0)} if (shape + layout) % 2 else {}
    run_and_check(make_prologue_inputs(pw, device="cuda"), **table)


@pytest.mark.parametrize("name", ["decode_hy3_tp8", "decode_fp8"])
@pytest.mark.parametrize("table", [False, True])
def test_decode_workloads(name, table):
    pw = PROLOGUES[name]
    inp = make_prologue_inputs(pw, device="cuda")
    _, _, flags, res = run_and_check(inp, **({"freq": freq_table(pw.rope_base)} if table else {}))
    assert flags == 0 and all(s is not None for s in res.slots)


def test_more_tokens_than_resident_ctas():
    """Many tokens per CTA: the staging ring wraps many times."""
    pw = PrologueWorkload("wrap", 8, 1, kv_dtype="e4m3", prefill_tokens=20000, seed=47)
    inp = make_prologue_inputs(pw, device="cuda")
    run_and_check(inp, tokens=list(range(0, 20000, 97)) + [19999], freq=freq_table(1e6))


@pytest.mark.parametrize("name", ["prefill_8k_fp8", "prefill_8k_bf16"])
def test_full_size_prefill_sampled(name):
    inp = make_prologue_inputs(PROLOGUES[name], device="cuda")
    q, qs, flags, _ = run_and_check(inp, tokens=sorted({0, 1, 63, 64, 4095, 8191} | set(
        np.random.default_rng(9).integers(0, 8192, 40).tolist())))
    assert flags == 0
    # every output, sampled or not: finite, and the caches fully written
    if qs is not None:
        assert torch.isfinite(qs).all() and (qs > 0).all()
        assert not ((q.view(torch.uint8) & 0x7F) == 0x7F).any()
        assert not ((inp.k_cache.view(torch.uint8) & 0x7F) == 0x7F).any()
    else:
        assert torch.isfinite(q.float()).all() and torch.isfinite(inp.k_cache.float()).all()


def test_long_positions_keep_their_angles():
    """Positions up to 2^20 with a small base: the extended-precision angle
    reduction must hold."""
    N, Hq, Hkv = 48, 4, 1
    rng = np.random.default_rng(11)
    pos = np.sort(rng.choice(1 << 20, N, replace=False)).astype(np.int32)
    pos[0], pos[-1] = 0, (1 << 20) - 1
    max_pages = (1 << 20) // 64
    bt = torch.full((N, max_pages), -1, dtype=torch.int32)
    for t in range(N):
        bt[t, pos[t] // 64] = t  # one page per token: every slot distinct
    qkv, wq, wk = draw_qkv(N, Hq, Hkv, 12, "cuda")
    kc = torch.zeros((N, 64, Hkv, 128), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pw = PrologueWorkload("long", Hq, Hkv, rope_base=10000.0)
    inp = PrologueInputs(pw, qkv, wq, wk, torch.from_numpy(pos).cuda(), None, bt.cuda(), kc, vc,
                         1.0, 1.0)
    run_and_check(inp)


def test_bad_positions_requests_and_pages_flag_and_skip():
    B, Hq, Hkv = 4, 8, 1
    w = Workload("bad", B, Hq, Hkv, seqlens=(100, 300, 64, 1000), seed=5)
    batch = make_batch(w, device="cuda")
    N = 8
    qkv, wq, wk = draw_qkv(N, Hq, Hkv, 13, "cuda")
    bt = batch.block_table.clone()
    bt[2, 0] = 10 ** 6  # page past the cache
    pos = torch.tensor([99, -1, 5, 64 * bt.shape[1], 299, 10, 999, 3], dtype=torch.int32)
    req = torch.tensor([0, 1, 2, 1, 1, 7, 3, -1], dtype=torch.int32)
    pw = PrologueWorkload("bad", Hq, Hkv)
    inp = PrologueInputs(pw, qkv, wq, wk, pos.cuda(), req.cuda(), bt, batch.k_cache,
                         batch.v_cache, 1.0, 1.0)
    _, _, flags, res = run_and_check(inp)
    assert flags == hd.binding.HPC_FLAG_BAD_SEQLEN | hd.binding.HPC_FLAG_BAD_PAGE
    assert [s is not None for s in res.slots] == [True, False, False, False, True, False, True,
                                                  False]


def test_zero_rows_eps_and_saturation():
    pw = PrologueWorkload("z", 8, 1, kv_dtype="e4m3", prefill_tokens=70, seed=14)
    inp = make_prologue_inputs(pw, device="cuda")
    R = 10
    rows = inp.qkv.view(70, R, 128)
    rows[3, 2] = 0  # a zero query head: scale 1, codes +-0
    rows[5, 8] = 0  # a zero key head
    rows[6, 9] = 1e4  # a value head far past the cache's scale: saturates at +-448
    q, qs, _, _ = run_and_check(inp, eps=0.5)
    assert qs[3, 2].item() == 1.0 and not (q[3, 2].view(torch.uint8) & 0x7F).any()
    v_row = inp.v_cache.view(torch.uint8)[inp.block_table[0, 0].item(), 6, 0]
    assert ((v_row & 0x7F) == 0x7E).all()


def test_empty_and_repeated_calls():
    pw = PROLOGUES["decode_fp8"]
    inp = make_prologue_inputs(pw, device="cuda")
    q1, s1, f1 = run_gpu(inp)
    q2, s2, f2 = run_gpu(inp)
    assert torch.equal(q1.view(torch.uint8), q2.view(torch.uint8)) and torch.equal(s1, s2)
    empty = dataclasses.replace(inp, positions=inp.positions[:0], qkv=inp.qkv[:0])
    k0 = inp.k_cache.clone()
    run_gpu(empty)
    assert torch.equal(k0.view(torch.uint8), inp.k_cache.view(torch.uint8))


@pytest.mark.parametrize("name", ["decode_hy3_tp8", "decode_fp8"])
def test_prologue_feeds_the_decode_step(name):
    """Prologue, then plan + attention + combine on its outputs, against the
    oracle attention over the oracle prologue's cache rows and query."""
    pw = PROLOGUES[name]
    inp = make_prologue_inputs(pw, device="cuda", seqlens=None)
    batch = inp.batch
    k0, v0 = snapshot(inp)
    q, qs, flags = run_gpu(inp)
    assert flags == 0
    res = check_against_oracle(inp, k0, v0, q, qs, flags)
    step_batch = dataclasses.replace(batch, q=q, q_scale=qs)
    out, ws = run_step(step_batch)
    assert ws.tmap.to_host()["flags"] == 0
    fp8 = pw.kv_dtype == "e4m3"
    if fp8:
        oq = torch.from_numpy(res.q_codes).view(torch.float8_e4m3fn)
        oqs = torch.from_numpy(res.q_scale).float()
        ok = torch.from_numpy(res.k_cache).view(torch.float8_e4m3fn)
        ov = torch.from_numpy(res.v_cache).view(torch.float8_e4m3fn)
    else:
        oq = torch.from_numpy(res.q_bits.view(np.int16)).view(torch.bfloat16)
        oqs = None
        ok = torch.from_numpy(res.k_cache.view(np.int16)).view(torch.bfloat16)
        ov = torch.from_numpy(res.v_cache.view(np.int16)).view(torch.bfloat16)
    ref_batch = dataclasses.replace(batch, q=oq, q_scale=oqs, k_cache=ok, v_cache=ov,
                                    seqlens=batch.seqlens.cpu(),
                                    block_table=batch.block_table.cpu())
    ref = oracle.attention(ref_batch.q, ref_batch.k_cache, ref_batch.v_cache,
                           ref_batch.block_table, ref_batch.seqlens, **ref_batch.oracle_kwargs())
    assert_close(out, ref, pw.kv_dtype)
