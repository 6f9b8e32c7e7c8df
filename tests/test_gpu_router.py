"""Router GEMM (BF16 hi/lo split of FP32 weights, tcgen05 tensor cores)
through the C ABI against its oracle: the split bit for bit, the scores
within FP32 accumulation error of the oracle's arithmetic and within the
page's 0.00177 max-abs anchor of the exact FP32-weight product."""

import numpy as np
import pytest
import torch

import load_balanced_paged_assign_gb300 as hd
from load_balanced_paged_assign_gb300.workloads import make_router_inputs
from oracle import router as ro

pytestmark = pytest.mark.gpu

ACC_TOL = 5e-5  # |gpu - oracle arithmetic|: fp32 accumulation of K products, scores ~N(0, 1)


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def split_gpu(w):
    hi = torch.empty(w.shape, dtype=torch.bfloat16, device="cuda")
    lo = torch.empty_like(hi)
    hd.hpc_router_split(w, hi, lo)
    return hi, lo


def gemm_gpu(x, hi, lo, use_workspace=True):
    M, K = x.shape
    N = hi.shape[0]
    out = torch.full((M, N), float("nan"), device="cuda")
    ws = None
    nbytes = hd.hpc_router_workspace_bytes(M, N, K)
    if use_workspace and nbytes > 0:
        ws = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    hd.hpc_router_gemm(x, hi, lo, out, workspace=ws, flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    return out


def test_split_matches_the_oracle_bit_for_bit():
    w = torch.randn(192, 4096, generator=torch.Generator().manual_seed(3)) / 64.0
    w[0, :4] = torch.tensor([0.0, -0.0, 1e-30, -3.0e38])
    hi, lo = split_gpu(w.cuda())
    ref_hi, ref_lo = ro.split_weights(w.numpy())
    assert np.array_equal(bits16(hi), ref_hi) and np.array_equal(bits16(lo), ref_lo)


@pytest.mark.parametrize("M", [1, 5, 17, 64, 127, 128, 129, 300, 1024, 4096, 16384])
def test_scores_against_the_oracle(M):
    x, w = make_router_inputs(M, seed=1400 + M, device="cuda")
    hi, lo = split_gpu(w)
    got = gemm_gpu(x, hi, lo).cpu().double().numpy()
    xb = bits16(x)
    ref = ro.router_scores(xb, bits16(hi), bits16(lo))
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert err.max() <= ACC_TOL, f"max |gpu - oracle| {err.max():.3e}"
    exact = ro.exact_scores(xb, w.cpu().numpy())
    assert np.abs(got - exact).max() <= 0.00177  # the page's anchor against FP32


@pytest.mark.parametrize("M,N,K", [(1, 16, 64), (200, 272, 128), (129, 256, 4096),
                                   (3, 192, 4096), (700, 64, 1024), (77, 176, 512),
                                   (1000, 48, 256), (4100, 192, 4096), (40, 16, 128),
                                   (5000, 48, 1024), (2000, 512, 512), (8, 192, 4096),
                                   (12, 64, 1024), (9, 16, 128), (16, 192, 8192)])
def test_other_shapes(M, N, K):
    x, w = make_router_inputs(M, K=K, N=N, seed=1500 + M + N, device="cuda")
    hi, lo = split_gpu(w)
    got = gemm_gpu(x, hi, lo).cpu().double().numpy()
    ref = ro.router_scores(bits16(x), bits16(hi), bits16(lo))
    assert np.abs(got - ref).max() <= ACC_TOL * max(1.0, (K / 4096) ** 0.5)


@pytest.mark.parametrize("M", [16, 64, 300, 4096])
def test_split_k_matches_a_single_pass_and_is_deterministic(M):
    x, w = make_router_inputs(M, seed=1601 + M, device="cuda")
    hi, lo = split_gpu(w)
    a = gemm_gpu(x, hi, lo, use_workspace=True)
    b = gemm_gpu(x, hi, lo, use_workspace=True)
    c = gemm_gpu(x, hi, lo, use_workspace=False)  # no room for partials: one pass
    assert torch.equal(a, b)
    assert (a - c).abs().max().item() <= ACC_TOL


def test_plans_reported_for_the_sweep():
    """The plan query reports the launch: the CUDA-core kernel up to 16
    tokens, K split over more CTAs the fewer the tokens, no split once the
    token tiles alone fill the GPU."""
    few = hd.hpc_router_plan(16, 192, 4096)
    assert not few["tensor_cores"] and few["ctas"] == 96
    plans = [hd.hpc_router_plan(M, 192, 4096) for M in (64, 1024, 4096, 16384)]
    assert all(p["tensor_cores"] and p["bn"] == 192 for p in plans)
    splits = [p["splits"] for p in plans]
    assert splits == sorted(splits, reverse=True) and splits[0] > 1 and splits[-1] == 1
    assert all(p["ctas"] <= torch.cuda.get_device_properties(0).multi_processor_count
               for p in plans)


@pytest.mark.parametrize("M,N", [(300, 192), (129, 176), (5000, 48)])
def test_nothing_is_written_past_the_scores(M, N):
    """The scores are a view into a larger buffer: the rows after them keep
    their sentinel (the tail tile's rows past M are clipped by the store)."""
    x, w = make_router_inputs(M, K=1024, N=N, seed=1700 + M, device="cuda")
    hi, lo = split_gpu(w)
    buf = torch.full((M + 130, N), 7.0, device="cuda")
    out = buf[:M]
    nbytes = hd.hpc_router_workspace_bytes(M, N, 1024)
    ws = torch.empty(max(nbytes // 4, 1), device="cuda") if nbytes > 0 else None
    hd.hpc_router_gemm(x, hi, lo, out, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(buf[M:], torch.full_like(buf[M:], 7.0))
    ref = ro.router_scores(bits16(x), bits16(hi), bits16(lo))
    assert np.abs(out.cpu().double().numpy() - ref).max() <= ACC_TOL
