"""Pins of the router-GEMM oracle (BF16 hi/lo split of FP32 weights).

The split is checked against torch's own bit operations and bf16 cast, its
reconstruction against the bound the formats give, and the scores against
the exact FP32-weight product: within the split's derived bound everywhere,
and within the page's stated error anchor (max-abs 0.00177 against FP32, at
K = 4096, N = 192) on data of that shape."""

import numpy as np
import pytest
import torch

from load_balanced_paged_assign_gb300.workloads import make_router_inputs
from oracle import router as ro
from oracle.rope_norm import bf16_decode


def bits16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_split_matches_torch_bit_operations_and_cast():
    w = torch.randn(64, 300, generator=torch.Generator().manual_seed(1)) * 3.0
    w[0, :5] = torch.tensor([0.0, -0.0, 1e-30, -65504.0, 3.0e38])
    hi_bits, lo_bits = ro.split_weights(w.numpy())
    hi_t = (w.view(torch.int32) & -65536).view(torch.float32)  # low 16 bits cleared
    assert np.array_equal(hi_bits, bits16(hi_t.to(torch.bfloat16)))  # exact: already bf16
    lo_t = ((w - hi_t) * 256.0).to(torch.bfloat16)  # residual and scaling exact in fp32
    assert np.array_equal(lo_bits, bits16(lo_t))


def test_truncation_rounds_toward_zero():
    w = np.array([1.0 + 2.0 ** -8 + 2.0 ** -20, -(1.0 + 2.0 ** -8 + 2.0 ** -20)], dtype=np.float32)
    hi_bits, lo_bits = ro.split_weights(w)
    assert np.array_equal(bf16_decode(hi_bits), [1.0, -1.0])  # a rounding split would give 1 + 2^-7
    assert np.all(bf16_decode(lo_bits) * np.sign(w) > 0)  # the residual keeps the weight's sign


def test_reconstruction_within_2_to_minus_16():
    w = (torch.randn(192, 4096, generator=torch.Generator().manual_seed(2)) / 64.0).numpy()
    hi, lo = ro.split_weights(w)
    rel = np.abs(ro.reconstruct(hi, lo) - w.astype(np.float64)) / np.abs(w.astype(np.float64))
    assert rel.max() <= 2.0 ** -16
    # and the low part carries real information: dropping it is ~2^-8 worse
    rel_hi = np.abs(bf16_decode(hi) - w.astype(np.float64)) / np.abs(w.astype(np.float64))
    assert rel_hi.mean() > 100 * rel.mean()


@pytest.mark.parametrize("M", [1, 7, 64])
def test_scores_within_the_split_bound_and_the_page_anchor(M):
    x, w = make_router_inputs(M, seed=1300 + M)
    xb = bits16(x)
    hi, lo = ro.split_weights(w.numpy())
    got = ro.router_scores(xb, hi, lo)
    exact = ro.exact_scores(xb, w.numpy())
    err = np.abs(got - exact)
    assert np.all(err <= ro.split_error_bound(xb, w.numpy()) + 1e-12)
    assert err.max() <= 0.00177  # the page's max-abs error against FP32 at K=4096, N=192
    # a plain BF16 cast of the weights misses that anchor by a wide margin
    plain = bf16_decode(xb) @ bf16_decode(bits16(w.to(torch.bfloat16))).T
    assert np.abs(plain - exact).max() > 10 * err.max()


def test_scores_are_the_two_products_in_order():
    x, w = make_router_inputs(5, K=256, N=24, seed=9)
    xb = bits16(x)
    hi, lo = ro.split_weights(w.numpy())
    # brute force over k on a few scores
    xv, hv, lv = bf16_decode(xb), bf16_decode(hi), bf16_decode(lo)
    got = ro.router_scores(xb, hi, lo)
    for m, n in [(0, 0), (3, 17), (4, 23)]:
        ref = sum(xv[m, k] * hv[n, k] for k in range(256)) + \
            sum(xv[m, k] * lv[n, k] for k in range(256)) / 256.0
        assert abs(got[m, n] - ref) <= 1e-12 * (1 + abs(ref))


def test_planted_mistakes_fail(monkeypatch):
    x, w = make_router_inputs(8, seed=11)
    xb = bits16(x)
    exact = ro.exact_scores(xb, w.numpy())
    hi, lo = ro.split_weights(w.numpy())
    # forgetting the 1/256 in the combine
    wrong = bf16_decode(xb) @ (bf16_decode(hi) + bf16_decode(lo)).T
    assert np.abs(wrong - exact).max() > 0.00177
    # the transposed weight layout cannot even be multiplied at this shape
    with pytest.raises(ValueError):
        ro.router_scores(xb, hi.T.copy(), lo.T.copy())
