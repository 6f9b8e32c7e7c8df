"""Oracle for the router GEMM with a BF16 hi/lo split of FP32 weights.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may use this module; the product path never does.

What the method computes follows the SGLang post, section "Router GEMM：在路由
精度与吞吐量之间取得平衡" (and its summary bullet on the router GEMM's accuracy):
the router projects BF16 hidden states onto expert scores with FP32 weights;
to run on BF16 tensor cores without dropping the weights' low mantissa bits,
each FP32 weight W is split into
    W_high = the BF16 truncation of W,
    W_low  = a BF16 of the scaled residual (W - W_high) * 256,
so W ~ W_high + W_low / 256, and the scores are
    S = X W_high^T + (X W_low^T) / 256,
both products accumulated in FP32 and the 1/256 applied at the end (the page
writes the result type as "FP36", a garbled FP32).

Readings where the page is silent (stated, not printed there):
  * truncation drops the low 16 bits of the FP32 word (rounds toward zero);
  * W_low is the round-to-nearest-even BF16 of the residual times 256 (the
    residual and its scaling are exact in FP32);
  * layouts follow a Linear layer: X [M, K] BF16 tokens x hidden, W [N, K]
    FP32 experts x hidden, S [M, N] FP32;
  * the page's shapes: K = 4096 hidden, N = 192 experts (its sweep), M tokens.

`router_scores` is the method's arithmetic taken step by step in fp64 (no
rounding beyond the split itself); `exact_scores` is the plain FP32-weight
product X W^T in fp64, against which the split's error is pinned.
"""

from __future__ import annotations

import numpy as np

from .rope_norm import bf16_decode, bf16_encode


def split_weights(w32):
    """(W_high, W_low) BF16 bit patterns (uint16) of FP32 weights."""
    w32 = np.ascontiguousarray(w32, dtype=np.float32)
    bits = w32.view(np.uint32)
    hi_bits = (bits >> 16).astype(np.uint16)  # truncation: drop the low 16 bits
    hi = (bits & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    resid = (w32.astype(np.float64) - hi) * 256.0  # exact
    return hi_bits, bf16_encode(resid)


def reconstruct(hi_bits, lo_bits):
    """W_high + W_low / 256 in fp64."""
    return bf16_decode(hi_bits) + bf16_decode(lo_bits) / 256.0


def router_scores(x_bits, hi_bits, lo_bits):
    """S = X W_high^T + (X W_low^T) / 256 in fp64; x_bits [M, K], hi/lo [N, K]."""
    x = bf16_decode(x_bits)
    return x @ bf16_decode(hi_bits).T + (x @ bf16_decode(lo_bits).T) / 256.0


def exact_scores(x_bits, w32):
    """The FP32-weight product X W^T in fp64."""
    return bf16_decode(x_bits) @ np.asarray(w32, dtype=np.float64).T


def split_error_bound(x_bits, w32):
    """Per-score bound on |router_scores - exact_scores| that the split
    guarantees: each weight is reconstructed within 2^-16 of its magnitude,
    so |S - XW^T| <= 2^-16 sum_k |x_k| |w_k|."""
    return 2.0 ** -16 * (np.abs(bf16_decode(x_bits)) @ np.abs(np.asarray(w32, dtype=np.float64)).T)
