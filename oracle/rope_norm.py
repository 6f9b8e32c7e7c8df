"""Oracle for the fused attention prologue (QK-Norm, RoPE, paged KV write,
FP8 query quantisation).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may use this module; the product path never does.

What the prologue computes follows the vLLM integration post ("A fused
attention prologue") and the SGLang post's description of the same op: from
the fused QKV projection of each new token it
  * applies QK-Norm (an RMS norm over each query and key head) and RoPE, in
    the model's order (Hy3: the norm first, then RoPE),
  * writes the token's K and V straight into the paged KV cache,
  * and, with FP8 KV, emits the query as FP8-E4M3 with one scale per
    (token, head), which the attention step consumes as it is.

The pages give none of the constants, so the readings below are stated, not
printed on the pages (they are the standard definitions of the pieces):
  * RMS norm of a head row x (D = 128): y = x / sqrt(mean(x^2) + eps) * w,
    one weight vector w [D] for all query heads and one for all key heads;
  * RoPE over the whole head: frequency i in [0, D/2) is
    theta_i = base^(-2i/D); the pair (a, b) of dims rotates by the angle
    pos * theta_i, (a, b) -> (a cos - b sin, b cos + a sin); the pair is
    (i, i + D/2) in the "halves" layout and (2i, 2i + 1) in the
    "interleaved" one;
  * V passes through untouched;
  * the new token of request r at position p lands in page
    block_table[r, p // 64], slot p % 64;
  * FP8 query: scale = amax / 448 over the head row (1 when the row is all
    zero), code = E4M3 round-to-nearest-even of y / scale, saturating at
    +-448; FP8 K and V use the cache's per-tensor scales the same way;
  * BF16 outputs are the round-to-nearest-even BF16 of the exact result.

Everything is computed in fp64 with numpy, one token and head at a time.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

HALVES = 0
INTERLEAVED = 1

E4M3_MAX = 448.0


# --------------------------------------------------------------- encoders

def _e4m3_positive_values() -> np.ndarray:
    """Values of the finite non-negative E4M3 codes 0x00..0x7E, in code order.

    The format: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent
    field 0 is subnormal (2^-6 * m/8); code 0x7F (all ones) is NaN; there
    are no infinities, so 0x7E = 1.75 * 2^8 = 448 is the largest value."""
    vals = np.empty(127, dtype=np.float64)
    for code in range(127):
        e, m = code >> 3, code & 7
        vals[code] = math.ldexp(m / 8.0, -6) if e == 0 else math.ldexp(1.0 + m / 8.0, e - 7)
    return vals


_E4M3_VALUES = _e4m3_positive_values()


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of fp64 values: round to nearest, ties to the even
    code, magnitudes past 448 saturate to 448, NaN becomes the NaN code."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_E4M3_VALUES, mag, side="left")  # first value >= mag
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _E4M3_VALUES[lo]
    d_hi = _E4M3_VALUES[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    code = np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)
    return code


def e4m3_decode(codes) -> np.ndarray:
    """fp64 values of E4M3 codes (NaN for 0x7F / 0xFF)."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag = codes & 0x7F
    out = np.where(mag == 0x7F, np.nan, _E4M3_VALUES[np.minimum(mag, 126)])
    return np.where(codes & 0x80, -out, out)


def bf16_encode(x) -> np.ndarray:
    """BF16 bit patterns (uint16) of fp64 values, rounded to nearest even
    directly from fp64 (8 significant bits, exponent range of fp32)."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    finite = np.isfinite(mag) & (mag > 0.0)
    safe = np.where(finite, mag, 1.0)
    _, e = np.frexp(safe)  # |x| = m * 2^e, m in [0.5, 1)
    e_eff = np.maximum(e, -125)  # below 2^-126 the spacing stops shrinking
    r = np.ldexp(np.rint(np.ldexp(safe, 8 - e_eff)), e_eff - 8)  # rint: ties to even
    r = np.where(r < 2.0 ** 128, r, np.inf)
    out = np.where(finite, np.copysign(r, x), x)
    bits = out.astype(np.float32).view(np.uint32)  # exact: r has 8 significant bits
    return (bits >> 16).astype(np.uint16)


def bf16_decode(bits) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- pieces

def rope_frequencies(head_dim: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/D) for i in [0, D/2)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / head_dim)


def rope_pairs(head_dim: int, style: int):
    """Index arrays (first, second) of the rotated pairs, frequency i at i."""
    half = head_dim // 2
    i = np.arange(half)
    if style == HALVES:
        return i, i + half
    if style == INTERLEAVED:
        return 2 * i, 2 * i + 1
    raise ValueError(f"unknown RoPE layout {style}")


def rope(x, pos: int, base: float, style: int) -> np.ndarray:
    """Rotate each pair of x [..., D] by pos * theta_i."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    a_idx, b_idx = rope_pairs(D, style)
    phi = float(pos) * rope_frequencies(D, base)
    c, s = np.cos(phi), np.sin(phi)
    a, b = x[..., a_idx], x[..., b_idx]
    out = np.empty_like(x)
    out[..., a_idx] = a * c - b * s
    out[..., b_idx] = b * c + a * s
    return out


def rms_norm(x, w, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * np.asarray(w, dtype=np.float64)


def norm_and_rope(x, w, pos: int, eps: float, base: float, style: int,
                  norm_first: bool) -> np.ndarray:
    """QK-Norm and RoPE of one head row, in the order the model asks for."""
    if norm_first:
        return rope(rms_norm(x, w, eps), pos, base, style)
    return rms_norm(rope(x, pos, base, style), w, eps)


def quantize_row_e4m3(y):
    """Per-row FP8 query: (codes, scale) with scale = amax / 448 (1 for a zero row)."""
    y = np.asarray(y, dtype=np.float64)
    amax = float(np.max(np.abs(y))) if y.size else 0.0
    scale = amax / E4M3_MAX if amax > 0.0 else 1.0
    return e4m3_encode(y / scale), scale


# ------------------------------------------------------------ whole op

@dataclass
class PrologueResult:
    q: np.ndarray  # fp64 [N, Hq, D]: the exact normalised, rotated query
    k: np.ndarray  # fp64 [N, Hkv, D]: the exact normalised, rotated key
    v: np.ndarray  # fp64 [N, Hkv, D]: the value rows as given
    q_codes: np.ndarray | None  # uint8 [N, Hq, D] (FP8) or None
    q_scale: np.ndarray | None  # fp64 [N, Hq] (FP8) or None
    q_bits: np.ndarray | None  # uint16 [N, Hq, D] (BF16) or None
    k_cache: np.ndarray  # storage words after the write (uint16 BF16 / uint8 E4M3)
    v_cache: np.ndarray
    slots: list  # per token: (page, offset) written, or None when skipped
    flags: int  # 1: a bad position or request index; 4: a bad page


def rope_norm(qkv_bits, q_norm_w_bits, k_norm_w_bits, positions, token_req, num_q_heads: int,
              num_kv_heads: int, block_table, k_cache, v_cache, kv_dtype: str, k_scale: float,
              v_scale: float, eps: float, base: float, style: int, norm_first: bool,
              head_dim: int = 128, page: int = 64) -> PrologueResult:
    """The whole prologue for N tokens.

    qkv_bits: uint16 BF16 words [N, (Hq + 2 Hkv) * D], head rows in the order
      Q heads, K heads, V heads; norm weights: uint16 BF16 words [D];
    positions [N]; token_req [N] or None (token t belongs to request t);
    block_table [B, max_pages]; k_cache, v_cache: storage words
    [num_pages, page, Hkv, D] (uint16 for "bf16", uint8 for "e4m3"),
    copied, not modified.  A token whose position or request is out of
    range, or whose page is outside the cache, gets its query but writes no
    cache slot, and raises the matching flag."""
    Hq, Hkv, D = num_q_heads, num_kv_heads, head_dim
    qkv = bf16_decode(qkv_bits).reshape(len(positions), Hq + 2 * Hkv, D)
    wq = bf16_decode(q_norm_w_bits)
    wk = bf16_decode(k_norm_w_bits)
    bt = np.asarray(block_table)
    B, max_pages = bt.shape
    num_pages = k_cache.shape[0]
    fp8 = kv_dtype == "e4m3"
    kc, vc = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    N = len(positions)
    q = np.zeros((N, Hq, D))
    k = np.zeros((N, Hkv, D))
    v = qkv[:, Hq + Hkv:, :].copy()
    q_codes = np.zeros((N, Hq, D), dtype=np.uint8) if fp8 else None
    q_scale = np.zeros((N, Hq)) if fp8 else None
    flags = 0
    slots = []
    for t in range(N):
        pos = int(positions[t])
        r = t if token_req is None else int(token_req[t])
        for h in range(Hq):
            q[t, h] = norm_and_rope(qkv[t, h], wq, pos, eps, base, style, norm_first)
            if fp8:
                q_codes[t, h], q_scale[t, h] = quantize_row_e4m3(q[t, h])
        for h in range(Hkv):
            k[t, h] = norm_and_rope(qkv[t, Hq + h], wk, pos, eps, base, style, norm_first)
        if not (0 <= r < B and 0 <= pos < max_pages * page):
            flags |= 1
            slots.append(None)
            continue
        pg = int(bt[r, pos // page])
        if not 0 <= pg < num_pages:
            flags |= 4
            slots.append(None)
            continue
        off = pos % page
        slots.append((pg, off))
        if fp8:
            kc[pg, off] = e4m3_encode(k[t] / k_scale)
            vc[pg, off] = e4m3_encode(v[t] / v_scale)
        else:
            kc[pg, off] = bf16_encode(k[t])
            vc[pg, off] = qkv_bits.reshape(N, Hq + 2 * Hkv, D)[t, Hq + Hkv:]
    q_bits = None if fp8 else bf16_encode(q)
    return PrologueResult(q, k, v, q_codes, q_scale, q_bits, kc, vc, slots, flags)
