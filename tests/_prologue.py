"""Helpers of the prologue parity tests: run hpc_rope_norm through the C ABI
and check its outputs against the fp64 prologue oracle.

What "matches" means: the kernel computes in fp32 and rounds once to BF16 or
E4M3; the oracle gives the exact (fp64) value r.  A GPU output is valid when
it is a rounding of some value within eps of r, i.e. it lies between the
oracle's own roundings of r - eps and r + eps, where eps bounds the fp32
error of the norm and the rotation (a few ulps of the row's largest value).
On top of that, outputs that differ from the rounding of r itself must be
rare (they can only sit next to a rounding midpoint)."""

from __future__ import annotations

import numpy as np
import torch

import load_balanced_paged_assign_gb300 as hd
from oracle import rope_norm as rn

REL_EPS = 4e-6  # fp32 error bound, relative to the row's largest |value|


def words(t: torch.Tensor) -> np.ndarray:
    """Storage words of a BF16 (uint16) or E4M3 (uint8) tensor, on the CPU."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)


def run_gpu(inp, **overrides):
    """One hpc_rope_norm call on inp (its caches are written in place)."""
    w = inp.workload
    N, Hq = inp.num_tokens, w.num_q_heads
    fp8 = w.kv_dtype == "e4m3"
    dev = inp.qkv.device
    q_out = torch.full((max(N, 1), Hq, 128), float("nan"), dtype=torch.float32, device=dev)
    q_out = q_out.to(torch.float8_e4m3fn if fp8 else torch.bfloat16)
    q_scale = torch.full((max(N, 1), Hq), float("nan"), device=dev) if fp8 else None
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    kw = dict(eps=w.eps, rope_base=w.rope_base, rope_layout=w.rope_layout,
              norm_first=w.norm_first)
    kw.update(overrides)
    hd.hpc_rope_norm(inp.qkv, inp.q_norm_w, inp.k_norm_w, inp.positions, inp.token_req, Hq,
                     w.num_kv_heads, inp.block_table, inp.k_cache, inp.v_cache, inp.k_scale,
                     inp.v_scale, q_out, q_scale, flags, **kw)
    torch.cuda.synchronize()
    return q_out[:N], (None if q_scale is None else q_scale[:N]), int(flags.item())


def run_oracle(inp, k_cache0, v_cache0, tokens=None, **overrides):
    """The oracle on the same inputs (optionally only the listed tokens)."""
    w = inp.workload
    qkv = words(inp.qkv)
    pos = inp.positions.cpu().numpy()
    req = None if inp.token_req is None else inp.token_req.cpu().numpy()
    if tokens is not None:
        qkv, pos = qkv[tokens], pos[tokens]
        req = np.asarray(tokens) if req is None else req[tokens]
    p = dict(eps=w.eps, base=w.rope_base, style=w.rope_layout, norm_first=w.norm_first)
    p.update(overrides)
    # the C ABI takes eps and the base as fp32: the oracle uses the same values
    p["eps"] = float(np.float32(p["eps"]))
    p["base"] = float(np.float32(p["base"]))
    return rn.rope_norm(qkv, words(inp.q_norm_w), words(inp.k_norm_w), pos, req, w.num_q_heads,
                        w.num_kv_heads, inp.block_table.cpu().numpy(), k_cache0, v_cache0,
                        w.kv_dtype, inp.k_scale, inp.v_scale, p["eps"], p["base"], p["style"],
                        p["norm_first"])


def bracketed(got, ref, eps, encode, decode):
    """got (decoded values) lies between the roundings of ref - eps and ref + eps."""
    lo = decode(encode(ref - eps))
    hi = decode(encode(ref + eps))
    return (got >= lo) & (got <= hi)


def row_eps(ref):
    return REL_EPS * np.max(np.abs(ref), axis=-1, keepdims=True) + 1e-30


def check_bf16(got_words, ref, what):
    g = rn.bf16_decode(got_words)
    ok = bracketed(g, ref, row_eps(ref), rn.bf16_encode, rn.bf16_decode)
    assert ok.all(), f"{what}: {np.count_nonzero(~ok)} values outside the rounding bracket"
    exact = rn.bf16_encode(ref)
    n_off = np.count_nonzero(got_words != exact)
    assert n_off <= max(4, 1e-3 * ref.size), f"{what}: {n_off} values off the exact rounding"


def check_e4m3(got_codes, ref_scaled, eps_scaled, what):
    g = rn.e4m3_decode(got_codes)
    ok = bracketed(g, ref_scaled, eps_scaled, rn.e4m3_encode, rn.e4m3_decode)
    assert ok.all(), f"{what}: {np.count_nonzero(~ok)} codes outside the rounding bracket"
    exact = rn.e4m3_encode(ref_scaled)
    off = (got_codes != exact) & ((got_codes | exact) & 0x7F != 0)  # +-0 are the same value
    n_off = np.count_nonzero(off)
    assert n_off <= max(4, 1e-3 * ref_scaled.size), f"{what}: {n_off} codes off the exact rounding"


def check_against_oracle(inp, k_cache0, v_cache0, q_out, q_scale, flags, tokens=None, **ov):
    """Every output of hpc_rope_norm against the oracle (all tokens, or `tokens`)."""
    w = inp.workload
    fp8 = w.kv_dtype == "e4m3"
    res = run_oracle(inp, k_cache0, v_cache0, tokens, **ov)
    sel = slice(None) if tokens is None else np.asarray(tokens)
    if tokens is None:
        assert flags == res.flags
    # query
    if fp8:
        s_gpu = q_scale.cpu().double().numpy()[sel]
        assert np.allclose(s_gpu, res.q_scale, rtol=REL_EPS, atol=0), "query scales"
        codes = words(q_out)[sel]
        check_e4m3(codes, res.q / s_gpu[..., None], row_eps(res.q) / s_gpu[..., None], "query")
    else:
        check_bf16(words(q_out)[sel], res.q, "query")
    # caches: written slots against the oracle, all others untouched
    kc, vc = words(inp.k_cache), words(inp.v_cache)
    written = np.zeros(kc.shape[:2], dtype=bool)
    V = res.v
    for i, slot in enumerate(res.slots):
        if slot is None:
            continue
        pg, off = slot
        written[pg, off] = True
        if fp8:
            check_e4m3(kc[pg, off], res.k[i] / inp.k_scale, row_eps(res.k[i]) / inp.k_scale,
                       f"K of token {i}")
            x = V[i] / inp.v_scale
            check_e4m3(vc[pg, off], x, np.abs(x) * 2.0 ** -22 + 1e-30, f"V of token {i}")
        else:
            check_bf16(kc[pg, off], res.k[i], f"K of token {i}")
            assert np.array_equal(vc[pg, off], res.v_cache[pg, off]), f"V of token {i}"
    if tokens is None:
        assert np.array_equal(kc[~written], k_cache0[~written]), "K cache slots not written"
        assert np.array_equal(vc[~written], v_cache0[~written]), "V cache slots not written"
    return res
