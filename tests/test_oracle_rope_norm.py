"""Pins of the prologue oracle (QK-Norm, RoPE, paged KV write, FP8 query).

Each check ties the oracle to something other than itself: torch's own
float8 / bfloat16 casts, numpy's complex exponential, closed forms of the
norm and the rotation, and invariants chosen so that a plausible slip (a
sign, a frequency exponent, the pairing of dims, the order of norm and
rotation, a page lookup) fails one of them."""

import math

import numpy as np
import pytest
import torch

from oracle import rope_norm as rn

D = 128


# ----------------------------------------------------------- encoders

def test_e4m3_encoder_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = rn.e4m3_decode(codes)
    back = rn.e4m3_encode(vals)
    # +0 and -0 both decode to zero; the sign survives through signbit
    assert np.array_equal(back, codes)


def test_e4m3_decoder_matches_torch_on_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = rn.e4m3_decode(codes.numpy())
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(np.where(both_nan, 0, ref), np.where(both_nan, 0, got))


def test_e4m3_encoder_matches_torch_cast_in_range():
    gen = torch.Generator().manual_seed(7)
    x = torch.randn(200_000, generator=gen) * torch.exp2(torch.randint(-9, 8, (200_000,),
                                                                        generator=gen).float())
    x = x.clamp(-448.0, 448.0)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = rn.e4m3_encode(x.double().numpy())
    assert np.array_equal(got, ref)


def test_e4m3_ties_go_to_the_even_code_and_large_values_saturate():
    assert rn.e4m3_encode(1.0625) == 0x38  # between 1.0 (0x38) and 1.125 (0x39)
    assert rn.e4m3_encode(1.1875) == 0x3A  # between 1.125 (0x39) and 1.25 (0x3A)
    assert rn.e4m3_encode(-1.0625) == 0xB8
    assert rn.e4m3_encode(1000.0) == 0x7E and rn.e4m3_encode(-1e9) == 0xFE
    assert rn.e4m3_encode(464.0) == 0x7E  # past 448 saturates rather than rounding up
    assert rn.e4m3_encode(2.0 ** -10) == 0x00  # half the smallest subnormal: tie to 0
    assert rn.e4m3_encode(3 * 2.0 ** -10) == 0x02  # 1.5 subnormal steps: tie to even 2
    assert rn.e4m3_encode(float("nan")) == 0x7F


def test_bf16_encoder_matches_torch_on_fp32_values():
    gen = torch.Generator().manual_seed(8)
    x = torch.randn(100_000, generator=gen) * 37.0
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = rn.bf16_encode(x.double().numpy())
    assert np.array_equal(got, ref)


def test_bf16_encoder_rounds_once_from_fp64():
    # 1 + 2^-8 + 2^-30 lies just above the midpoint between 1 and 1 + 2^-7:
    # rounding it to fp32 first would land on the midpoint and tie down to 1.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert rn.bf16_decode(rn.bf16_encode(x)) == 1.0 + 2.0 ** -7
    assert rn.bf16_decode(rn.bf16_encode(1.0 + 2.0 ** -8)) == 1.0  # exact tie: even
    assert rn.bf16_decode(rn.bf16_encode(1.0 + 3 * 2.0 ** -8)) == 1.0 + 2.0 ** -6


# ----------------------------------------------------------- RMS norm

def test_rms_norm_closed_forms():
    w = np.linspace(0.5, 1.5, D)
    c = 3.0
    eps = 1e-6
    y = rn.rms_norm(np.full(D, c), w, eps)
    assert np.allclose(y, w * c / math.sqrt(c * c + eps), rtol=1e-15)
    x = np.random.default_rng(1).normal(size=D)
    y0 = rn.rms_norm(x, np.ones(D), 0.0)
    assert math.isclose(np.mean(y0 * y0), 1.0, rel_tol=1e-14)  # unit mean square
    assert np.allclose(rn.rms_norm(7.5 * x, w, 0.0), rn.rms_norm(x, w, 0.0), rtol=1e-14)
    # eps acts inside the root: a tiny row is not blown up to unit scale
    small = rn.rms_norm(np.full(D, 1e-4), np.ones(D), 1e-6)
    assert np.allclose(small, 1e-4 / math.sqrt(1e-8 + 1e-6), rtol=1e-14)


# --------------------------------------------------------------- RoPE

@pytest.mark.parametrize("style", [rn.HALVES, rn.INTERLEAVED])
def test_rope_is_the_complex_rotation(style):
    rng = np.random.default_rng(2)
    x = rng.normal(size=D)
    base, pos = 10000.0, 12345
    a_idx, b_idx = rn.rope_pairs(D, style)
    z = (x[a_idx] + 1j * x[b_idx]) * np.exp(1j * pos * base ** (-np.arange(D // 2) / (D // 2)))
    y = rn.rope(x, pos, base, style)
    assert np.allclose(y[a_idx], z.real, atol=1e-12)
    assert np.allclose(y[b_idx], z.imag, atol=1e-12)


def test_rope_one_hot_closed_form():
    # frequency 32 of 64 with base 10^4 is 10^4^(-1/2) = 0.01: position 100 turns it by 1 rad
    y = rn.rope(np.eye(D)[32], 100, 10000.0, rn.HALVES)
    assert math.isclose(y[32], math.cos(1.0), rel_tol=1e-13)
    assert math.isclose(y[96], math.sin(1.0), rel_tol=1e-13)
    assert np.count_nonzero(np.abs(y) > 1e-15) == 2
    # the same frequency in the interleaved layout pairs dims 64 and 65
    y = rn.rope(np.eye(D)[65], 100, 10000.0, rn.INTERLEAVED)
    assert math.isclose(y[64], -math.sin(1.0), rel_tol=1e-13)
    assert math.isclose(y[65], math.cos(1.0), rel_tol=1e-13)
    # frequency 0 turns by the position itself
    y = rn.rope(np.eye(D)[0], 3, 500000.0, rn.HALVES)
    assert math.isclose(y[0], math.cos(3.0), rel_tol=1e-13)
    assert math.isclose(y[64], math.sin(3.0), rel_tol=1e-13)


@pytest.mark.parametrize("style", [rn.HALVES, rn.INTERLEAVED])
def test_rope_invariants(style):
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=D), rng.normal(size=D)
    base = 1e6
    assert np.array_equal(rn.rope(q, 0, base, style), q)
    assert math.isclose(np.linalg.norm(rn.rope(q, 99_999, base, style)), np.linalg.norm(q),
                        rel_tol=1e-13)
    # attention scores depend on relative positions only
    s1 = rn.rope(q, 5000, base, style) @ rn.rope(k, 1200, base, style)
    s2 = rn.rope(q, 5000 + 777, base, style) @ rn.rope(k, 1200 + 777, base, style)
    assert math.isclose(s1, s2, rel_tol=1e-10, abs_tol=1e-10)
    # rotating by -p undoes rotating by p
    assert np.allclose(rn.rope(rn.rope(q, 4321, base, style), -4321, base, style), q,
                       atol=1e-12)


def test_norm_and_rope_order():
    rng = np.random.default_rng(4)
    x = rng.normal(size=D) * 3.0
    w = 1.0 + 0.3 * rng.normal(size=D)
    pos, base = 777, 10000.0
    first = rn.norm_and_rope(x, w, pos, 0.0, base, rn.HALVES, norm_first=True)
    after = rn.norm_and_rope(x, w, pos, 0.0, base, rn.HALVES, norm_first=False)
    # norm then rotate: undo the rotation and the weights to get a unit-RMS row
    un = rn.rope(first, -pos, base, rn.HALVES) / w
    assert math.isclose(np.mean(un * un), 1.0, rel_tol=1e-12)
    # rotate then norm: the weights sit outside the rotation
    assert math.isclose(np.mean((after / w) ** 2), 1.0, rel_tol=1e-12)
    assert not np.allclose(first, after, atol=1e-3)
    # with unit weights the two orders agree (the rotation keeps the RMS)
    one = np.ones(D)
    assert np.allclose(rn.norm_and_rope(x, one, pos, 0.0, base, rn.HALVES, True),
                       rn.norm_and_rope(x, one, pos, 0.0, base, rn.HALVES, False), atol=1e-13)


# ---------------------------------------------------------- whole op

def bf16_bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def small_case(kv_dtype, Hq=4, Hkv=2, seed=5):
    rng = np.random.default_rng(seed)
    N = 3
    qkv = bf16_bits(rng.normal(size=(N, (Hq + 2 * Hkv) * D)) * 2.0)
    wq = bf16_bits(1.0 + 0.2 * rng.normal(size=D))
    wk = bf16_bits(1.0 + 0.2 * rng.normal(size=D))
    bt = np.array([[5, 9, 2], [0, 7, -1], [3, 1, 4]], dtype=np.int32)
    num_pages = 10
    word = np.uint8 if kv_dtype == "e4m3" else np.uint16
    kc = rng.integers(0, 2 ** (8 * np.dtype(word).itemsize), size=(num_pages, 64, Hkv, D)) \
        .astype(word)
    vc = rng.integers(0, 2 ** (8 * np.dtype(word).itemsize), size=(num_pages, 64, Hkv, D)) \
        .astype(word)
    return qkv, wq, wk, bt, kc, vc


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_kv_write_lands_in_the_looked_up_slot_only(kv_dtype):
    Hq, Hkv = 4, 2
    qkv, wq, wk, bt, kc, vc = small_case(kv_dtype, Hq, Hkv)
    positions = [130, 64, 5]  # pages bt[0,2]=2 slot 2, bt[1,1]=7 slot 0, bt[2,0]=3 slot 5
    res = rn.rope_norm(qkv, wq, wk, positions, None, Hq, Hkv, bt, kc, vc, kv_dtype, 0.02, 0.03,
                       1e-6, 10000.0, rn.HALVES, True)
    assert res.slots == [(2, 2), (7, 0), (3, 5)]
    assert res.flags == 0
    changed = np.argwhere((res.k_cache != kc).any(axis=(2, 3)))
    assert {tuple(x) for x in changed} <= {(2, 2), (7, 0), (3, 5)}
    for (pg, off), t in zip(res.slots, range(3)):
        other = np.ones(kc.shape[:2], dtype=bool)
        other[pg, off] = False
        if kv_dtype == "bf16":
            # V is copied word for word; K is the BF16 of the exact rotated row
            assert np.array_equal(res.v_cache[pg, off],
                                  qkv.reshape(3, Hq + 2 * Hkv, D)[t, Hq + Hkv:])
            assert np.array_equal(rn.bf16_decode(res.k_cache[pg, off]),
                                  rn.bf16_decode(rn.bf16_encode(res.k[t])))
        else:
            assert np.array_equal(res.v_cache[pg, off], rn.e4m3_encode(res.v[t] / 0.03))
            assert np.array_equal(res.k_cache[pg, off], rn.e4m3_encode(res.k[t] / 0.02))
    untouched = np.ones(kc.shape[:2], dtype=bool)
    for pg, off in res.slots:
        untouched[pg, off] = False
    assert np.array_equal(res.k_cache[untouched], kc[untouched])
    assert np.array_equal(res.v_cache[untouched], vc[untouched])


def test_bad_positions_and_pages_skip_the_write_and_flag():
    Hq, Hkv = 4, 2
    qkv, wq, wk, bt, kc, vc = small_case("bf16", Hq, Hkv)
    # token 0: position past the table; token 1: page -1; token 2: fine
    res = rn.rope_norm(qkv, wq, wk, [192, 130, 0], None, Hq, Hkv, bt, kc, vc, "bf16", 1.0, 1.0,
                       1e-6, 10000.0, rn.HALVES, True)
    assert res.slots == [None, None, (3, 0)]
    assert res.flags == 1 | 4
    res = rn.rope_norm(qkv, wq, wk, [0, 0, 0], [0, 5, 2], Hq, Hkv, bt, kc, vc, "bf16", 1.0, 1.0,
                       1e-6, 10000.0, rn.HALVES, True)
    assert res.slots == [(5, 0), None, (3, 0)] and res.flags == 1


def test_fp8_query_scale_and_codes():
    Hq, Hkv = 4, 2
    qkv, wq, wk, bt, kc, vc = small_case("e4m3", Hq, Hkv)
    qkv = qkv.copy().reshape(3, Hq + 2 * Hkv, D)
    qkv[1, 2] = 0  # an all-zero query head
    res = rn.rope_norm(qkv.reshape(3, -1), wq, wk, [1, 2, 3], None, Hq, Hkv, bt, kc, vc, "e4m3",
                       1.0, 1.0, 1e-6, 10000.0, rn.INTERLEAVED, True)
    for t in range(3):
        for h in range(Hq):
            y = res.q[t, h]
            if t == 1 and h == 2:
                assert res.q_scale[t, h] == 1.0 and not (res.q_codes[t, h] & 0x7F).any()  # +-0
                continue
            amax = np.abs(y).max()
            assert res.q_scale[t, h] == amax / 448.0
            # the largest element maps to the largest code, every code is the
            # nearest E4M3 value of y / scale
            assert (res.q_codes[t, h][np.argmax(np.abs(y))] & 0x7F) == 0x7E
            deq = rn.e4m3_decode(res.q_codes[t, h]) * res.q_scale[t, h]
            assert np.all(np.abs(deq - y) <= amax / 448.0 * 16.0 + 1e-12)  # half the top gap of 32
            assert np.all(np.abs(deq - y) <= np.abs(y) / 16.0 + amax / 448.0 * 2.0 ** -9)


# ------------------------------------------------- planted mistakes
# Each slip below is planted in the oracle (on the CPU) and must fail a pin.

def one_hot_pin_holds():
    y = rn.rope(np.eye(D)[32], 100, 10000.0, rn.HALVES)
    return math.isclose(y[32], math.cos(1.0), rel_tol=1e-13) and \
        math.isclose(y[96], math.sin(1.0), rel_tol=1e-13)


def complex_pin_holds(style):
    x = np.random.default_rng(2).normal(size=D)
    a_idx, b_idx = np.arange(64), np.arange(64) + 64
    if style == rn.INTERLEAVED:
        a_idx, b_idx = 2 * np.arange(64), 2 * np.arange(64) + 1
    z = (x[a_idx] + 1j * x[b_idx]) * np.exp(1j * 321 * 10000.0 ** (-np.arange(64) / 64))
    y = rn.rope(x, 321, 10000.0, style)
    return np.allclose(y[a_idx], z.real, atol=1e-12) and np.allclose(y[b_idx], z.imag, atol=1e-12)


def test_planted_frequency_exponent_fails(monkeypatch):
    assert one_hot_pin_holds()
    monkeypatch.setattr(rn, "rope_frequencies",
                        lambda d, base: np.power(float(base), -np.arange(d // 2) / d))
    assert not one_hot_pin_holds()


def test_planted_rotation_direction_fails(monkeypatch):
    orig = rn.rope

    def clockwise(x, pos, base, style):
        return orig(x, -pos, base, style)

    monkeypatch.setattr(rn, "rope", clockwise)
    assert not complex_pin_holds(rn.HALVES)


def test_planted_pair_layout_fails(monkeypatch):
    orig = rn.rope_pairs
    monkeypatch.setattr(rn, "rope_pairs", lambda d, style: orig(d, 1 - style))
    assert not complex_pin_holds(rn.HALVES)
    assert not one_hot_pin_holds()


def test_planted_order_fails(monkeypatch):
    rng = np.random.default_rng(4)
    x, w = rng.normal(size=D), 1.0 + 0.3 * rng.normal(size=D)
    monkeypatch.setattr(rn, "norm_and_rope",
                        lambda x, w, pos, eps, base, style, norm_first:
                        rn.rms_norm(rn.rope(x, pos, base, style), w, eps))
    first = rn.norm_and_rope(x, w, 777, 0.0, 10000.0, rn.HALVES, True)
    un = rn.rope(first, -777, 10000.0, rn.HALVES) / w
    assert not math.isclose(np.mean(un * un), 1.0, rel_tol=1e-12)


def test_planted_page_lookup_fails(monkeypatch):
    Hq, Hkv = 4, 2
    qkv, wq, wk, bt, kc, vc = small_case("bf16", Hq, Hkv)
    res = rn.rope_norm(qkv, wq, wk, [130, 64, 5], None, Hq, Hkv, bt.T.copy()[:3, :3], kc, vc,
                       "bf16", 1.0, 1.0, 1e-6, 10000.0, rn.HALVES, True)
    assert res.slots != [(2, 2), (7, 0), (3, 5)]  # a transposed block table is caught
