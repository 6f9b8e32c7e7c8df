"""Pins for the task-map oracle (CPU only).

The assign rule is the vLLM post's Assign bullet ("The solution: a per-step,
load-balanced decode scheduler") and the SGLang post's live-KV scheduling
section.  The oracle is pinned by (1) a hand-derived worked example,
(2) agreement of two independent constructions, and (3) the defining
properties of the rule checked directly on the produced map.
"""

import os
import random

import numpy as np
import pytest

import oracle
from oracle import assign_closed_form, assign_simulate, static_plan
from oracle.assign import budget_of, tiles_of

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "assign_tiny.txt")


def load_golden():
    desc, bins, head, rest = [], [], None, None
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *nums = line.split()
        nums = [int(x) for x in nums]
        if key == "desc":
            desc.append(tuple(nums[:4]))
            bins.append(nums[4])
        elif key == "bin_ptr_head":
            head = nums
        elif key == "bin_ptr_rest":
            rest = nums[0]
        else:
            vals[key] = nums if len(nums) > 1 else nums[0]
    bin_ptr = head + [rest] * (133 - len(head))
    return desc, bins, bin_ptr, vals


def check_invariants(tm, seqlens, num_kv_heads, num_ctas, floor):
    """Properties that define the fill-and-spill rule, checked on a map."""
    B = len(seqlens)
    n = [oracle.tiles_of(L) for L in seqlens]
    T = num_kv_heads * sum(n)
    assert tm.total_tiles == T
    # the budget is the smallest value >= floor (and >= 1) that lets C bins hold T tiles
    assert tm.budget >= max(floor, 1)
    assert tm.budget * num_ctas >= T
    if tm.budget > max(floor, 1):
        assert (tm.budget - 1) * num_ctas < T
    assert len(tm.bin_ptr) == num_ctas + 1
    assert tm.bin_ptr[0] == 0 and tm.bin_ptr[-1] == tm.num_desc
    assert all(a <= b for a, b in zip(tm.bin_ptr, tm.bin_ptr[1:]))
    # every (h, r, tile) exactly once, walked head-major then batch-minor
    walk = []
    fills = []
    for b in range(num_ctas):
        fill = 0
        for i in range(tm.bin_ptr[b], tm.bin_ptr[b + 1]):
            h, r, tb, te = tm.desc[i]
            assert 0 <= h < num_kv_heads and 0 <= r < B
            assert 0 <= tb < te <= n[r], "empty or out-of-range descriptor"
            walk += [(h, r, t) for t in range(tb, te)]
            fill += te - tb
        fills.append(fill)
    assert walk == [(h, r, t) for h in range(num_kv_heads) for r in range(B) for t in range(n[r])]
    # no bin over budget; every bin before the last used one is full
    assert max(fills, default=0) <= tm.budget
    used = [b for b, f in enumerate(fills) if f > 0]
    if used:
        assert used == list(range(len(used)))
        assert all(f == tm.budget for f in fills[: used[-1]])
    # descriptors break only where a bin or a unit ends
    for b in range(num_ctas):
        ds = tm.desc[tm.bin_ptr[b]:tm.bin_ptr[b + 1]]
        assert len({(h, r) for h, r, _, _ in ds}) == len(ds), "unit split inside one bin"
    # chunk counts and offsets
    assert len(tm.chunk_count) == num_kv_heads * B
    off = 0
    for u in range(num_kv_heads * B):
        h, r = divmod(u, B)
        mine = [i for i, d in enumerate(tm.desc) if (d[0], d[1]) == (h, r)]
        assert tm.chunk_count[u] == len(mine)
        assert tm.chunk_off[u] == off
        assert mine == list(range(off, off + len(mine)))
        off += len(mine)
    # capacity bound used to size the descriptor array
    assert tm.num_desc <= num_ctas + num_kv_heads * B - 1 or tm.num_desc == 0


def test_golden_worked_example():
    desc, bins, bin_ptr, vals = load_golden()
    for build in (assign_closed_form, assign_simulate):
        tm = build([64, 200, 1000, 2048], 1, 132, 2)
        assert tm.total_tiles == vals["total_tiles"]
        assert tm.budget == vals["budget"]
        assert tm.num_desc == vals["num_desc"]
        assert tm.chunk_count == vals["chunk_count"]
        assert tm.chunk_off == vals["chunk_off"]
        assert tm.desc == desc
        assert tm.bin_ptr == bin_ptr
        # the bin column of the fixture agrees with the CSR offsets
        for i, b in enumerate(bins):
            assert bin_ptr[b] <= i < bin_ptr[b + 1]


EDGE_CASES = [
    ([1], 1, 4, 1),
    ([64], 1, 4, 1),
    ([65], 1, 4, 1),
    ([1, 63, 64, 65, 128, 129], 2, 5, 1),
    ([0, 5, 0, 300], 2, 3, 2),  # zero-length requests
    ([0, 0, 0], 4, 8, 2),  # no work at all
    ([4096] * 8, 8, 16, 2),  # uniform
    ([131072] + [4096] * 31, 1, 152, 2),  # one very long request
    ([100] * 3, 1, 1000, 2),  # T < C: floor binds
    ([8192] * 16, 8, 1, 2),  # one CTA takes everything
    ([10, 20000, 30, 70000, 5], 3, 7, 50),  # large floor
]


@pytest.mark.parametrize("seqlens,hkv,ctas,floor", EDGE_CASES)
def test_edge_cases(seqlens, hkv, ctas, floor):
    a = assign_closed_form(seqlens, hkv, ctas, floor)
    b = assign_simulate(seqlens, hkv, ctas, floor)
    assert a == b
    check_invariants(a, seqlens, hkv, ctas, floor)


def test_random_maps_agree_and_hold_invariants():
    rng = random.Random(7)
    for _ in range(150):
        B = rng.randint(1, 24)
        hkv = rng.choice([1, 2, 4, 8])
        ctas = rng.choice([1, 3, 16, 132, 152, 304])
        floor = rng.choice([0, 1, 2, 4, 16])
        kind = rng.random()
        if kind < 0.3:
            lens = [rng.randint(0, 300) for _ in range(B)]
        elif kind < 0.6:
            lens = [int(2 ** rng.uniform(0, 17)) for _ in range(B)]
        else:
            lens = [rng.choice([1, 63, 64, 65, 4096, 50000]) for _ in range(B)]
        a = assign_closed_form(lens, hkv, ctas, floor)
        b = assign_simulate(lens, hkv, ctas, floor)
        assert a == b, (lens, hkv, ctas, floor)
        check_invariants(a, lens, hkv, ctas, floor)


def _mutations(tm):
    """Plausible construction mistakes, planted in copies of a correct map."""
    import copy
    out = []
    m = copy.deepcopy(tm)  # a dropped tile
    h, r, tb, te = m.desc[-1]
    m.desc[-1] = (h, r, tb, te - 1)
    out.append(m)
    m = copy.deepcopy(tm)  # batch-major instead of head-major walk
    m.desc = sorted(m.desc, key=lambda d: (d[1], d[0], d[2]))
    out.append(m)
    m = copy.deepcopy(tm)  # floor budget rounding instead of ceiling
    m.budget -= 1
    out.append(m)
    m = copy.deepcopy(tm)  # an off-by-one chunk offset
    m.chunk_off[1] += 1
    out.append(m)
    return out


def test_invariant_checker_catches_planted_mistakes():
    lens = [1000, 70, 4000, 129]
    tm = assign_closed_form(lens, 2, 12, 1)
    check_invariants(tm, lens, 2, 12, 1)
    for bad in _mutations(tm):
        with pytest.raises(AssertionError):
            check_invariants(bad, lens, 2, 12, 1)


def test_static_plan_properties():
    rng = random.Random(11)
    for _ in range(60):
        B = rng.randint(1, 12)
        hkv = rng.choice([1, 2, 8])
        S = rng.choice([1, 2, 3, 4, 8, 16, 32])
        lens = [rng.choice([0, 1, 64, 65, 700, 4096, 33000]) for _ in range(B)]
        tm = static_plan(lens, hkv, S)
        assert tm.num_desc == hkv * B * S
        assert tm.bin_ptr == list(range(hkv * B * S + 1))
        for u in range(hkv * B):
            h, r = divmod(u, B)
            n = oracle.tiles_of(lens[r])
            ds = tm.desc[u * S:(u + 1) * S]
            assert all((d[0], d[1]) == (h, r) for d in ds)
            assert tm.chunk_off[u] == u * S
            # the splits tile [0, n) in order, equal-sized except the last non-empty one
            covered = [t for d in ds for t in range(d[2], d[3])]
            assert covered == list(range(n))
            sizes = [d[3] - d[2] for d in ds]
            nonempty = [s for s in sizes if s > 0]
            assert tm.chunk_count[u] == len(nonempty) <= S
            assert sizes[:len(nonempty)] == nonempty, "empty split before a non-empty one"
            if nonempty:
                assert all(s == nonempty[0] for s in nonempty[:-1])
                assert nonempty[-1] <= nonempty[0]
                # fixed split count: the chunk is the smallest that covers n in S pieces
                assert nonempty[0] * S >= n and (nonempty[0] - 1) * S < n


def bin_from_lengths(seqlens, hkv, ctas, floor, c):
    """Bin c's descriptors with their map indices and chunk layouts, from the
    lengths alone, by the identities the attention kernel uses before the
    assign kernel's map is visible: every bin before c holds one descriptor
    plus one per unit with tiles starting strictly inside it, so bin c's first
    descriptor is c + #(such starts before tile c * budget); a unit spans bins
    first .. last, its chunks consecutive in the map, and its descriptor in
    bin c is chunk c - first."""
    n = [tiles_of(L) for L in seqlens]
    N = sum(n)
    T = hkv * N
    b = budget_of(T, ctas, floor)
    X = c * b
    if X >= T:
        return []
    pre = [sum(n[:r]) for r in range(len(n))]
    starts = [h * N + pre[r] for h in range(hkv) for r in range(len(n)) if n[r] > 0]
    base = c + sum(1 for s in starts if s < X and s % b != 0)
    out, t, end = [], X, min(X + b, T)
    h, tl = divmod(t, N)
    r = next(i for i in range(len(n)) if pre[i] + n[i] > tl)
    tb = tl - pre[r]
    while t < end:
        te = tb + min(n[r] - tb, end - t)
        s = h * N + pre[r]
        first, last = s // b, (s + n[r] - 1) // b
        idx = base + len(out)
        out.append(((h, r, tb, te), idx, last - first + 1, idx - (c - first)))
        t += te - tb
        while t < end:
            r += 1
            if r == len(n):
                r, h = 0, h + 1
            if n[r] > 0:
                break
        tb = 0
    return out


@pytest.mark.parametrize("seed", range(40))
def test_a_bin_follows_from_the_lengths_alone(seed):
    """The identities hold on random batches: each bin's descriptors, their
    indices in the map and their units' chunk counts and first chunks equal
    the closed-form map's (empty requests, floors and bins past the last
    tile included)."""
    rng = np.random.default_rng(4000 + seed)
    B = int(rng.integers(1, 65))
    hkv = int(rng.choice([1, 2, 4, 8]))
    ctas = int(rng.choice([8, 37, 132, 152]))
    floor = int(rng.choice([1, 2, 5]))
    seqlens = [int(x) for x in rng.integers(0, 3000, B)]
    if seed % 3 == 0:
        seqlens[int(rng.integers(0, B))] = int(rng.integers(20000, 140000))
    if seed % 5 == 0:
        seqlens = [0 if rng.random() < 0.3 else L for L in seqlens]
    tm = assign_closed_form(seqlens, hkv, ctas, floor)
    for c in range(ctas):
        got = bin_from_lengths(seqlens, hkv, ctas, floor, c)
        want = []
        for d in range(tm.bin_ptr[c], tm.bin_ptr[c + 1]):
            h, r, tb, te = tm.desc[d]
            u = h * B + r
            want.append(((h, r, tb, te), d, tm.chunk_count[u], tm.chunk_off[u]))
        assert got == want, (c, got, want)
