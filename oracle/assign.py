"""Task-map oracle for the load-balanced assign step and the static split-KV plan.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may use this module; the product path never does.

The load-balanced rule follows the vLLM integration post ("The solution: a
per-step, load-balanced decode scheduler", Assign bullet) and the SGLang post
(section on scheduling around live KV work):

  * every request's live KV is cut into uniform 64-token tiles,
    n_r = ceil(L_r / 64) (a partial last tile counts as a whole tile);
  * tiles are counted over all KV heads and requests, T = Hkv * sum_r n_r;
  * the per-CTA budget ("bucket size") is T divided by the number of
    persistent CTAs, rounded up, and raised to a minimum-work floor;
    a budget of at least one tile is implied whenever T = 0;
  * tiles are walked head-major, batch-minor (unit u = h * B + r) and poured
    into CTA bins in order; a full bin spills into the next one;
  * the task map lists, bin by bin, (kv_head, request, tile_begin, tile_end)
    descriptors, one per non-empty intersection of a unit with a bin, plus
    the chunk count of every (head, request) unit.

Readings where the pages are silent (stated, not printed on the pages):
  heads = KV heads (one descriptor serves the whole GQA group); the budget
  division rounds up; descriptors split only at bin or unit boundaries;
  bins after the last used one are empty; L = 0 gives no tiles.

The static split-KV comparator follows the pages' "fixed number of splits"
strategy (vLLM post, "The challenge"; SGLang post, the static split-KV
paragraph): split s of request r covers tiles [s*k_r, min((s+1)*k_r, n_r))
with k_r = ceil(n_r / S); every (head, request, split) gets its own CTA.

Two load-balanced constructions are given on purpose: a closed form per unit
and a tile-by-tile simulation of the fill-and-spill rule.  They share nothing
but the tile count and the budget.
"""

from __future__ import annotations

from dataclasses import dataclass, field

TILE = 64


def tiles_of(length: int) -> int:
    """Number of 64-token tiles holding `length` live tokens (0 for L <= 0)."""
    if length <= 0:
        return 0
    return (length + TILE - 1) // TILE


def budget_of(total_tiles: int, num_ctas: int, floor: int) -> int:
    """Per-CTA tile budget: ceil(T / C) raised to the floor (and to 1)."""
    return max((total_tiles + num_ctas - 1) // num_ctas, floor, 1)


@dataclass
class TaskMap:
    """A task map in plain Python lists.

    desc:        list of (kv_head, request, tile_begin, tile_end), bin-major.
    bin_ptr:     CSR offsets, length num_bins + 1; bin b owns desc[bin_ptr[b]:bin_ptr[b+1]].
    chunk_count: per unit u = h * B + r, number of descriptors of that unit.
    chunk_off:   per unit, index of the unit's first descriptor.
    total_tiles, budget: T and the per-bin budget (static plan: budget = S).
    """

    desc: list = field(default_factory=list)
    bin_ptr: list = field(default_factory=list)
    chunk_count: list = field(default_factory=list)
    chunk_off: list = field(default_factory=list)
    total_tiles: int = 0
    budget: int = 0

    @property
    def num_desc(self) -> int:
        return len(self.desc)


def assign_closed_form(seqlens, num_kv_heads: int, num_ctas: int, floor: int) -> TaskMap:
    """Load-balanced task map, computed unit by unit from each unit's first tile index."""
    B = len(seqlens)
    n = [tiles_of(int(L)) for L in seqlens]
    per_head = sum(n)
    T = num_kv_heads * per_head
    b = budget_of(T, num_ctas, floor)
    tm = TaskMap(total_tiles=T, budget=b)
    bin_of_desc = []
    start = 0  # global index of the unit's first tile
    for h in range(num_kv_heads):
        for r in range(B):
            nu = n[r]
            tm.chunk_off.append(len(tm.desc))
            if nu == 0:
                tm.chunk_count.append(0)
                continue
            first_bin = start // b
            last_bin = (start + nu - 1) // b
            tm.chunk_count.append(last_bin - first_bin + 1)
            for bin_id in range(first_bin, last_bin + 1):
                lo = max(start, bin_id * b)
                hi = min(start + nu, (bin_id + 1) * b)
                tm.desc.append((h, r, lo - start, hi - start))
                bin_of_desc.append(bin_id)
            start += nu
    tm.bin_ptr = _csr_from_bins(bin_of_desc, num_ctas)
    return tm


def assign_simulate(seqlens, num_kv_heads: int, num_ctas: int, floor: int) -> TaskMap:
    """Load-balanced task map, built by pouring tiles one at a time into bins."""
    B = len(seqlens)
    n = [tiles_of(int(L)) for L in seqlens]
    T = num_kv_heads * sum(n)
    b = budget_of(T, num_ctas, floor)
    tm = TaskMap(total_tiles=T, budget=b)
    bins = [[] for _ in range(num_ctas)]  # each bin: list of [h, r, begin, end]
    current, fill = 0, 0
    for h in range(num_kv_heads):
        for r in range(B):
            for j in range(n[r]):
                if fill == b:  # bin full: spill into the next one
                    current += 1
                    fill = 0
                cur = bins[current]
                if cur and cur[-1][0] == h and cur[-1][1] == r and cur[-1][3] == j:
                    cur[-1][3] = j + 1
                else:
                    cur.append([h, r, j, j + 1])
                fill += 1
    for bin_list in bins:
        tm.bin_ptr.append(len(tm.desc))
        tm.desc.extend(tuple(d) for d in bin_list)
    tm.bin_ptr.append(len(tm.desc))
    counts = [0] * (num_kv_heads * B)
    offs = [-1] * (num_kv_heads * B)
    for i, (h, r, _, _) in enumerate(tm.desc):
        u = h * B + r
        if offs[u] < 0:
            offs[u] = i
        counts[u] += 1
    # a unit without descriptors points at the next unit's first descriptor
    nxt = len(tm.desc)
    for u in range(num_kv_heads * B - 1, -1, -1):
        if offs[u] < 0:
            offs[u] = nxt
        nxt = offs[u]
    tm.chunk_count, tm.chunk_off = counts, offs
    return tm


def static_plan(seqlens, num_kv_heads: int, num_splits: int) -> TaskMap:
    """Static fixed-split schedule: one descriptor (possibly empty) per (h, r, split)."""
    B = len(seqlens)
    S = num_splits
    n = [tiles_of(int(L)) for L in seqlens]
    tm = TaskMap(total_tiles=num_kv_heads * sum(n), budget=S)
    for h in range(num_kv_heads):
        for r in range(B):
            per_split = (n[r] + S - 1) // S
            nonempty = 0
            tm.chunk_off.append(len(tm.desc))
            for s in range(S):
                lo = min(s * per_split, n[r])
                hi = min((s + 1) * per_split, n[r])
                tm.desc.append((h, r, lo, hi))
                nonempty += hi > lo
            tm.chunk_count.append(nonempty)
    tm.bin_ptr = list(range(len(tm.desc) + 1))
    return tm


def _csr_from_bins(bin_of_desc, num_bins):
    ptr = [0] * (num_bins + 1)
    for b in bin_of_desc:
        ptr[b + 1] += 1
    for i in range(num_bins):
        ptr[i + 1] += ptr[i]
    return ptr
