"""Seeded synthetic decode batches.

This module only draws inputs; it holds none of the attention or assign
arithmetic, and it is the one piece of Python shared by the CUDA path, the
oracle-based tests and the benchmark.

The workloads stand in for the pages' mixed-length decode batches (vLLM
integration post, Table 3 and "The challenge: mixed-length decode in every
batch"; Hy3's GQA shape of 64 query heads, 8 KV heads, head dim 128 from
"A Quick Word on Hy3-series models", sliced 8-way for a TP8 GPU).  There is
no dataset: lengths, page placement and values are drawn from seeds.

Recipe (draw order: seqlens, page permutation, Q, K, V):
  * seqlens from a CPU torch.Generator seeded with the config's seed;
    log-uniform lengths are floor(exp(U(ln a, ln b))), uniform ones are
    integer-uniform on [a, b];
  * pages: P = sum_r ceil(L_r / 64) physical pages; a random permutation of
    [0, P) is handed out to the requests in request order; unused
    block-table entries are -1;
  * Q ~ N(0, 1) from the same CPU generator, [B, Hq, 128], or
    [B, q_len, Hq, 128] for multi-query decode (q_len > 1: the request's
    last q_len live tokens are the queries);
  * K, V ~ N(0, 1), drawn on the target device from a generator seeded with
    seed + 1 (K) and seed + 2 (V); slots past L_r in a request's last page
    are part of the draw, or are poisoned (NaN / the E4M3 NaN code) on request;
  * BF16 tensors are the fp32 draws rounded to BF16;
  * FP8-E4M3: K and V scaled by a per-tensor scale amax / 448, Q by a
    per-(token, head) scale amax_row / 448, then converted with torch's
    float8_e4m3fn cast (round to nearest even).  This stands in for the
    fused prologue that emits FP8 Q and writes the FP8 cache, which lies
    outside this path.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEAD_DIM = 128
PAGE = 64


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    seqlens: tuple = ()  # explicit lengths, or empty when drawn
    draw: tuple = ()  # ((count, kind, a, b), ...), kind in {"log", "uniform", "fixed"}
    kv_dtype: str = "bf16"  # "bf16" or "e4m3"
    seed: int = 1000
    num_ctas: int = 0  # 0: one persistent CTA per resident slot on the GPU
    min_tiles: int = 2
    description: str = ""
    q_len: int = 1  # query tokens per request (> 1: speculative / MTP decode)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(HEAD_DIM)


WORKLOADS = {
    "tiny": Workload(
        "tiny", 4, 8, 1, seqlens=(64, 200, 1000, 2048), seed=1001, num_ctas=132, min_tiles=2,
        description="tiny BF16 paged GQA decode, B=4, L={64,200,1000,2048}, Hq=8, Hkv=1, "
                    "132 persistent CTAs, floor 2"),
    "hy3_tp8": Workload(
        "hy3_tp8", 32, 8, 1, draw=((32, "log", 1024, 32768),), seed=1002,
        description="Hy3-shaped TP8 slice, BF16, B=32, Hq=8, Hkv=1, L log-uniform [1K, 32K]"),
    "skewed": Workload(
        "skewed", 64, 64, 8, draw=((60, "uniform", 512, 2048), (4, "uniform", 65536, 131072)),
        seed=1003,
        description="skewed BF16 TP1 shape, B=64, Hq=64, Hkv=8, 60 x U[512,2K] + 4 x U[64K,128K]"),
    "uniform": Workload(
        "uniform", 16, 64, 8, draw=((16, "fixed", 8192, 8192),), seed=1004,
        description="uniform-length control, BF16, B=16, L=8192, Hq=64, Hkv=8"),
    "fp8": Workload(
        "fp8", 64, 8, 1, draw=((64, "log", 1024, 131072),), kv_dtype="e4m3", seed=1005,
        description="FP8-E4M3 KV and Q, B=64, Hq=8, Hkv=1, L log-uniform [1K, 128K]"),
}

# The six KV-length mixes of the vLLM post's Table 3 (FP8 decode), at the
# TP8 head shape.  A x B means A requests at KV length B.
TABLE3 = {
    "t3_64x0.5k": ((64, "fixed", 512, 512),),
    "t3_64x4k": ((64, "fixed", 4096, 4096),),
    "t3_32x0.125k_32x4k": ((32, "fixed", 128, 128), (32, "fixed", 4096, 4096)),
    "t3_2x32k_30x4k": ((2, "fixed", 32768, 32768), (30, "fixed", 4096, 4096)),
    "t3_1x64k_15x4k": ((1, "fixed", 65536, 65536), (15, "fixed", 4096, 4096)),
    "t3_1x128k_31x4k": ((1, "fixed", 131072, 131072), (31, "fixed", 4096, 4096)),
}
for _i, (_name, _draw) in enumerate(TABLE3.items()):
    WORKLOADS[_name] = Workload(_name, sum(c for c, *_ in _draw), 8, 1, draw=_draw,
                                kv_dtype="e4m3", seed=1100 + _i,
                                description=f"Table-3 mix {_name[3:]}, FP8, Hq=8, Hkv=1")


# The prefill and extend rows of the vLLM post's attention comparison (Table
# 4): "qAsB" is q_len = A new tokens over a request of B tokens (a cached
# prefix of B - A), "qA prefill" is q_len = L = A, the leading number is the
# batch.  The table gives neither heads nor precision; these take Hy3's TP1
# GQA shape (64 query heads, 8 KV heads, head dim 128) in BF16.
TABLE4_PREFILL = {
    "t4_q512": (1, 512, 512),
    "t4_q1ks2k": (1, 1024, 2048),
    "t4_q2k": (1, 2048, 2048),
    "t4_q4k": (1, 4096, 4096),
    "t4_q8k": (1, 8192, 8192),
    "t4_2q1ks4k": (2, 1024, 4096),
}
for _i, (_name, (_b, _q, _l)) in enumerate(TABLE4_PREFILL.items()):
    WORKLOADS[_name] = Workload(_name, _b, 64, 8, draw=((_b, "fixed", _l, _l),), seed=1300 + _i,
                                q_len=_q,
                                description=f"Table-4 {'extend' if _q < _l else 'prefill'} "
                                            f"{_name[3:]}: B={_b}, q_len={_q}, L={_l}, Hq=64, "
                                            f"Hkv=8, BF16")


# The decode rows of the same table ("Bq1sL": batch B, one query token, KV
# length L), at the same head shape.  The H20 latencies fit it: 64q1s4k moves
# 1.07 GB of BF16 KV in 0.299 ms (~3.6 TB/s on a 4 TB/s part).
TABLE4_DECODE = {
    "t4_8q1s1k": (8, 1024),
    "t4_16q1s2k": (16, 2048),
    "t4_32q1s1k": (32, 1024),
    "t4_64q1s4k": (64, 4096),
}
for _i, (_name, (_b, _l)) in enumerate(TABLE4_DECODE.items()):
    WORKLOADS[_name] = Workload(_name, _b, 64, 8, draw=((_b, "fixed", _l, _l),), seed=1400 + _i,
                                description=f"Table-4 decode {_name[3:]}: B={_b}, L={_l}, Hq=64, "
                                            f"Hkv=8, BF16")


def draw_seqlens(w: Workload, gen: torch.Generator) -> list:
    if w.seqlens:
        return [int(x) for x in w.seqlens]
    out = []
    for count, kind, a, b in w.draw:
        if kind == "fixed":
            out += [int(a)] * count
        elif kind == "uniform":
            out += torch.randint(a, b + 1, (count,), generator=gen).tolist()
        elif kind == "log":
            u = torch.rand(count, generator=gen, dtype=torch.float64)
            out += [int(math.floor(math.exp(math.log(a) + float(x) * (math.log(b) - math.log(a)))))
                    for x in u]
        else:
            raise ValueError(kind)
    return out


@dataclass
class Batch:
    """One decode batch.  Tensors live on `device`; CPU copies are made on demand."""

    workload: Workload
    seqlens: torch.Tensor  # int32 [B]
    block_table: torch.Tensor  # int32 [B, max_pages], -1 past each request's pages
    q: torch.Tensor  # bf16 or float8_e4m3fn [B, Hq, 128] ([B, q_len, Hq, 128] for q_len > 1)
    k_cache: torch.Tensor  # bf16 or float8_e4m3fn [P, 64, Hkv, 128]
    v_cache: torch.Tensor
    q_scale: torch.Tensor | None = None  # fp32 [B, Hq] ([B, q_len, Hq] for q_len > 1; FP8 only)
    k_scale: float = 1.0
    v_scale: float = 1.0
    extras: dict = field(default_factory=dict)

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def live_tokens(self) -> int:
        return int(self.seqlens.sum().item())

    def oracle_kwargs(self) -> dict:
        w = self.workload
        fp8 = w.kv_dtype == "e4m3"
        return dict(num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, sm_scale=w.sm_scale,
                    q_dtype=1 if fp8 else 0, kv_dtype=1 if fp8 else 0,
                    q_scale=None if self.q_scale is None else self.q_scale.cpu(),
                    k_scale=self.k_scale, v_scale=self.v_scale)


def _normal(shape, seed, device):
    gen = torch.Generator(device=device).manual_seed(seed)
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def make_batch(w: Workload, device="cpu", seed: int | None = None, poison_tail: bool = False,
               seqlens: list | None = None, extra_pages: int = 0) -> Batch:
    """Draw one batch of workload `w` (optionally with explicit seqlens)."""
    seed = w.seed if seed is None else seed
    gen = torch.Generator().manual_seed(seed)
    lens = draw_seqlens(w, gen) if seqlens is None else [int(x) for x in seqlens]
    B = len(lens)
    pages_per = [(L + PAGE - 1) // PAGE if L > 0 else 0 for L in lens]
    total_pages = sum(pages_per) + extra_pages
    perm = torch.randperm(max(total_pages, 1), generator=gen)[:total_pages]
    max_pages = max(max(pages_per, default=0), 1)
    bt = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for r, n in enumerate(pages_per):
        bt[r, :n] = perm[off:off + n].to(torch.int32)
        off += n
    Hq, Hkv = w.num_q_heads, w.num_kv_heads
    q_shape = (B, Hq, HEAD_DIM) if w.q_len == 1 else (B, w.q_len, Hq, HEAD_DIM)
    q32 = torch.randn(q_shape, generator=gen, dtype=torch.float32)
    kv_shape = (max(total_pages, 1), PAGE, Hkv, HEAD_DIM)
    k32 = _normal(kv_shape, seed + 1, device)
    v32 = _normal(kv_shape, seed + 2, device)
    fp8 = w.kv_dtype == "e4m3"
    batch_kw = {}
    if fp8:
        e4m3 = torch.float8_e4m3fn
        q_amax = q32.abs().amax(dim=-1).clamp_min(1e-12)
        q_scale = (q_amax / 448.0).to(torch.float32)
        q = (q32 / q_scale[..., None]).to(e4m3)
        k_scale = float(k32.abs().max().item()) / 448.0
        v_scale = float(v32.abs().max().item()) / 448.0
        k = (k32 / k_scale).to(e4m3)
        v = (v32 / v_scale).to(e4m3)
        batch_kw = dict(q_scale=q_scale.to(device), k_scale=k_scale, v_scale=v_scale)
    else:
        q = q32.to(torch.bfloat16)
        k = k32.to(torch.bfloat16)
        v = v32.to(torch.bfloat16)
    del k32, v32
    if poison_tail:
        _poison_tails(k, v, bt, lens)
    return Batch(w, torch.tensor(lens, dtype=torch.int32).to(device), bt.to(device), q.to(device),
                 k, v, **batch_kw)


def _poison_tails(k, v, bt, lens):
    """Fill the unused slots of every last page with NaN (the E4M3 NaN code for FP8)."""
    for r, L in enumerate(lens):
        if L <= 0 or L % PAGE == 0:
            continue
        page = int(bt[r, (L - 1) // PAGE])
        for t in (k, v):
            if t.dtype == torch.float8_e4m3fn:
                t.view(torch.uint8)[page, L % PAGE:] = 0x7F
            else:
                t[page, L % PAGE:] = float("nan")


# ---------------------------------------------------------------- prologue
# Inputs of the fused attention prologue (QK-Norm, RoPE, paged KV write, FP8
# query), which produces the decode path's Q and the new token's cache rows.
# The pages give its shapes (the Hy3 head layout) but none of its constants:
# RoPE base, epsilon and norm weights are synthetic.
#
# Recipe: the fused QKV rows are N(0, 1) draws; each query and key head row
# is multiplied by its own magnitude, log-uniform on [1/4, 8], so that the
# norm has something to undo (value rows keep unit scale); the norm weights
# are 1 + N(0, 1)/4; all rounded to BF16.  Decode: one new token per request
# of a decode workload, at position L_r - 1 of that request's pages (it
# overwrites the slot the batch drew there).  Prefill: one request of N
# tokens at positions 0..N-1 over a shuffled page list, the caches starting
# at zero; FP8 cache scales are fixed at 8/448 for K (normalised rows stay
# within about 8) and amax(V)/448 for V.


@dataclass(frozen=True)
class PrologueWorkload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    kv_dtype: str = "bf16"
    decode_of: str = ""  # decode: one new token per request of this decode workload
    prefill_tokens: int = 0  # prefill: one request of this many tokens
    rope_base: float = 1e6
    eps: float = 1e-6
    rope_layout: int = 0  # 0: pairs (i, i + 64); 1: pairs (2i, 2i + 1)
    norm_first: bool = True
    seed: int = 1200
    description: str = ""


PROLOGUES = {
    "decode_hy3_tp8": PrologueWorkload(
        "decode_hy3_tp8", 8, 1, decode_of="hy3_tp8", seed=1201,
        description="prologue of one decode step of hy3_tp8: 32 tokens, Hq=8, Hkv=1, BF16"),
    "decode_fp8": PrologueWorkload(
        "decode_fp8", 8, 1, kv_dtype="e4m3", decode_of="fp8", seed=1202,
        description="prologue of one decode step of the FP8 workload: 64 tokens, Hq=8, Hkv=1"),
    "prefill_8k_fp8": PrologueWorkload(
        "prefill_8k_fp8", 64, 8, kv_dtype="e4m3", prefill_tokens=8192, seed=1203,
        description="8K-token prefill prologue at the Hy3 TP1 head shape (Hq=64, Hkv=8), FP8"),
    "prefill_8k_bf16": PrologueWorkload(
        "prefill_8k_bf16", 64, 8, prefill_tokens=8192, seed=1204,
        description="8K-token prefill prologue at the Hy3 TP1 head shape (Hq=64, Hkv=8), BF16"),
}


@dataclass
class PrologueInputs:
    workload: PrologueWorkload
    qkv: torch.Tensor  # bf16 [N, (Hq + 2 Hkv) * 128]
    q_norm_w: torch.Tensor  # bf16 [128]
    k_norm_w: torch.Tensor  # bf16 [128]
    positions: torch.Tensor  # int32 [N]
    token_req: torch.Tensor | None  # int32 [N], or None: token t is request t
    block_table: torch.Tensor  # int32 [B, max_pages]
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_scale: float
    v_scale: float
    batch: Batch | None = None  # the decode batch whose caches are written

    @property
    def num_tokens(self) -> int:
        return int(self.positions.numel())


def draw_qkv(N: int, Hq: int, Hkv: int, seed: int, device) -> tuple:
    """(qkv bf16 [N, (Hq + 2 Hkv) * 128], q_norm_w, k_norm_w) per the recipe above."""
    gen = torch.Generator().manual_seed(seed)
    R = Hq + 2 * Hkv
    mag = torch.exp(torch.empty((N, Hq + Hkv, 1)).uniform_(math.log(0.25), math.log(8.0),
                                                           generator=gen))
    mag = torch.cat([mag, torch.ones((N, Hkv, 1))], dim=1)
    rows = _normal((N, R, HEAD_DIM), seed + 1, device) * mag.to(device)
    qkv = rows.to(torch.bfloat16).reshape(N, R * HEAD_DIM)
    wq = (1.0 + 0.25 * torch.randn(HEAD_DIM, generator=gen)).to(torch.bfloat16).to(device)
    wk = (1.0 + 0.25 * torch.randn(HEAD_DIM, generator=gen)).to(torch.bfloat16).to(device)
    return qkv, wq, wk


def make_prologue_inputs(pw: PrologueWorkload, device="cpu", seed: int | None = None,
                         seqlens: list | None = None) -> PrologueInputs:
    seed = pw.seed if seed is None else seed
    Hq, Hkv = pw.num_q_heads, pw.num_kv_heads
    if pw.decode_of:
        w = WORKLOADS[pw.decode_of]
        batch = make_batch(w, device=device, seqlens=seqlens)
        N = int(batch.seqlens.numel())
        qkv, wq, wk = draw_qkv(N, Hq, Hkv, seed, device)
        positions = (batch.seqlens - 1).to(torch.int32)
        return PrologueInputs(pw, qkv, wq, wk, positions, None, batch.block_table,
                              batch.k_cache, batch.v_cache, batch.k_scale, batch.v_scale, batch)
    N = pw.prefill_tokens
    gen = torch.Generator().manual_seed(seed + 7)
    pages = (N + PAGE - 1) // PAGE
    bt = torch.randperm(pages, generator=gen).to(torch.int32).reshape(1, pages).to(device)
    qkv, wq, wk = draw_qkv(N, Hq, Hkv, seed, device)
    shape = (pages, PAGE, Hkv, HEAD_DIM)
    fp8 = pw.kv_dtype == "e4m3"
    dtype = torch.float8_e4m3fn if fp8 else torch.bfloat16
    k_cache = torch.zeros(shape, dtype=dtype, device=device)
    v_cache = torch.zeros(shape, dtype=dtype, device=device)
    k_scale = v_scale = 1.0
    if fp8:
        k_scale = 8.0 / 448.0
        v_rows = qkv.reshape(N, Hq + 2 * Hkv, HEAD_DIM)[:, Hq + Hkv:]
        v_scale = float(v_rows.float().abs().max().item()) / 448.0
    positions = torch.arange(N, dtype=torch.int32, device=device)
    token_req = torch.zeros(N, dtype=torch.int32, device=device)
    return PrologueInputs(pw, qkv, wq, wk, positions, token_req, bt, k_cache, v_cache, k_scale,
                          v_scale)


# ---------------------------------------------------------------- router GEMM
# Inputs of the router GEMM (BF16 hidden states x FP32 router weights), at
# the SGLang post's router shape: K = 4096 hidden, N = 192 experts, M tokens.
# Recipe: X ~ N(0, 1) rounded to BF16 [M, K]; W ~ N(0, 1/K) in FP32 [N, K]
# (a Linear layer's weight), so the scores are about N(0, 1).  The post's
# sweep prints no M values; the workloads span decode (a few tokens) to
# prefill (thousands).

ROUTER_K, ROUTER_N = 4096, 192
ROUTER_MS = (1, 16, 64, 256, 1024, 4096, 16384)


def make_router_inputs(M: int, K: int = ROUTER_K, N: int = ROUTER_N, seed: int = 1300,
                       device="cpu") -> tuple:
    """(x bf16 [M, K], w fp32 [N, K]) per the recipe above."""
    gen = torch.Generator().manual_seed(seed)
    w = (torch.randn((N, K), generator=gen, dtype=torch.float32) / math.sqrt(K)).to(device)
    x = _normal((M, K), seed + 1, device).to(torch.bfloat16)
    return x, w
