"""Benchmark: one decode step (assign + persistent attention + combine) of a
synthetic mixed-length batch on GB300, timed on the device.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline] [--no-static] ...

The headline workload defaults to `skewed` (B = 64, Hq = 64, Hkv = 8, BF16,
60 short + 4 very long requests: the largest single-GPU configuration).
Prints one JSON line (rank 0).  `value` is device-timed microseconds per
step; `roofline` relates the attention kernel's algorithmic bytes per launch
to its CUDA-event duration and the measured HBM copy peak; `e2e` is the same
step through the host-buffer C entry point with the per-step inputs copied in
and the output copied out inside the timed region; `cpu_baseline` is the fp64
oracle timed on a bounded sample on the host cores; `static` is the in-house
static split-KV schedule on the same batch.  Side legs: the fused prologue
(`rope_norm`), multi-query decode (`mtp`), the router GEMM sweep
(`router_gemm`), extend / prefill attention on the vLLM comparison's
shapes (`prefill`, TFLOP/s against the measured BF16 tensor peak) and that
table's decode rows (`table4_decode`, with the best static split-KV).  The
line ends with two compact objects: `table3` (the six KV-length mixes of the
vLLM post's Table 3, FP8, dynamic against the best static split) and
`per_config` (every decode workload: step and attention time, attention
bytes and fraction of the copy peak, best static split and the speed-up over
it).  Under torchrun every rank runs an independent replica (the path has no
exchange step).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 2 * 129 * 1024 * 1024  # twice the GB300 L2
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "decode-attn µs/step and achieved HBM GB/s (% of GB300 peak) on mixed-length batches"


# ------------------------------------------------------------------ byte model
def algorithmic_bytes(seqlens, Hq, Hkv, kv_dtype, num_desc, split_desc, q_len=1):
    """Bytes each kernel must move at minimum.

    KV: every live token's K and V row of every KV head once,
      sum_r L_r * Hkv * 128 * 2 * bpe;  Q: B * q_len * Hq * 128 * bpe (+ fp32
      q-scales for FP8);  out: B * q_len * Hq * 128 * 2;  a partial:
      q_len * G * (128 + 1) * 4 (q_len query tokens per request, 1 for decode).
    attn (separate combine): KV + Q + one partial written per descriptor.
    combine: those partials read + out.
    attn_fused (the launch the roofline uses): KV + Q + out + the partials of
      split units written and read back (a unit with one chunk writes its
      output directly).
    step: the timed step, assign + fused attention (the task map is a few KB).
    Block table and seqlens (a few KB) are not counted.
    """
    bpe = 1 if kv_dtype == "e4m3" else 2
    B = len(seqlens)
    rows = q_len * (Hq // Hkv)  # query rows per KV head (q_len query tokens per request)
    kv = sum(seqlens) * Hkv * 128 * 2 * bpe
    q = B * q_len * Hq * 128 * bpe + (B * q_len * Hq * 4 if kv_dtype == "e4m3" else 0)
    part = rows * (128 + 1) * 4
    out = B * q_len * Hq * 128 * 2
    fused = kv + q + out + 2 * split_desc * part
    return {"kv": kv, "q": q, "partials": num_desc * part, "out": out,
            "attn": kv + q + num_desc * part, "combine": num_desc * part + out,
            "attn_fused": fused, "step": fused}


def aggregate(per_rank_us, per_rank_bytes):
    """Replica aggregation: the step time is the slowest rank's; bytes add up."""
    t = max(per_rank_us)
    return t, sum(per_rank_bytes) / (t * 1e-6) / 1e9


def prologue_bytes(N, Hq, Hkv, kv_dtype):
    """Bytes the fused prologue must move for N tokens: the fused QKV rows in,
    the query (+ fp32 scales for FP8) and the new K and V cache rows out, plus
    each token's position and block-table entry and the two norm weights."""
    bpe = 1 if kv_dtype == "e4m3" else 2
    read = N * (Hq + 2 * Hkv) * 128 * 2 + N * 8 + 2 * 128 * 2
    write = N * Hq * 128 * bpe + (N * Hq * 4 if kv_dtype == "e4m3" else 0) + \
        N * 2 * Hkv * 128 * bpe
    return read + write


# ------------------------------------------------------------------ environment
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense BF16 tensor peak (burst, for a kernel timed alone)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def router_cost(M, N, K, splits):
    """FLOPs (two BF16 products) and algorithmic bytes of one router GEMM:
    X once, W_high and W_low once, the scores written, plus the split-K
    partials written and read back when the K range is split."""
    flops = 2 * 2 * M * N * K
    nbytes = M * K * 2 + 2 * N * K * 2 + M * N * 4 + (2 * splits * M * N * 4 if splits > 1 else 0)
    return flops, nbytes


def prefill_flops(seqlens, q_len, Hq):
    """FLOPs of causal extend / prefill attention: query token i of a request
    of L tokens sees max(0, L - q_len + 1 + i) tokens; each (row, token) pair
    costs 2 * 128 for Q K^T and 2 * 128 for P V."""
    pairs = 0
    for L in seqlens:
        for_all = max(0, L - q_len + 1)  # tokens seen by query 0 (when L >= q_len)
        if L >= q_len:
            pairs += q_len * for_all + q_len * (q_len - 1) // 2
        else:
            n = L  # queries q_len - L .. q_len - 1 see 1 .. L tokens
            pairs += n * (n + 1) // 2
    return 4 * 128 * Hq * pairs


def profiled_traffic(kernel_src_hash, kv_dtype, workload):
    """DRAM bytes per attention launch from the committed ncu capture of this
    workload (the JSON sidecar next to its summary under profiles/), if it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"attn_{kv_dtype.replace('e4m3', 'fp8')}_{workload}.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256") != kernel_src_hash:
        return None
    try:
        return float(d["dram_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


_CODE_TOKENS = re.compile(r'"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'|//[^\n]*|/\*.*?\*/', re.S)


def code_only(src):
    """C/CUDA source without its comments, trailing blanks and empty lines
    (string and character literals kept): what a capture's counters depend on."""
    text = _CODE_TOKENS.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", src)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash():
    """sha256 of the attention kernel's code (comments and blank lines excluded)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "load_balanced_paged_assign_gb300", "csrc")
    for name in ("attn_kernel.cuh", "attn_bf16.cu", "attn_fp8.cu", "ptx.cuh"):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi samples (every 20 ms) with host timestamps, kept while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={device_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        return self.summary_over([(t0, t1)])

    def summary_over(self, intervals):
        """Samples whose host timestamp falls inside any of the intervals."""
        inside = [p for t, p in self.samples if any(a <= t <= b for a, b in intervals)]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(p[0]) for p in inside]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in inside for n, v in zip(names, p[4:8]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": num(inside[0][1]),
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max(num(p[2]) for p in inside)}


# ------------------------------------------------------------------ oracle timing
class OracleTimer:
    """Times the oracle as it stands on bounded samples of (request, query
    head) rows and extrapolates to the whole step by work (a row's work is its
    live length)."""

    def __init__(self, batch):
        import numpy as np

        import oracle
        self.np, self.oracle = np, oracle
        w = batch.workload
        self.w = w
        self.lens = batch.seqlens.cpu().tolist()
        self.rows_all = np.arange(len(self.lens) * w.num_q_heads)
        self.work = np.array([self.lens[r // w.num_q_heads] for r in self.rows_all],
                             dtype=np.float64)
        self.total_work = float(self.work.sum())
        self.kw = batch.oracle_kwargs()
        self.cpu = dict(q=batch.q.cpu(), k_cache=batch.k_cache.cpu(),
                        v_cache=batch.v_cache.cpu(), block_table=batch.block_table.cpu(),
                        seqlens=batch.seqlens.cpu())
        probe = np.random.default_rng(12345).permutation(self.rows_all)[:64]
        t = time.perf_counter()
        self.oracle.attention(rows=probe, **self.cpu, **self.kw)
        self.per_work = (time.perf_counter() - t) / max(float(self.work[probe].sum()), 1.0)

    def run(self, budget_s, seed=0):
        np = self.np
        order = np.random.default_rng(seed).permutation(self.rows_all)
        n_rows = len(order)
        if self.per_work * self.total_work > budget_s:
            cum = np.cumsum(self.work[order])
            n_rows = min(int(np.searchsorted(cum, budget_s / self.per_work)) + 1, len(order))
        rows = np.sort(order[:n_rows])
        t = time.perf_counter()
        self.oracle.attention(rows=rows, **self.cpu, **self.kw)
        dt = time.perf_counter() - t
        t = time.perf_counter()
        self.oracle.assign_closed_form(self.lens, self.w.num_kv_heads, 152, self.w.min_tiles)
        dt_assign = time.perf_counter() - t
        sample_work = float(self.work[rows].sum())
        us = (dt * self.total_work / sample_work + dt_assign) * 1e6
        desc = (f"{len(rows)} of {len(self.rows_all)} (request, query-head) rows "
                f"({sample_work / self.total_work:.1%} of the live-token work), fp64, "
                f"extrapolated by work; plus the assign oracle on the full batch")
        return us, desc

    def single_thread(self, budget_s, seed=1):
        """The same on one host thread, on a smaller sample: (us per step, rows)."""
        np = self.np
        order = np.random.default_rng(seed).permutation(self.rows_all)
        per_work_1 = self.per_work * (os.cpu_count() or 1)  # rough single-thread cost
        cum = np.cumsum(self.work[order])
        n_rows = min(int(np.searchsorted(cum, budget_s / per_work_1)) + 1, len(order))
        rows = np.sort(order[:n_rows])
        t = time.perf_counter()
        self.oracle.attention(rows=rows, num_threads=1, **self.cpu, **self.kw)
        dt = time.perf_counter() - t
        return dt * self.total_work / float(self.work[rows].sum()) * 1e6, int(n_rows)


# ------------------------------------------------------------------ main
def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="skewed")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-static", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prologue", action="store_true")
    ap.add_argument("--no-mtp", action="store_true")
    ap.add_argument("--no-router", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-table4-decode", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the compact per-workload summary at the end of the line")
    ap.add_argument("--no-table3", action="store_true",
                    help="skip the six Table-3 mixes (dynamic vs best static)")
    ap.add_argument("--prefill-shapes", default="",
                    help="comma-separated prefill/extend workloads (default: all of Table 4's)")
    ap.add_argument("--floor", type=int, default=None)
    ap.add_argument("--ctas", type=int, default=0)
    ap.add_argument("--graph", action="store_true",
                    help="replay each step from a CUDA graph instead of launching its kernels")
    ap.add_argument("--bins-per-cta", type=int, default=1,
                    help="bins planned per persistent CTA (1 = one bin per CTA)")
    return ap.parse_args()


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return [x]
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    out = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(out, t)
    return [float(o.item()) for o in out]


def config_of(w, lens, floor, world):
    """The workload's defining facts; both arms print this same dict."""
    return {"workload": w.name, "description": w.description, "batch": w.batch,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": 128,
            "page": 64, "kv_dtype": w.kv_dtype, "live_tokens": int(sum(lens)), "floor": floor,
            "l2": "GPU arm: L2 flushed before every step (256 MiB write outside the events)",
            "parallelism": f"replicas x{world}"}


def run_reference(args, world, rank):
    """Reference arm: the fp64 oracle on the host cores, each step a bounded
    sample of the same workload, extrapolated by work."""
    if rank != 0:
        return
    from load_balanced_paged_assign_gb300.workloads import WORKLOADS, make_batch
    w = WORKLOADS[args.workload]
    batch = make_batch(w, device="cpu")
    budget = max(0.02, 150.0 / (args.steps + args.warmup))
    timer = OracleTimer(batch)
    per = []
    desc = ""
    for i in range(args.warmup + args.steps):
        us, desc = timer.run(budget, seed=i)
        if i >= args.warmup:
            per.append(us)
    value = statistics.median(per)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "us/step",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": value / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, batch.seqlens.tolist(),
                            w.min_tiles if args.floor is None else args.floor, world),
        "cpu_baseline": {"value": value, "unit": "us/step", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":  # host-only: no process group, rank 0 alone works
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")),
                      int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup(args)

    import torch

    from load_balanced_paged_assign_gb300 import _build
    _build.build()
    import load_balanced_paged_assign_gb300 as hd
    from load_balanced_paged_assign_gb300.workloads import WORKLOADS, make_batch

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    capture_stream = torch.cuda.Stream(device=dev)
    sampler = ClockSampler(local)
    timed_spans = []  # host (start, end) of every timed leg, for the clock record

    def graphed(fn):
        """fn captured once into a CUDA graph (the programmatic launch edges between
        the kernels are kept); returns a replay function."""
        fn()  # first call outside capture: one-time attribute and occupancy set-up
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=capture_stream):
            fn()
        torch.cuda.synchronize()
        return g.replay

    def timed(n_steps, n_warm, run, before=None):
        """Per-step device times (us) of run(), L2 flushed before each step
        (and before() run, untimed, after the flush); no event sits between the
        kernels of a step, so programmatic launches overlap."""
        for _ in range(n_warm):
            flush.fill_(1)
            if before:
                before()
            run()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_steps)]
        t0 = time.time()
        for e0, e1 in evs:
            flush.fill_(1)
            if before:
                before()
            e0.record(stream)
            run()
            e1.record(stream)
        torch.cuda.synchronize()
        timed_spans.append((t0, time.time()))
        return [e0.elapsed_time(e1) * 1e3 for e0, e1 in evs]

    class Rig:
        """One decode workload on the device: its batch, a load-balanced
        workspace, and the step / attention / static-schedule timings."""

        def __init__(self, wl, floor=None, bins_per_cta=1, ctas=0):
            self.w = wl
            self.fp8 = wl.kv_dtype == "e4m3"
            self.batch = make_batch(wl, device=dev)
            self.B, self.Hq, self.Hkv = wl.batch, wl.num_q_heads, wl.num_kv_heads
            self.floor = wl.min_tiles if floor is None else floor
            self.resident = hd.hpc_decode_num_ctas(
                local, hd.HPC_KV_FP8_E4M3 if self.fp8 else hd.HPC_KV_BF16)
            self.ctas = ctas or wl.num_ctas or self.resident * bins_per_cta  # bins of the plan
            self.ws = hd.Workspace(self.B, self.Hq, self.Hkv, num_ctas=self.ctas, device=dev)
            self.lens = self.batch.seqlens.cpu().tolist()

        def plan(self, tm, num_splits=0):
            b = self.batch
            if num_splits:
                hd.hpc_decode_plan_static(b.seqlens, self.Hkv, b.max_pages, num_splits, tm)
            else:
                hd.hpc_decode_plan(b.seqlens, self.Hkv, b.max_pages, self.ctas, self.floor, tm)

        def attention(self, w_s):
            b = self.batch
            hd.hpc_decode_attn_combine(b.q, b.q_scale, b.k_cache, b.v_cache, b.k_scale, b.v_scale,
                                       b.block_table, b.seqlens, self.Hq, self.Hkv,
                                       self.w.sm_scale, w_s.tmap, w_s.part_o, w_s.part_lse,
                                       w_s.unit_done, w_s.out)

        def step(self, w_s=None, num_splits=0, fused=True):
            """One decode step through the public step call: the assign kernel, then
            the attention grid right behind it (fused combine unless fused=False)."""
            w_s = w_s or self.ws
            b = self.batch
            hd.hpc_decode_step(b.q, b.q_scale, b.k_cache, b.v_cache, b.k_scale, b.v_scale,
                               b.block_table, b.seqlens, self.Hq, self.Hkv, self.w.sm_scale,
                               self.ctas, self.floor, num_splits, w_s.tmap, w_s.part_o,
                               w_s.part_lse, w_s.out, unit_done=w_s.unit_done if fused else None)

        def attn_alone(self, n_steps, n_warm, w_s=None, num_splits=0):
            """The dominant kernel alone, as every layer runs it on the step's map:
            flush, rebuild the map (untimed, so it sits in L2 as in a model where all
            layers share it), then time the attention launch by itself (a
            standalone launch on a reused map waits for the kernel ahead of it)."""
            w_s = w_s or self.ws
            for _ in range(2):
                self.step(w_s, num_splits)
            return timed(n_steps, n_warm, lambda: self.attention(w_s),
                         before=lambda: self.plan(w_s.tmap, num_splits))

        def plan_facts(self, w_s=None):
            w_s = w_s or self.ws
            meta = hd.hpc_decode_read_meta(w_s.tmap)
            if meta[3] != 0:
                raise RuntimeError(f"{self.w.name}: device error flags {meta[3]}")
            counts = w_s.tmap.chunk_count[:self.B * self.Hkv].tolist()
            split_desc = sum(c for c in counts if c > 1)
            nbytes = algorithmic_bytes(self.lens, self.Hq, self.Hkv, self.w.kv_dtype, meta[2],
                                       split_desc)
            return meta, nbytes

        def static_sweep(self, n_steps, n_warm, with_attn=False):
            """The in-house static split-KV schedule over S in {1, 2, 4, 8, 16, 32}
            and the default S (smallest with B * Hkv * S >= the CTA count, capped
            at the longest request's tiles); {S: (step us, attention us or None)}."""
            max_n = max(max((L + 63) // 64 for L in self.lens), 1)
            s_default = min(max(1, math.ceil(self.ctas / (self.B * self.Hkv))), max_n)
            sweep = sorted({x for x in (1, 2, 4, 8, 16, 32, s_default) if x <= max_n})
            res = {}
            for S in sweep:
                sws = hd.Workspace(self.B, self.Hq, self.Hkv, num_splits=S, device=dev)
                tot = statistics.fmean(timed(n_steps, n_warm,
                                             lambda sws=sws, S=S: self.step(sws, num_splits=S)))
                att = (statistics.fmean(self.attn_alone(n_steps, n_warm, sws, S))
                       if with_attn else None)
                res[S] = (tot, att)
                del sws
            return res, s_default

        def free(self):
            del self.batch, self.ws

    w = WORKLOADS[args.workload]
    rig = Rig(w, args.floor, args.bins_per_cta, args.ctas)
    batch, ws, kv_dtype, fp8 = rig.batch, rig.ws, w.kv_dtype, rig.fp8
    B, Hq, Hkv, floor, ctas, resident = rig.B, rig.Hq, rig.Hkv, rig.floor, rig.ctas, rig.resident
    lens = rig.lens
    step = rig.step

    # ---- the timed region: K decode steps (assign + attention with fused combine),
    # launched directly (or replayed from a CUDA graph with --graph)
    run_step = graphed(lambda: step(ws)) if args.graph else (lambda: step(ws))
    for _ in range(args.warmup):
        flush.fill_(1)
        run_step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for e0, e1 in evs:
        flush.fill_(1)
        e0.record(stream)
        run_step()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    timed_spans.append((t0, t1))
    step_us = [e0.elapsed_time(e1) * 1e3 for e0, e1 in evs]
    meta, nbytes = rig.plan_facts()
    num_desc = meta[2]
    mean_step = statistics.fmean(step_us)
    all_steps = max_over_ranks(mean_step, world)
    value, agg_gbps = aggregate(all_steps, [nbytes["step"]] * world)
    headline_clocks = sampler.summary(t0, t1)

    attn_us_list = rig.attn_alone(args.steps, args.warmup)
    mean_attn = statistics.fmean(attn_us_list)
    peak, peak_kind = measured_peaks()
    achieved = nbytes["attn_fused"] / (mean_attn * 1e-6) / 1e9
    traffic = profiled_traffic(kernel_source_hash(), kv_dtype, w.name)

    # ---- the same step replayed from a CUDA graph (host launch cost removed;
    # each kernel's device-side launch remains), the second timing column
    graph_us = None
    if not args.graph:
        graph_us = statistics.fmean(timed(min(args.steps, 1000), args.warmup,
                                          graphed(lambda: step(ws))))

    # ---- the same step with the combine as its own kernel
    n_unf = min(args.steps, 1000)
    unf = graphed(lambda: step(ws, fused=False)) if args.graph else (lambda: step(ws, fused=False))
    unfused_us = statistics.fmean(timed(n_unf, args.warmup, unf))

    # ---- e2e: the same step through the host-buffer C entry points: the
    # step's inputs packed in one pinned host buffer (one copy in, one out),
    # and for context the separate-buffer call (one copy per input array)
    e2e = None
    if not args.no_e2e:
        kvd = hd.HPC_KV_FP8_E4M3 if fp8 else hd.HPC_KV_BF16
        total, off = hd.hpc_decode_packed_layout(B, Hq, batch.max_pages, kvd)
        h_in = torch.zeros(total, dtype=torch.uint8).pin_memory()

        def put(o, t):
            raw = t.cpu().contiguous().view(torch.uint8).reshape(-1)
            h_in[o:o + raw.numel()] = raw

        put(off[0], batch.q)
        if fp8:
            put(off[1], batch.q_scale)
        put(off[2], batch.seqlens)
        put(off[3], batch.block_table)
        d_in = torch.empty(total, dtype=torch.uint8, device=dev)
        h_out = torch.empty((B, Hq, 128), dtype=torch.bfloat16).pin_memory()

        def e2e_step():  # the output stored straight into the pinned host buffer
            hd.hpc_decode_step_host_packed(h_in, d_in, h_out, None, batch.k_cache, batch.v_cache,
                                           batch.k_scale, batch.v_scale, B, Hq, Hkv,
                                           batch.max_pages, w.sm_scale, ctas, floor, 0, ws.tmap,
                                           ws.part_o, ws.part_lse, ws.unit_done)

        h_q = batch.q.cpu().pin_memory()
        h_qs = batch.q_scale.cpu().pin_memory() if fp8 else None
        h_sl = batch.seqlens.cpu().pin_memory()
        h_bt = batch.block_table.cpu().pin_memory()
        d_q, d_sl, d_bt = (torch.empty_like(batch.q), torch.empty_like(batch.seqlens),
                           torch.empty_like(batch.block_table))
        d_qs = torch.empty_like(batch.q_scale) if fp8 else None

        def e2e_step_separate():
            hd.hpc_decode_step_host(h_q, h_qs, h_sl, h_bt, h_out, d_q, d_qs, d_sl, d_bt, ws.out,
                                    batch.k_cache, batch.v_cache, batch.k_scale, batch.v_scale,
                                    Hq, Hkv, w.sm_scale, ctas, floor, 0, ws.tmap, ws.part_o,
                                    ws.part_lse, ws.unit_done)

        n_e2e = min(args.steps, 1000)
        tot = timed(n_e2e, args.warmup, e2e_step)
        sep = timed(n_e2e, args.warmup, e2e_step_separate)
        d2h = h_out.numel() * 2
        e2e = {"value": max(max_over_ranks(statistics.fmean(tot), world)), "unit": "us/step",
               "h2d_bytes_per_step": total, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "api": "hpc_decode_step_host_packed (one pinned input buffer read in by a copy kernel through its device alias; the output stored by the attention grid into pinned host memory)",
               "gpu_launches_per_step": 3,  # copy-in, assign, attention (combine fused)
               "separate_buffers_us": statistics.fmean(sep),
               "separate_buffers_api": "hpc_decode_step_host (one copy kernel over the pinned input arrays; the output copied out by the copy engine)"}

    # ---- in-house static split-KV comparator on the same batch
    static = None
    if not args.no_static:
        results, s_default = rig.static_sweep(min(args.steps, 300), 5, with_attn=True)
        best = min(results, key=lambda x: results[x][0])
        static = {"splits_default": s_default, "us_per_step_default": results[s_default][0],
                  "best_splits": best, "us_per_step_best": results[best][0],
                  "attn_us_best": results[best][1],
                  "sweep_us_per_step": {str(k): round(v[0], 3) for k, v in results.items()},
                  "dynamic_speedup_vs_best_static": results[best][0] / mean_step,
                  "dynamic_attn_speedup_vs_best_static": results[best][1] / mean_attn}

    # ---- the fused attention prologue: this step's new tokens, then the
    # prologue followed by the per-layer attention on its outputs, then the
    # HBM-bound 8K-token prefill shape against the roofline
    prologue = None
    if not args.no_prologue:
        from load_balanced_paged_assign_gb300.workloads import (PROLOGUES, PrologueInputs,
                                                                draw_qkv, make_prologue_inputs)

        freq_tables = {}

        def prologue_call(inp, q_out, q_scale_out):
            pw_ = inp.workload
            if pw_.rope_base not in freq_tables:  # built once, as a model keeps it
                f = torch.empty(64, dtype=torch.float64, device=dev)
                hd.hpc_rope_frequencies(pw_.rope_base, f)
                freq_tables[pw_.rope_base] = f
            hd.hpc_rope_norm(inp.qkv, inp.q_norm_w, inp.k_norm_w, inp.positions, inp.token_req,
                             pw_.num_q_heads, pw_.num_kv_heads, inp.block_table, inp.k_cache,
                             inp.v_cache, inp.k_scale, inp.v_scale, q_out, q_scale_out,
                             eps=pw_.eps, rope_base=pw_.rope_base, rope_layout=pw_.rope_layout,
                             norm_first=pw_.norm_first, freq=freq_tables[pw_.rope_base])

        def outputs_for(inp):
            pw_ = inp.workload
            n = inp.num_tokens
            qdt = torch.float8_e4m3fn if pw_.kv_dtype == "e4m3" else torch.bfloat16
            q_o = torch.empty((n, pw_.num_q_heads, 128), dtype=qdt, device=dev)
            qs_o = (torch.empty((n, pw_.num_q_heads), device=dev)
                    if pw_.kv_dtype == "e4m3" else None)
            return q_o, qs_o

        n_pro = min(args.steps, 500)
        prologue = {"launches_per_call": 1}
        pw = next((p for p in PROLOGUES.values() if p.decode_of == w.name), None)
        if pw is not None:
            qkv, wq, wk = draw_qkv(B, Hq, Hkv, pw.seed, dev)
            inp = PrologueInputs(pw, qkv, wq, wk, (batch.seqlens - 1).to(torch.int32), None,
                                 batch.block_table, batch.k_cache, batch.v_cache, batch.k_scale,
                                 batch.v_scale, batch)
            q_o, qs_o = outputs_for(inp)
            dec_us = statistics.fmean(timed(n_pro, args.warmup,
                                            lambda: prologue_call(inp, q_o, qs_o)))

            def layer():  # prologue, then the attention on its query and cache rows
                prologue_call(inp, q_o, qs_o)
                hd.hpc_decode_attn_combine(q_o, qs_o, batch.k_cache, batch.v_cache,
                                           batch.k_scale, batch.v_scale, batch.block_table,
                                           batch.seqlens, Hq, Hkv, w.sm_scale, ws.tmap,
                                           ws.part_o, ws.part_lse, ws.unit_done, ws.out)

            rig.plan(ws.tmap)
            layer_us = statistics.fmean(timed(n_pro, args.warmup, layer))
            prologue["decode"] = {"workload": pw.name, "tokens": B, "us": dec_us,
                                  "bytes": prologue_bytes(B, Hq, Hkv, kv_dtype),
                                  "layer_us": layer_us,
                                  "layer": "prologue + attention with fused combine on the "
                                           "step's task map (two launches)"}
        pre = PROLOGUES["prefill_8k_fp8"]
        inp = make_prologue_inputs(pre, device=dev)
        q_o, qs_o = outputs_for(inp)
        pre_us = statistics.fmean(timed(n_pro, args.warmup, lambda: prologue_call(inp, q_o, qs_o)))
        pre_bytes = prologue_bytes(inp.num_tokens, pre.num_q_heads, pre.num_kv_heads,
                                   pre.kv_dtype)
        pre_gbs = pre_bytes / (pre_us * 1e-6) / 1e9
        prologue["prefill"] = {
            "workload": pre.name, "description": pre.description, "tokens": inp.num_tokens,
            "us": pre_us, "bytes": pre_bytes,
            "roofline": {"bound": "hbm", "achieved": pre_gbs, "peak": peak, "unit": "GB/s",
                         "frac": pre_gbs / peak, "peak_kind": peak_kind}}
        del inp, q_o, qs_o

    # ---- multi-query decode (one draft token, q_len = 2) on the same lengths:
    # one step reads the KV once for both query tokens
    mtp = None
    if not args.no_mtp and 2 * (Hq // Hkv) <= hd.binding.MAX_QUERY_ROWS:
        import dataclasses
        w2 = dataclasses.replace(w, q_len=2)
        b2 = make_batch(w2, device=dev)
        ws2 = hd.Workspace(B, Hq, Hkv, num_ctas=ctas, device=dev, q_len=2)

        def mtp_step():
            hd.hpc_decode_step_mq(b2.q, b2.q_scale, b2.k_cache, b2.v_cache, b2.k_scale,
                                  b2.v_scale, b2.block_table, b2.seqlens, Hq, Hkv, 2, w.sm_scale,
                                  ctas, floor, 0, ws2.tmap, ws2.part_o, ws2.part_lse, ws2.out,
                                  unit_done=ws2.unit_done)

        n_m = min(args.steps, 1000)
        mtp_us = statistics.fmean(timed(n_m, args.warmup, mtp_step))
        m2 = hd.hpc_decode_read_meta(ws2.tmap)
        counts2 = ws2.tmap.chunk_count[:B * Hkv].tolist()
        nb2 = algorithmic_bytes(lens, Hq, Hkv, kv_dtype, m2[2], sum(c for c in counts2 if c > 1),
                                q_len=2)
        mtp = {"q_len": 2, "us_per_step": mtp_us, "bytes": nb2["step"],
               "gbps": nb2["step"] / (mtp_us * 1e-6) / 1e9,
               "frac": nb2["step"] / (mtp_us * 1e-6) / 1e9 / peak,
               "two_decode_steps_us": 2 * mean_step,
               "speedup_vs_two_decode_steps": 2 * mean_step / mtp_us}
        del b2, ws2

    # ---- router GEMM (BF16 hi/lo split of FP32 weights, tcgen05) over the
    # token sweep at the post's shape; cuBLAS FP32 / TF32 timed beside it as
    # the post's own comparison points (context, not part of the path)
    router = None
    if not args.no_router:
        from load_balanced_paged_assign_gb300.workloads import (ROUTER_K, ROUTER_MS, ROUTER_N,
                                                                make_router_inputs)
        tf_peak, tf_kind = measured_bf16_tflops()
        rows = []
        n_r = min(args.steps, 200)
        for M in ROUTER_MS:
            x, wr = make_router_inputs(M, device=dev)
            hi = torch.empty((ROUTER_N, ROUTER_K), dtype=torch.bfloat16, device=dev)
            lo = torch.empty_like(hi)
            hd.hpc_router_split(wr, hi, lo)
            out_r = torch.empty((M, ROUTER_N), device=dev)
            nbw = hd.hpc_router_workspace_bytes(M, ROUTER_N, ROUTER_K)
            ws_r = torch.empty(max(nbw // 4, 1), device=dev) if nbw > 0 else None
            splits = nbw // (M * ROUTER_N * 4) if nbw > 0 else 1
            us = statistics.fmean(timed(n_r, args.warmup,
                                        lambda: hd.hpc_router_gemm(x, hi, lo, out_r, ws_r)))
            xf, wt = x.float(), wr.t().contiguous()
            torch.backends.cuda.matmul.allow_tf32 = False
            fp32_us = statistics.fmean(timed(n_r, args.warmup, lambda: torch.matmul(xf, wt)))
            torch.backends.cuda.matmul.allow_tf32 = True
            tf32_us = statistics.fmean(timed(n_r, args.warmup, lambda: torch.matmul(xf, wt)))
            torch.backends.cuda.matmul.allow_tf32 = False
            flops, nb = router_cost(M, ROUTER_N, ROUTER_K, splits)
            tflops, gbs = flops / (us * 1e-6) / 1e12, nb / (us * 1e-6) / 1e9
            bound = "tensor" if tflops / tf_peak > gbs / peak else "hbm"
            rows.append({"M": M, "us": us, "splits": splits, "tflops": tflops, "gbps": gbs,
                         "bound": bound,
                         "frac": tflops / tf_peak if bound == "tensor" else gbs / peak,
                         "cublas_fp32_us": fp32_us, "cublas_tf32_us": tf32_us,
                         "speedup_vs_fp32": fp32_us / us, "speedup_vs_tf32": tf32_us / us})
            del x, wr, hi, lo, out_r, ws_r, xf, wt
        router = {"K": ROUTER_K, "N": ROUTER_N, "peaks": {"bf16_tflops": tf_peak,
                                                          "hbm_gbs": peak, "kind": tf_kind},
                  "sweep": rows}

    # ---- extend / prefill attention (tcgen05) on the vLLM comparison's
    # prefill and extend shapes.  torch's scaled_dot_product_attention on
    # contiguous copies (K/V expanded to the query heads) is timed beside the
    # prefills as context: a library kernel on the same GPU, not the path.
    prefill = None
    if not args.no_prefill:
        from load_balanced_paged_assign_gb300.workloads import TABLE4_PREFILL
        tf_peak, tf_kind = measured_bf16_tflops()
        rows = []
        n_p = min(args.steps, 50)
        shapes = [x for x in args.prefill_shapes.split(",") if x] or list(TABLE4_PREFILL)
        for name in shapes:
            wp = WORKLOADS[name]
            bp = make_batch(wp, device=dev)
            Bp, qn, Hqp, Hkvp = int(bp.seqlens.numel()), wp.q_len, wp.num_q_heads, wp.num_kv_heads
            lens_p = bp.seqlens.cpu().tolist()
            outp = torch.empty((Bp, qn, Hqp, 128), dtype=torch.bfloat16, device=dev)
            pflags = torch.zeros(1, dtype=torch.int32, device=dev)

            def prefill_call():
                hd.hpc_prefill_attn(bp.q, bp.k_cache, bp.v_cache, bp.block_table, bp.seqlens,
                                    Hqp, Hkvp, qn, wp.sm_scale, outp, flags=pflags)

            us = statistics.fmean(timed(n_p, args.warmup, prefill_call))
            if int(pflags.item()) != 0:
                raise RuntimeError(f"prefill error flags {int(pflags.item())}")
            flops = prefill_flops(lens_p, qn, Hqp)
            tfl = flops / (us * 1e-6) / 1e12
            row = {"workload": name, "batch": Bp, "q_len": qn, "seqlen": lens_p[0],
                   "us": us, "flops": flops, "tflops": tfl, "frac": tfl / tf_peak}
            if all(L == qn for L in lens_p) and Bp == 1:
                try:
                    npg = (qn + 63) // 64
                    pages = bp.block_table[0, :npg].long()
                    kc = bp.k_cache[pages].reshape(npg * 64, Hkvp, 128)[:qn]
                    vc = bp.v_cache[pages].reshape(npg * 64, Hkvp, 128)[:qn]
                    G = Hqp // Hkvp
                    qs = bp.q[0].transpose(0, 1).contiguous()[None]
                    ks = kc.repeat_interleave(G, dim=1).transpose(0, 1).contiguous()[None]
                    vs = vc.repeat_interleave(G, dim=1).transpose(0, 1).contiguous()[None]
                    sdpa = torch.nn.functional.scaled_dot_product_attention
                    t_us = statistics.fmean(timed(n_p, args.warmup, lambda: sdpa(
                        qs, ks, vs, is_causal=True, scale=wp.sm_scale)))
                    row["torch_sdpa_us"] = t_us
                    row["speedup_vs_torch_sdpa"] = t_us / us
                    del qs, ks, vs, kc, vc
                except RuntimeError as exc:  # no fused kernel for this shape: leave it out
                    row["torch_sdpa_us"] = None
                    row["torch_sdpa_error"] = str(exc)[:120]
            rows.append(row)
            del bp, outp
        prefill = {"heads": "Hq=64, Hkv=8, head_dim 128, BF16 (Hy3 TP1 shape)",
                   "peak_bf16_tflops": tf_peak, "peak_kind": tf_kind,
                   "l2": "flushed before every call", "shapes": rows}
        # the fp64 oracle beside it (rank 0, one GPU): a bounded sample of one
        # shape's query rows on the host cores, scaled to the whole shape by
        # the causal (row, token) pairs it covers
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            import numpy as np

            import oracle
            name = "t4_q4k" if "t4_q4k" in shapes else shapes[-1]
            wp = WORKLOADS[name]
            bp = make_batch(wp, device="cpu")
            Hqp, qn = wp.num_q_heads, wp.q_len
            lens_p = bp.seqlens.tolist()
            n_rows = len(lens_p) * qn * Hqp
            rng = np.random.default_rng(7)
            sample = np.sort(rng.choice(n_rows, min(n_rows, 4096), replace=False))

            def visible(row):
                rq, i = row // (qn * Hqp), (row // Hqp) % qn
                return max(0, lens_p[rq] - qn + 1 + i)

            t = time.perf_counter()
            oracle.attention_mq(bp.q, bp.k_cache, bp.v_cache, bp.block_table, bp.seqlens, qn,
                                rows=sample, **bp.oracle_kwargs())
            dt = time.perf_counter() - t
            pairs_sample = sum(visible(int(x)) for x in sample)
            pairs_all = prefill_flops(lens_p, qn, Hqp) / (4 * 128)
            prefill["cpu_baseline"] = {
                "workload": name, "value": dt * pairs_all / max(pairs_sample, 1) * 1e6,
                "unit": "us", "cores": os.cpu_count(), "kind": "oracle",
                "sample": f"{len(sample)} of {n_rows} query rows, fp64, scaled by causal pairs"}
            del bp

    # ---- the decode rows of the vLLM comparison's Table 4 at the same head
    # shape: the whole step (assign + attention with the fused combine), and
    # the best static split-KV step of a small sweep, L2 flushed before each
    table4_decode = None
    if not args.no_table4_decode:
        from load_balanced_paged_assign_gb300.workloads import TABLE4_DECODE
        rows = []
        n_d = min(args.steps, 300)
        bf16_ctas = hd.hpc_decode_num_ctas(local, hd.HPC_KV_BF16)
        for name in TABLE4_DECODE:
            wd = WORKLOADS[name]
            bd = make_batch(wd, device=dev)
            Bd, Hqd, Hkvd = wd.batch, wd.num_q_heads, wd.num_kv_heads
            lens_d = bd.seqlens.cpu().tolist()

            def dstep(w_s, S=0, bd=bd, wd=wd):
                hd.hpc_decode_step(bd.q, bd.q_scale, bd.k_cache, bd.v_cache, bd.k_scale,
                                   bd.v_scale, bd.block_table, bd.seqlens, wd.num_q_heads,
                                   wd.num_kv_heads, wd.sm_scale, bf16_ctas, wd.min_tiles, S,
                                   w_s.tmap, w_s.part_o, w_s.part_lse, w_s.out,
                                   unit_done=w_s.unit_done)

            wsd = hd.Workspace(Bd, Hqd, Hkvd, num_ctas=bf16_ctas, device=dev)
            us = statistics.fmean(timed(n_d, args.warmup, lambda: dstep(wsd)))
            md = hd.hpc_decode_read_meta(wsd.tmap)
            if md[3] != 0:
                raise RuntimeError(f"device error flags {md[3]}")
            cnt = wsd.tmap.chunk_count[:Bd * Hkvd].tolist()
            nb_d = algorithmic_bytes(lens_d, Hqd, Hkvd, "bf16", md[2], sum(c for c in cnt if c > 1))
            st = {}
            for S in (1, 2, 4, 8, 16):
                sw = hd.Workspace(Bd, Hqd, Hkvd, num_splits=S, device=dev)
                st[S] = statistics.fmean(timed(min(n_d, 100), 5, lambda sw=sw, S=S: dstep(sw, S)))
            best = min(st, key=st.get)
            rows.append({"workload": name, "batch": Bd, "seqlen": lens_d[0], "us_per_step": us,
                         "gbps": nb_d["step"] / (us * 1e-6) / 1e9,
                         "frac": nb_d["step"] / (us * 1e-6) / 1e9 / peak,
                         "best_static_splits": best, "best_static_us": st[best],
                         "dynamic_speedup_vs_best_static": st[best] / us})
            del bd, wsd
        table4_decode = {"heads": "Hq=64, Hkv=8, head_dim 128, BF16", "shapes": rows}

    # ---- every decode workload and the six Table-3 mixes, each in the
    # headline's launch configuration: step, attention alone against the copy
    # peak, and the best static split-KV step (compact, at the end of the line)
    def decode_summary(r, step_mean=None, attn_mean=None, n=None):
        n = n or min(max(args.steps, 200), 300)  # at least 200 timed steps after 20 warm-ups
        if step_mean is None:
            step_mean = statistics.fmean(timed(n, 20, r.step))
        if attn_mean is None:
            attn_mean = statistics.fmean(r.attn_alone(n, 20))
        _, nb = r.plan_facts()
        res, _ = r.static_sweep(n, 20)
        S = min(res, key=lambda x: res[x][0])
        return {"step_us": round(step_mean, 2), "attn_us": round(attn_mean, 2),
                "attn_bytes": nb["attn_fused"],
                "frac": round(nb["attn_fused"] / (attn_mean * 1e-6) / 1e9 / peak, 4),
                "static_S": S, "static_us": round(res[S][0], 2),
                "x_static": round(res[S][0] / step_mean, 3)}

    per_config = None
    if not args.no_per_config:
        per_config = {}
        for name in ("tiny", "hy3_tp8", "skewed", "uniform", "fp8"):
            if name == w.name and args.bins_per_cta == 1 and not args.ctas and args.floor is None:
                per_config[name] = decode_summary(rig, mean_step, mean_attn)
                continue
            r = Rig(WORKLOADS[name])
            per_config[name] = decode_summary(r)
            r.free()
            del r
    table3 = None
    if not args.no_table3:
        from load_balanced_paged_assign_gb300.workloads import TABLE3
        table3 = {}
        for name in TABLE3:
            r = Rig(WORKLOADS[name])
            d = decode_summary(r)
            table3[name[3:]] = {k: d[k] for k in ("step_us", "frac", "static_S", "static_us",
                                                  "x_static")}
            r.free()
            del r

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        timer = OracleTimer(batch)
        us, desc = timer.run(budget_s=12.0)
        us1, rows1 = timer.single_thread(budget_s=3.0)
        cpu_baseline = {"value": us, "unit": "us/step", "cores": os.cpu_count(),
                        "kind": "oracle", "sample": desc,
                        "single_thread_us": us1,
                        "single_thread_sample": f"{rows1} rows on 1 thread, extrapolated by work"}

    sampler.stop()
    clocks = sampler.summary_over(timed_spans)
    clocks["span"] = "every timed leg of this run"
    clocks["headline_samples"] = headline_clocks["samples"]

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "us/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if fp8 else "bf16", "data": "synthetic",
        "config": config_of(w, lens, floor, world),
        "plan": {"persistent_ctas": min(ctas, resident), "bins": ctas, "num_desc": num_desc,
                 "budget": meta[1], "total_tiles": meta[0]},
        "gbps": agg_gbps, "pct_of_peak": agg_gbps / (peak * world),
        "attn_us": mean_attn, "unfused_us_per_step": unfused_us,
        "median_us_per_step": statistics.median(step_us),
        "launch": "cuda graph replay per step" if args.graph else "direct launches",
        "graph_us_per_step": graph_us, "bytes": nbytes,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "attn_kernel, fused combine (per-layer launch)",
                     "peak_kind": peak_kind,
                     "pct_of_8tbs_nominal": achieved / 8000.0},
        "e2e": e2e,
        "cpu_baseline": cpu_baseline,
        "static": static,
        "rope_norm": prologue,
        "mtp": mtp,
        "router_gemm": router,
        "prefill": prefill,
        "table4_decode": table4_decode,
        "clocks": clocks,
        "gpu_launches": 2 * args.steps,
        "table3": table3,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
