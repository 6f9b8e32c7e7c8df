"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare it with the oracle."""

from __future__ import annotations

import numpy as np
import torch

import load_balanced_paged_assign_gb300 as hd
import oracle
from load_balanced_paged_assign_gb300.workloads import Batch

# Tolerances on |gpu - oracle| over the compared outputs: BF16 KV max 1e-2 and
# mean 1e-3; FP8 KV max 2e-2 (mean 2e-3), the oracle running on the
# dequantised FP8 values.
TOL = {"bf16": (1e-2, 1e-3), "e4m3": (2e-2, 2e-3)}


def device_ctas(kv_dtype: str) -> int:
    return hd.hpc_decode_num_ctas(torch.cuda.current_device(),
                                  hd.HPC_KV_FP8_E4M3 if kv_dtype == "e4m3" else hd.HPC_KV_BF16)


def run_step(batch: Batch, num_ctas: int | None = None, floor: int | None = None,
             num_splits: int = 0, fused: bool = True):
    """One plan + attention + combine through the C ABI; returns (out, workspace).

    fused: the combine runs inside the attention grid (hpc_decode_attn_combine);
    otherwise hpc_decode_attn is followed by the combine kernel."""
    w = batch.workload
    if num_ctas is None:
        num_ctas = w.num_ctas or device_ctas(w.kv_dtype)
    floor = w.min_tiles if floor is None else floor
    B = int(batch.seqlens.numel())
    ws = hd.Workspace(B, w.num_q_heads, w.num_kv_heads, num_ctas=num_ctas, num_splits=num_splits,
                      device=batch.q.device)
    ws.out.fill_(float("nan"))  # anything the kernels fail to write shows up
    hd.hpc_decode_step(batch.q, batch.q_scale, batch.k_cache, batch.v_cache, batch.k_scale,
                       batch.v_scale, batch.block_table, batch.seqlens, w.num_q_heads,
                       w.num_kv_heads, w.sm_scale, num_ctas, floor, num_splits, ws.tmap,
                       ws.part_o, ws.part_lse, ws.out, unit_done=ws.unit_done if fused else None)
    torch.cuda.synchronize()
    if fused:  # every launch must leave the chunk counters at zero
        assert int(torch.count_nonzero(ws.unit_done)) == 0
    return ws.out[:B], ws


def oracle_out(batch: Batch, rows=None):
    return oracle.attention(batch.q, batch.k_cache, batch.v_cache, batch.block_table,
                            batch.seqlens, rows=rows, **batch.oracle_kwargs())


def assert_close(got: torch.Tensor, ref: np.ndarray, kv_dtype: str, rows=None):
    g = got.float().cpu().numpy()
    if rows is not None:
        g = g.reshape(-1, g.shape[-1])[np.asarray(rows)]
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - ref)
    tol_max, tol_mean = TOL[kv_dtype]
    assert err.max() <= tol_max, f"max |err| {err.max():.3e} > {tol_max}"
    assert err.mean() <= tol_mean, f"mean |err| {err.mean():.3e} > {tol_mean}"
    return float(err.max()), float(err.mean())


def assert_map_matches(ws, seqlens, Hkv, num_ctas, floor):
    got = ws.tmap.to_host()
    ref = oracle.assign_closed_form(list(seqlens), Hkv, num_ctas, floor)
    assert got["flags"] == 0
    assert got["total_tiles"] == ref.total_tiles
    assert got["budget"] == ref.budget
    assert got["num_desc"] == ref.num_desc
    assert got["desc"] == ref.desc
    assert got["bin_ptr"] == ref.bin_ptr
    assert got["chunk_count"] == ref.chunk_count
    assert got["chunk_off"] == ref.chunk_off
