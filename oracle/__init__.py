"""CPU oracle for load-balanced paged GQA decode attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library and never imports it: the attention reference is plain fp64
C (`oracle.c`, OpenMP over query rows) and the task-map reference is plain
Python (`assign.py`).

Arrays cross into C as numpy buffers of the storage words: bf16 tensors as
uint16 bit patterns, FP8-E4M3 tensors as uint8 codes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .assign import (TaskMap, assign_closed_form, assign_simulate, budget_of, static_plan,
                     tiles_of)

__all__ = [
    "TaskMap", "assign_closed_form", "assign_simulate", "budget_of", "static_plan", "tiles_of",
    "build", "bf16_to_double", "e4m3_to_double", "attention", "partial", "combine",
    "split_attention", "attention_mq", "BF16", "E4M3",
]

BF16 = 0
E4M3 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, OpenMP)."""
    stale = not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", _SRC, "-o", tmp,
               "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    dp = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_bf16_to_double.restype = f64
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_e4m3_to_double.restype = f64
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    common = [dp, i32, dp, dp, dp, i32, f64, f64, dp, i32, dp, i32, i32, i32, i32, i32, f64]
    lib.oracle_attention.restype = i32
    lib.oracle_attention.argtypes = common + [dp, i64, dp, i32]
    lib.oracle_partial.restype = i32
    lib.oracle_partial.argtypes = common + [i32, i32, i32, i32, dp, dp]
    lib.oracle_attention_mq.restype = i32
    lib.oracle_attention_mq.argtypes = common + [i32, dp, i64, dp, i32]
    lib.oracle_combine.restype = None
    lib.oracle_combine.argtypes = [dp, dp, i32, i32, dp]
    _lib = lib
    return lib


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def e4m3_to_double(code: int) -> float:
    return _load().oracle_e4m3_to_double(int(code))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _words(x, dtype_code):
    """Storage words of a tensor/array as a contiguous numpy array."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: reinterpret the raw storage
        import torch
        x = x.detach().cpu().contiguous()
        x = x.view(torch.uint8 if dtype_code == E4M3 else torch.int16).numpy()
    want = np.uint8 if dtype_code == E4M3 else np.uint16
    return np.ascontiguousarray(x).view(want)


def _i32(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _f32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


class _Problem:
    """Marshalled arguments shared by the attention entry points."""

    def __init__(self, q, k_cache, v_cache, block_table, seqlens, *, num_q_heads, num_kv_heads,
                 sm_scale, q_dtype=BF16, kv_dtype=BF16, q_scale=None, k_scale=1.0, v_scale=1.0,
                 head_dim=128, page_size=64):
        self.q = _words(q, q_dtype)
        self.k = _words(k_cache, kv_dtype)
        self.v = _words(v_cache, kv_dtype)
        self.bt = _i32(block_table)
        self.sl = _i32(seqlens)
        self.qs = _f32(q_scale)
        self.B = int(self.sl.shape[0])
        self.max_pages = int(self.bt.shape[1]) if self.bt.ndim == 2 else int(self.bt.size // max(self.B, 1))
        self.Hq, self.Hkv, self.D, self.page = num_q_heads, num_kv_heads, head_dim, page_size
        self.q_dtype, self.kv_dtype = q_dtype, kv_dtype
        self.k_scale, self.v_scale, self.sm_scale = float(k_scale), float(v_scale), float(sm_scale)
        if q_dtype == E4M3 and self.qs is None:
            raise ValueError("FP8 queries need q_scale")

    def head(self):
        return [_ptr(self.q), self.q_dtype, _ptr(self.qs), _ptr(self.k), _ptr(self.v),
                self.kv_dtype, self.k_scale, self.v_scale, _ptr(self.bt), self.max_pages,
                _ptr(self.sl), self.B, self.Hq, self.Hkv, self.D, self.page, self.sm_scale]


def attention(q, k_cache, v_cache, block_table, seqlens, *, rows=None, num_threads=0, **kw):
    """Unsplit fp64 decode attention.

    Returns float64 [B, Hq, D], or [len(rows), D] when `rows` (flat indices
    r * Hq + hq) is given.  Keyword arguments: num_q_heads, num_kv_heads,
    sm_scale, q_dtype, kv_dtype, q_scale, k_scale, v_scale.
    """
    p = _Problem(q, k_cache, v_cache, block_table, seqlens, **kw)
    if rows is None:
        out = np.zeros((p.B, p.Hq, p.D), dtype=np.float64)
        rows_arr, n = None, p.B * p.Hq
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = int(rows_arr.size)
        out = np.zeros((n, p.D), dtype=np.float64)
    rc = _load().oracle_attention(*p.head(), _ptr(rows_arr), n, _ptr(out), int(num_threads))
    if rc != 0:
        raise MemoryError("oracle_attention: scratch allocation failed")
    return out


def attention_mq(q, k_cache, v_cache, block_table, seqlens, q_len, *, rows=None, num_threads=0,
                 **kw):
    """Multi-query decode attention: q [B, q_len, Hq, D] (q_scale [B, q_len, Hq]
    for FP8), query token i of request r sees live tokens j < L_r - q_len + 1 + i.

    Returns float64 [B, q_len, Hq, D], or [len(rows), D] for flat rows
    (r * q_len + i) * Hq + hq."""
    q_len = int(q_len)
    qs = kw.get("q_scale")
    B = int(_i32(seqlens).shape[0])
    Hq = kw["num_q_heads"]
    # the query rows are handed over as B * q_len "requests" of Hq heads
    q2 = q.reshape(B * q_len, Hq, -1) if hasattr(q, "reshape") else q
    kw2 = dict(kw)
    if qs is not None:
        kw2["q_scale"] = qs.reshape(B * q_len, Hq)
    p = _Problem(q2, k_cache, v_cache, block_table, seqlens, **kw2)
    p.B = B
    if rows is None:
        out = np.zeros((B, q_len, p.Hq, p.D), dtype=np.float64)
        rows_arr, n = None, B * q_len * p.Hq
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = int(rows_arr.size)
        out = np.zeros((n, p.D), dtype=np.float64)
    rc = _load().oracle_attention_mq(*p.head(), q_len, _ptr(rows_arr), n, _ptr(out),
                                     int(num_threads))
    if rc != 0:
        raise MemoryError("oracle_attention_mq: scratch allocation failed")
    return out


def partial(q, k_cache, v_cache, block_table, seqlens, r, hq, j0, j1, **kw):
    """Normalised partial output and natural-log LSE of (r, hq) over tokens [j0, j1)."""
    p = _Problem(q, k_cache, v_cache, block_table, seqlens, **kw)
    o = np.zeros(p.D, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    rc = _load().oracle_partial(*p.head(), int(r), int(hq), int(j0), int(j1), _ptr(o), _ptr(lse))
    if rc != 0:
        raise MemoryError("oracle_partial: scratch allocation failed")
    return o, float(lse[0])


def combine(parts, lses):
    """Merge normalised partials [n, D] with their LSEs [n] under the global softmax."""
    parts = np.ascontiguousarray(parts, dtype=np.float64)
    lses = np.ascontiguousarray(lses, dtype=np.float64)
    out = np.zeros(parts.shape[1], dtype=np.float64)
    _load().oracle_combine(_ptr(parts), _ptr(lses), int(parts.shape[0]), int(parts.shape[1]),
                           _ptr(out))
    return out


def split_attention(q, k_cache, v_cache, block_table, seqlens, task_map: TaskMap, **kw):
    """Attention evaluated the split way: one partial per descriptor, merged per unit.

    Follows the persistent-kernel-plus-combine description (vLLM post,
    "Compute and combine"): descriptor (h, r, tb, te) yields, for each query
    head of KV head h, the partial over tokens [64 tb, min(64 te, L_r)); the
    unit's partials are then merged.  Returns float64 [B, Hq, D].
    """
    Hq, Hkv = kw["num_q_heads"], kw["num_kv_heads"]
    G = Hq // Hkv
    sl = _i32(seqlens)
    B = int(sl.shape[0])
    D = kw.get("head_dim", 128)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for u in range(Hkv * B):
        h, r = divmod(u, B)
        first, count = task_map.chunk_off[u], task_map.chunk_count[u]
        for g in range(G):
            hq = h * G + g
            parts, lses = [], []
            for i in range(first, first + count):
                dh, dr, tb, te = task_map.desc[i]
                assert (dh, dr) == (h, r)
                j0, j1 = tb * 64, min(te * 64, int(sl[r]))
                o, lse = partial(q, k_cache, v_cache, block_table, seqlens, r, hq, j0, j1, **kw)
                parts.append(o)
                lses.append(lse)
            if parts:
                out[r, hq] = combine(np.stack(parts), np.array(lses))
    return out
