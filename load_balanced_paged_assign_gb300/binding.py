"""Python binding of the C ABI in include/hpc_decode.h (ctypes, argument marshalling only).

Every function here has the name of the C entry point it forwards to and does
nothing but turn torch tensors into pointers and sizes, call the library and
raise on a non-zero status.  All compute happens in libhpcdecode.so; there is
no fallback path: if the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import _build

HPC_OK, HPC_ERR_ARG, HPC_ERR_UNSUPPORTED, HPC_ERR_WORKSPACE, HPC_ERR_CUDA = 0, -1, -2, -3, -4
HPC_KV_BF16, HPC_KV_FP8_E4M3 = 0, 1
HPC_FLAG_BAD_SEQLEN, HPC_FLAG_DESC_OVERFLOW, HPC_FLAG_BAD_PAGE, HPC_FLAG_TIMEOUT = 1, 2, 4, 8
HEAD_DIM, PAGE_SIZE, MAX_GROUP, MAX_QUERY_ROWS = 128, 64, 16, 16
HPC_ROPE_HALVES, HPC_ROPE_INTERLEAVED = 0, 1

# Every symbol the header declares; the CPU tests check the library exports them all.
EXPORTS = (
    "hpc_decode_version", "hpc_status_string", "hpc_decode_num_ctas", "hpc_decode_desc_capacity",
    "hpc_decode_static_capacity", "hpc_decode_plan", "hpc_decode_plan_static", "hpc_decode_attn",
    "hpc_decode_attn_combine", "hpc_decode_combine", "hpc_decode_step", "hpc_decode_step_host", "hpc_decode_read_meta",
    "hpc_decode_step_noalloc", "hpc_rope_norm", "hpc_rope_frequencies", "hpc_decode_attn_mq",
    "hpc_decode_attn_combine_mq", "hpc_decode_combine_mq", "hpc_decode_step_mq",
    "hpc_selftest_wait_timeout", "hpc_router_split", "hpc_router_workspace_bytes", "hpc_router_plan",
    "hpc_router_gemm", "hpc_prefill_attn",
    "hpc_decode_packed_layout", "hpc_decode_step_host_packed",
)


class HpcError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


class hpc_task_map(ctypes.Structure):
    _fields_ = [
        ("desc", ctypes.c_void_p), ("bin_ptr", ctypes.c_void_p),
        ("chunk_count", ctypes.c_void_p), ("chunk_off", ctypes.c_void_p),
        ("meta", ctypes.c_void_p),
        ("cap_desc", ctypes.c_int32), ("cap_bins", ctypes.c_int32), ("cap_units", ctypes.c_int32),
        ("B", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
        ("persistent", ctypes.c_int32), ("min_tiles", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
    ]


class hpc_rope_norm_params(ctypes.Structure):
    _fields_ = [("eps", ctypes.c_float), ("rope_base", ctypes.c_float),
                ("rope_layout", ctypes.c_int32), ("norm_first", ctypes.c_int32),
                ("freq", ctypes.c_void_p)]


_LIB = None


def library_path() -> str:
    """The in-tree library, or the file named by HPC_DECODE_LIB (another build
    of the same sources, e.g. with a different pipeline shape)."""
    return os.environ.get("HPC_DECODE_LIB") or _build.LIB_PATH


def lib():
    """The loaded libhpcdecode.so; raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    tm = ctypes.POINTER(hpc_task_map)
    sig = {
        "hpc_decode_version": (ctypes.c_char_p, []),
        "hpc_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "hpc_decode_num_ctas": (i32, [i32, ctypes.c_int]),
        "hpc_decode_desc_capacity": (i64, [i32, i32, i32]),
        "hpc_decode_static_capacity": (i64, [i32, i32, i32]),
        "hpc_decode_plan": (ctypes.c_int, [vp, i32, i32, i32, i32, i32, tm, vp]),
        "hpc_decode_plan_static": (ctypes.c_int, [vp, i32, i32, i32, i32, tm, vp]),
        "hpc_decode_attn": (ctypes.c_int, [vp, vp, vp, vp, i32, f32, f32, ctypes.c_int, vp, i32,
                                           vp, i32, i32, i32, i32, f32, tm, vp, vp, vp]),
        "hpc_decode_attn_combine": (ctypes.c_int, [vp, vp, vp, vp, i32, f32, f32, ctypes.c_int,
                                                   vp, i32, vp, i32, i32, i32, i32, f32, tm, vp,
                                                   vp, vp, vp, vp]),
        "hpc_decode_combine": (ctypes.c_int, [vp, vp, tm, i32, i32, i32, i32, vp, vp]),
        "hpc_decode_step": (ctypes.c_int, [vp, vp, vp, vp, i32, f32, f32, ctypes.c_int, vp, i32,
                                           vp, i32, i32, i32, i32, f32, i32, i32, i32, tm, vp,
                                           vp, vp, vp, vp]),
        "hpc_decode_step_host": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                i32, f32, f32, ctypes.c_int, i32, i32, i32, i32,
                                                i32, f32, i32, i32, i32, tm, vp, vp, vp, vp]),
        "hpc_decode_read_meta": (ctypes.c_int, [tm, ctypes.POINTER(ctypes.c_int32), vp]),
        "hpc_decode_step_noalloc": (ctypes.c_int, [vp, vp, vp, vp, i32, f32, f32, ctypes.c_int,
                                                   vp, i32, vp, i32, i32, i32, i32, f32, i32, i32,
                                                   vp, vp, vp]),
        "hpc_rope_frequencies": (ctypes.c_int, [f32, vp, vp]),
        "hpc_router_split": (ctypes.c_int, [vp, i32, i32, vp, vp, vp]),
        "hpc_router_workspace_bytes": (i64, [i32, i32, i32]),
        "hpc_router_plan": (ctypes.c_int, [i32, i32, i32, vp]),
        "hpc_selftest_wait_timeout": (ctypes.c_int, [vp, i32, vp]),
        "hpc_router_gemm": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, vp, vp, i64, vp, vp]),
        "hpc_prefill_attn": (ctypes.c_int, [vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                            i32, f32, vp, vp, vp]),
        "hpc_decode_packed_layout": (i64, [i32, i32, i32, ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_int64)]),
        "hpc_decode_step_host_packed": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, i32, f32, f32,
                                                       ctypes.c_int, i32, i32, i32, i32, i32, f32,
                                                       i32, i32, i32, tm, vp, vp, vp, vp]),
        "hpc_decode_attn_mq": (ctypes.c_int, [vp, vp, vp, vp, i32, f32, f32, ctypes.c_int, vp,
                                              i32, vp, i32, i32, i32, i32, i32, f32, tm, vp, vp,
                                              vp]),
        "hpc_decode_attn_combine_mq": (ctypes.c_int, [vp, vp, vp, vp, i32, f32, f32, ctypes.c_int,
                                                      vp, i32, vp, i32, i32, i32, i32, i32, f32,
                                                      tm, vp, vp, vp, vp, vp]),
        "hpc_decode_combine_mq": (ctypes.c_int, [vp, vp, tm, i32, i32, i32, i32, i32, vp, vp]),
        "hpc_decode_step_mq": (ctypes.c_int, [vp, vp, vp, vp, i32, f32, f32, ctypes.c_int, vp,
                                              i32, vp, i32, i32, i32, i32, i32, f32, i32, i32,
                                              i32, tm, vp, vp, vp, vp, vp]),
        "hpc_rope_norm": (ctypes.c_int, [vp, i64, vp, vp, vp, vp, i32, i32, i32, i32, vp, i32,
                                         i32, vp, vp, i32, ctypes.c_int, f32, f32, vp, vp, vp,
                                         ctypes.POINTER(hpc_rope_norm_params), vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    _LIB = L
    return L


def status_string(status: int) -> str:
    try:
        return lib().hpc_status_string(int(status)).decode()
    except RuntimeError:
        return "unknown"


def _check(fn: str, status: int):
    if status != HPC_OK:
        raise HpcError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def kv_dtype_of(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return HPC_KV_BF16
    if t.dtype == torch.float8_e4m3fn:
        return HPC_KV_FP8_E4M3
    raise TypeError(f"unsupported KV cache dtype {t.dtype}")


class TaskMap:
    """Caller-owned device buffers of one task map and the C struct describing them."""

    def __init__(self, B: int, Hkv: int, cap_desc: int, cap_bins: int, device="cuda"):
        dev = torch.device(device)
        self.desc = torch.zeros((max(cap_desc, 1), 4), dtype=torch.int32, device=dev)
        self.bin_ptr = torch.zeros(max(cap_bins, 1), dtype=torch.int32, device=dev)
        units = max(B * Hkv, 1)
        self.chunk_count = torch.zeros(units, dtype=torch.int32, device=dev)
        self.chunk_off = torch.zeros(units, dtype=torch.int32, device=dev)
        self.meta = torch.zeros(8, dtype=torch.int32, device=dev)
        self.c = hpc_task_map(_ptr(self.desc), _ptr(self.bin_ptr), _ptr(self.chunk_count),
                              _ptr(self.chunk_off), _ptr(self.meta), cap_desc, cap_bins, units, 0,
                              0, 0, 0, 0, 0)

    @classmethod
    def dynamic(cls, B: int, Hkv: int, num_ctas: int, device="cuda"):
        return cls(B, Hkv, int(lib().hpc_decode_desc_capacity(B, Hkv, num_ctas)), num_ctas + 1,
                   device)

    @classmethod
    def static(cls, B: int, Hkv: int, num_splits: int, device="cuda"):
        n = int(lib().hpc_decode_static_capacity(B, Hkv, num_splits))
        return cls(B, Hkv, n, n + 1, device)

    @property
    def cap_desc(self) -> int:
        return int(self.c.cap_desc)

    @property
    def num_ctas(self) -> int:
        return int(self.c.num_ctas)

    def to_host(self) -> dict:
        """The map as host lists (synchronises the current stream)."""
        meta = self.meta.tolist()
        n = int(meta[2])
        B, Hkv = int(self.c.B), int(self.c.Hkv)
        return dict(total_tiles=meta[0], budget=meta[1], num_desc=n, flags=meta[3],
                    desc=[tuple(d) for d in self.desc[:n].tolist()],
                    bin_ptr=self.bin_ptr[:self.num_ctas + 1].tolist(),
                    chunk_count=self.chunk_count[:B * Hkv].tolist(),
                    chunk_off=self.chunk_off[:B * Hkv].tolist())


def hpc_decode_version() -> str:
    return lib().hpc_decode_version().decode()


def hpc_decode_num_ctas(device: int = 0, kv_dtype: int = HPC_KV_BF16) -> int:
    n = int(lib().hpc_decode_num_ctas(int(device), int(kv_dtype)))
    if n < 0:
        raise HpcError("hpc_decode_num_ctas", n)
    return n


def hpc_decode_desc_capacity(B: int, Hkv: int, num_ctas: int) -> int:
    return int(lib().hpc_decode_desc_capacity(B, Hkv, num_ctas))


def hpc_decode_static_capacity(B: int, Hkv: int, num_splits: int) -> int:
    return int(lib().hpc_decode_static_capacity(B, Hkv, num_splits))


def hpc_decode_plan(seqlens, Hkv, max_pages_per_req, num_ctas, min_tiles_per_cta, tmap: TaskMap,
                    stream=None):
    B = int(seqlens.numel())
    _check("hpc_decode_plan", lib().hpc_decode_plan(
        _ptr(seqlens), B, int(Hkv), int(max_pages_per_req), int(num_ctas),
        int(min_tiles_per_cta), ctypes.byref(tmap.c), _stream(stream)))


def hpc_decode_plan_static(seqlens, Hkv, max_pages_per_req, num_splits, tmap: TaskMap,
                           stream=None):
    B = int(seqlens.numel())
    _check("hpc_decode_plan_static", lib().hpc_decode_plan_static(
        _ptr(seqlens), B, int(Hkv), int(max_pages_per_req), int(num_splits),
        ctypes.byref(tmap.c), _stream(stream)))


def hpc_decode_attn(q, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, seqlens, Hq, Hkv,
                    sm_scale, tmap: TaskMap, part_o, part_lse, stream=None):
    _check("hpc_decode_attn", lib().hpc_decode_attn(
        _ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]),
        float(k_scale), float(v_scale), kv_dtype_of(k_cache), _ptr(block_table),
        int(block_table.shape[1]), _ptr(seqlens), int(seqlens.numel()), int(Hq), int(Hkv),
        HEAD_DIM, float(sm_scale), ctypes.byref(tmap.c), _ptr(part_o), _ptr(part_lse),
        _stream(stream)))


def hpc_decode_attn_combine(q, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, seqlens,
                            Hq, Hkv, sm_scale, tmap: TaskMap, part_o, part_lse, unit_done, out,
                            stream=None):
    _check("hpc_decode_attn_combine", lib().hpc_decode_attn_combine(
        _ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]),
        float(k_scale), float(v_scale), kv_dtype_of(k_cache), _ptr(block_table),
        int(block_table.shape[1]), _ptr(seqlens), int(seqlens.numel()), int(Hq), int(Hkv),
        HEAD_DIM, float(sm_scale), ctypes.byref(tmap.c), _ptr(part_o), _ptr(part_lse),
        _ptr(unit_done), _ptr(out), _stream(stream)))


def hpc_decode_combine(part_o, part_lse, tmap: TaskMap, B, Hq, Hkv, out, stream=None):
    _check("hpc_decode_combine", lib().hpc_decode_combine(
        _ptr(part_o), _ptr(part_lse), ctypes.byref(tmap.c), int(B), int(Hq), int(Hkv), HEAD_DIM,
        _ptr(out), _stream(stream)))


def hpc_decode_step(q, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, seqlens, Hq,
                    Hkv, sm_scale, num_ctas, min_tiles_per_cta, num_splits, tmap: TaskMap, part_o,
                    part_lse, out, unit_done=None, stream=None):
    """unit_done given: fused attention + combine; None: separate combine kernel."""
    _check("hpc_decode_step", lib().hpc_decode_step(
        _ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]),
        float(k_scale), float(v_scale), kv_dtype_of(k_cache), _ptr(block_table),
        int(block_table.shape[1]), _ptr(seqlens), int(seqlens.numel()), int(Hq), int(Hkv),
        HEAD_DIM, float(sm_scale), int(num_ctas), int(min_tiles_per_cta), int(num_splits),
        ctypes.byref(tmap.c), _ptr(part_o), _ptr(part_lse), _ptr(unit_done), _ptr(out),
        _stream(stream)))


def hpc_decode_attn_mq(q, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, seqlens, Hq,
                       Hkv, q_len, sm_scale, tmap: TaskMap, part_o, part_lse, stream=None):
    """Multi-query attention: q [B, q_len, Hq, 128]; partials [cap, q_len * G, ...]."""
    _check("hpc_decode_attn_mq", lib().hpc_decode_attn_mq(
        _ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]),
        float(k_scale), float(v_scale), kv_dtype_of(k_cache), _ptr(block_table),
        int(block_table.shape[1]), _ptr(seqlens), int(seqlens.numel()), int(Hq), int(Hkv),
        HEAD_DIM, int(q_len), float(sm_scale), ctypes.byref(tmap.c), _ptr(part_o),
        _ptr(part_lse), _stream(stream)))


def hpc_decode_attn_combine_mq(q, q_scale, k_cache, v_cache, k_scale, v_scale, block_table,
                               seqlens, Hq, Hkv, q_len, sm_scale, tmap: TaskMap, part_o, part_lse,
                               unit_done, out, stream=None):
    _check("hpc_decode_attn_combine_mq", lib().hpc_decode_attn_combine_mq(
        _ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]),
        float(k_scale), float(v_scale), kv_dtype_of(k_cache), _ptr(block_table),
        int(block_table.shape[1]), _ptr(seqlens), int(seqlens.numel()), int(Hq), int(Hkv),
        HEAD_DIM, int(q_len), float(sm_scale), ctypes.byref(tmap.c), _ptr(part_o),
        _ptr(part_lse), _ptr(unit_done), _ptr(out), _stream(stream)))


def hpc_decode_combine_mq(part_o, part_lse, tmap: TaskMap, B, Hq, Hkv, q_len, out, stream=None):
    _check("hpc_decode_combine_mq", lib().hpc_decode_combine_mq(
        _ptr(part_o), _ptr(part_lse), ctypes.byref(tmap.c), int(B), int(Hq), int(Hkv), HEAD_DIM,
        int(q_len), _ptr(out), _stream(stream)))


def hpc_decode_step_mq(q, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, seqlens, Hq,
                       Hkv, q_len, sm_scale, num_ctas, min_tiles_per_cta, num_splits,
                       tmap: TaskMap, part_o, part_lse, out, unit_done=None, stream=None):
    """hpc_decode_step with q_len query tokens per request (causal among them)."""
    _check("hpc_decode_step_mq", lib().hpc_decode_step_mq(
        _ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]),
        float(k_scale), float(v_scale), kv_dtype_of(k_cache), _ptr(block_table),
        int(block_table.shape[1]), _ptr(seqlens), int(seqlens.numel()), int(Hq), int(Hkv),
        HEAD_DIM, int(q_len), float(sm_scale), int(num_ctas), int(min_tiles_per_cta),
        int(num_splits), ctypes.byref(tmap.c), _ptr(part_o), _ptr(part_lse), _ptr(unit_done),
        _ptr(out), _stream(stream)))


def hpc_router_split(w, w_hi, w_lo, stream=None):
    """Split fp32 router weights [N, K] into BF16 W_high / W_low [N, K]."""
    N, K = w.shape
    _check("hpc_router_split", lib().hpc_router_split(_ptr(w), int(N), int(K), _ptr(w_hi),
                                                        _ptr(w_lo), _stream(stream)))


def hpc_router_workspace_bytes(M, N, K) -> int:
    return int(lib().hpc_router_workspace_bytes(int(M), int(N), int(K)))


def hpc_selftest_wait_timeout(flags, limit_us, stream=None):
    """One CTA waits on a barrier nothing completes for limit_us, then raises
    HPC_FLAG_TIMEOUT in flags (device int32) and returns."""
    _check("hpc_selftest_wait_timeout",
           lib().hpc_selftest_wait_timeout(_ptr(flags), int(limit_us), _stream(stream)))


def hpc_router_plan(M, N, K) -> dict:
    """The launch hpc_router_gemm makes for this shape on the current device."""
    plan = (ctypes.c_int32 * 4)()
    _check("hpc_router_plan", lib().hpc_router_plan(int(M), int(N), int(K), plan))
    return {"tensor_cores": bool(plan[0]), "bn": int(plan[1]), "splits": int(plan[2]),
            "ctas": int(plan[3])}


def hpc_router_gemm(x, w_hi, w_lo, out, workspace=None, flags=None, stream=None):
    """Router scores out [M, N] fp32 = X W_high^T + (X W_low^T) / 256."""
    M, K = x.shape
    N = w_hi.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("hpc_router_gemm", lib().hpc_router_gemm(
        _ptr(x), _ptr(w_hi), _ptr(w_lo), int(M), int(N), int(K), _ptr(out), _ptr(workspace),
        int(ws_bytes), _ptr(flags), _stream(stream)))


def hpc_prefill_attn(q, k_cache, v_cache, block_table, seqlens, Hq, Hkv, q_len, sm_scale, out,
                     flags=None, stream=None):
    """Extend / prefill attention: q and out [B, q_len, Hq, 128] bf16, causal
    over each request's last q_len live tokens."""
    _check("hpc_prefill_attn", lib().hpc_prefill_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]), _ptr(block_table),
        int(block_table.shape[1]), _ptr(seqlens), int(seqlens.numel()), int(Hq), int(Hkv),
        HEAD_DIM, int(q_len), float(sm_scale), _ptr(out), _ptr(flags), _stream(stream)))


def hpc_decode_step_host(h_q, h_q_scale, h_seqlens, h_block_table, h_out, d_q, d_q_scale,
                         d_seqlens, d_block_table, d_out, k_cache, v_cache, k_scale, v_scale, Hq,
                         Hkv, sm_scale, num_ctas, min_tiles_per_cta, num_splits, tmap: TaskMap,
                         part_o, part_lse, unit_done=None, stream=None):
    _check("hpc_decode_step_host", lib().hpc_decode_step_host(
        _ptr(h_q), _ptr(h_q_scale), _ptr(h_seqlens), _ptr(h_block_table), _ptr(h_out), _ptr(d_q),
        _ptr(d_q_scale), _ptr(d_seqlens), _ptr(d_block_table), _ptr(d_out), _ptr(k_cache),
        _ptr(v_cache), int(k_cache.shape[0]), float(k_scale), float(v_scale),
        kv_dtype_of(k_cache), int(h_block_table.shape[1]), int(h_seqlens.numel()), int(Hq),
        int(Hkv), HEAD_DIM, float(sm_scale), int(num_ctas), int(min_tiles_per_cta),
        int(num_splits), ctypes.byref(tmap.c), _ptr(part_o), _ptr(part_lse), _ptr(unit_done),
        _stream(stream)))


def hpc_decode_packed_layout(B, Hq, max_pages, kv_dtype=HPC_KV_BF16):
    """(total bytes, [q, q_scale or -1, seqlens, block_table] byte offsets) of the
    packed per-step input."""
    off = (ctypes.c_int64 * 4)()
    total = int(lib().hpc_decode_packed_layout(int(B), int(Hq), int(max_pages), int(kv_dtype),
                                                 off))
    if total < 0:
        raise HpcError("hpc_decode_packed_layout", HPC_ERR_ARG)
    return total, list(off)


def hpc_decode_step_host_packed(h_in, d_in, h_out, d_out, k_cache, v_cache, k_scale, v_scale, B,
                                Hq, Hkv, max_pages, sm_scale, num_ctas, min_tiles_per_cta,
                                num_splits, tmap: TaskMap, part_o, part_lse, unit_done=None,
                                stream=None):
    """One decode step from one packed pinned host buffer (see hpc_decode_packed_layout)."""
    _check("hpc_decode_step_host_packed", lib().hpc_decode_step_host_packed(
        _ptr(h_in), _ptr(d_in), _ptr(h_out), _ptr(d_out), _ptr(k_cache), _ptr(v_cache),
        int(k_cache.shape[0]), float(k_scale), float(v_scale), kv_dtype_of(k_cache),
        int(max_pages), int(B), int(Hq), int(Hkv), HEAD_DIM, float(sm_scale), int(num_ctas),
        int(min_tiles_per_cta), int(num_splits), ctypes.byref(tmap.c), _ptr(part_o),
        _ptr(part_lse), _ptr(unit_done), _stream(stream)))


def hpc_decode_read_meta(tmap: TaskMap, stream=None) -> list:
    host = (ctypes.c_int32 * 4)()
    _check("hpc_decode_read_meta", lib().hpc_decode_read_meta(ctypes.byref(tmap.c), host,
                                                              _stream(stream)))
    return list(host)


def hpc_decode_step_noalloc(q, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, seqlens,
                            Hq, Hkv, sm_scale, num_ctas, min_tiles_per_cta, out, meta_out=None,
                            stream=None):
    """Whole step with the library's built-in scratch; see the C header."""
    _check("hpc_decode_step_noalloc", lib().hpc_decode_step_noalloc(
        _ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]),
        float(k_scale), float(v_scale), kv_dtype_of(k_cache), _ptr(block_table),
        int(block_table.shape[1]), _ptr(seqlens), int(seqlens.numel()), int(Hq), int(Hkv),
        HEAD_DIM, float(sm_scale), int(num_ctas), int(min_tiles_per_cta), _ptr(out),
        _ptr(meta_out), _stream(stream)))


def hpc_rope_frequencies(rope_base, freq, stream=None):
    """The fp64 RoPE frequency table [64] for rope_base, written into `freq`."""
    _check("hpc_rope_frequencies",
           lib().hpc_rope_frequencies(float(rope_base), _ptr(freq), _stream(stream)))


def hpc_rope_norm(qkv, q_norm_w, k_norm_w, positions, token_req, Hq, Hkv, block_table, k_cache,
                  v_cache, k_scale, v_scale, q_out, q_scale_out=None, flags=None, *, eps=1e-6,
                  rope_base=1e6, rope_layout=HPC_ROPE_HALVES, norm_first=True, freq=None,
                  stream=None):
    """Fused prologue: QK-Norm + RoPE of the new tokens' heads, K/V written into
    the paged cache, the query into q_out (and q_scale_out for FP8).  `freq`:
    the table from hpc_rope_frequencies(rope_base), or None."""
    params = hpc_rope_norm_params(float(eps), float(rope_base), int(rope_layout),
                                  1 if norm_first else 0,
                                  None if freq is None else freq.data_ptr())
    _check("hpc_rope_norm", lib().hpc_rope_norm(
        _ptr(qkv), int(qkv.stride(0)), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions),
        _ptr(token_req), int(positions.numel()), int(Hq), int(Hkv), HEAD_DIM, _ptr(block_table),
        int(block_table.shape[1]), int(block_table.shape[0]), _ptr(k_cache), _ptr(v_cache),
        int(k_cache.shape[0]), kv_dtype_of(k_cache), float(k_scale), float(v_scale), _ptr(q_out),
        _ptr(q_scale_out), _ptr(flags), ctypes.byref(params), _stream(stream)))


class Workspace:
    """Split buffer, output and task map sized for one batch shape."""

    def __init__(self, B: int, Hq: int, Hkv: int, *, num_ctas: int = 0, num_splits: int = 0,
                 device="cuda", kv_dtype: int = HPC_KV_BF16, q_len: int = 1):
        dev = torch.device(device)
        if num_splits:
            self.tmap = TaskMap.static(B, Hkv, num_splits, dev)
        else:
            if num_ctas <= 0:
                num_ctas = hpc_decode_num_ctas(dev.index or 0, kv_dtype)
            self.tmap = TaskMap.dynamic(B, Hkv, num_ctas, dev)
        self.num_ctas, self.num_splits = num_ctas, num_splits
        rows = q_len * (Hq // Hkv)  # query rows of one KV head in a descriptor
        cap = max(self.tmap.cap_desc, 1)
        self.q_len = q_len
        self.part_o = torch.empty((cap, rows, HEAD_DIM), dtype=torch.float32, device=dev)
        self.part_lse = torch.empty((cap, rows), dtype=torch.float32, device=dev)
        out_shape = (max(B, 1), Hq, HEAD_DIM) if q_len == 1 else (max(B, 1), q_len, Hq, HEAD_DIM)
        self.out = torch.empty(out_shape, dtype=torch.bfloat16, device=dev)
        # chunk counters of the fused combine: zero once, left zero by every launch
        self.unit_done = torch.zeros(max(B * Hkv, 1), dtype=torch.int32, device=dev)
