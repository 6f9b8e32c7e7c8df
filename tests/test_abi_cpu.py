"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point the header declares, and rejects bad
arguments before touching CUDA (fake, never-dereferenced device pointers)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hpc_decode.h")


@pytest.fixture(scope="module")
def hd():
    from load_balanced_paged_assign_gb300 import _build
    _build.build()
    import load_balanced_paged_assign_gb300 as pkg
    return pkg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hpc_[a-z_0-9]+)\s*\(", text)))


def test_header_and_binding_agree(hd):
    assert declared_functions() == sorted(hd.EXPORTS)


def test_library_exports_every_declared_symbol(hd):
    L = hd.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert "sm_103a" in hd.hpc_decode_version()


def test_capacities(hd):
    assert hd.hpc_decode_desc_capacity(4, 1, 132) == 136
    assert hd.hpc_decode_desc_capacity(64, 8, 152) == 152 + 512
    assert hd.hpc_decode_static_capacity(64, 8, 4) == 2048
    assert hd.hpc_decode_desc_capacity(-1, 1, 1) == -1


FAKE = 0x10000  # 16-byte aligned, never dereferenced on the host


def fake_map(hd, cap_desc=200, cap_bins=200, cap_units=64):
    m = hd.binding.hpc_task_map(FAKE, FAKE, FAKE, FAKE, FAKE, cap_desc, cap_bins, cap_units, 0, 0,
                                0, 0, 0, 0)
    return m


def call_plan(hd, B=4, Hkv=1, max_pages=32, ctas=132, floor=2, m=None, seqlens=FAKE):
    m = m if m is not None else fake_map(hd)
    return hd.lib().hpc_decode_plan(seqlens, B, Hkv, max_pages, ctas, floor, ctypes.byref(m),
                                    None)


def test_plan_argument_checks(hd):
    assert call_plan(hd, B=-1) == hd.binding.HPC_ERR_ARG
    assert call_plan(hd, Hkv=0) == hd.binding.HPC_ERR_ARG
    assert call_plan(hd, ctas=0) == hd.binding.HPC_ERR_ARG
    assert call_plan(hd, floor=-1) == hd.binding.HPC_ERR_ARG
    assert call_plan(hd, seqlens=None) == hd.binding.HPC_ERR_ARG
    assert call_plan(hd, B=20000) == hd.binding.HPC_ERR_UNSUPPORTED
    # capacities: desc below num_ctas + B*Hkv, bin_ptr below num_ctas + 1, units below B*Hkv
    assert call_plan(hd, m=fake_map(hd, cap_desc=135)) == hd.binding.HPC_ERR_WORKSPACE
    assert call_plan(hd, m=fake_map(hd, cap_bins=132)) == hd.binding.HPC_ERR_WORKSPACE
    assert call_plan(hd, B=8, Hkv=8, m=fake_map(hd, cap_desc=500, cap_units=63)) == \
        hd.binding.HPC_ERR_WORKSPACE
    bad = fake_map(hd)
    bad.desc = FAKE + 4  # misaligned descriptor array
    assert call_plan(hd, m=bad) == hd.binding.HPC_ERR_ARG
    bad = fake_map(hd)
    bad.meta = None
    assert call_plan(hd, m=bad) == hd.binding.HPC_ERR_ARG


def test_static_plan_argument_checks(hd):
    L = hd.lib()
    m = fake_map(hd, cap_desc=16, cap_bins=17, cap_units=4)
    assert L.hpc_decode_plan_static(FAKE, 4, 1, 8, 0, ctypes.byref(m), None) == \
        hd.binding.HPC_ERR_ARG
    assert L.hpc_decode_plan_static(FAKE, 4, 1, 8, 5, ctypes.byref(m), None) == \
        hd.binding.HPC_ERR_WORKSPACE
    m = fake_map(hd, cap_desc=16, cap_bins=16, cap_units=4)
    assert L.hpc_decode_plan_static(FAKE, 4, 1, 8, 4, ctypes.byref(m), None) == \
        hd.binding.HPC_ERR_WORKSPACE


def call_attn(hd, m, q=FAKE, q_scale=None, k=FAKE, v=FAKE, num_pages=10, dtype=0, bt=FAKE,
              max_pages=4, seqlens=FAKE, B=4, Hq=8, Hkv=1, D=128, sm=0.088, po=FAKE, pl=FAKE):
    return hd.lib().hpc_decode_attn(q, q_scale, k, v, num_pages, 1.0, 1.0, dtype, bt, max_pages,
                                    seqlens, B, Hq, Hkv, D, sm, ctypes.byref(m), po, pl, None)


def test_attn_argument_checks(hd):
    m = fake_map(hd)
    m.B, m.Hkv, m.num_ctas = 4, 1, 132
    E = hd.binding
    assert call_attn(hd, m, D=64) == E.HPC_ERR_UNSUPPORTED
    assert call_attn(hd, m, Hq=17, Hkv=1) == E.HPC_ERR_UNSUPPORTED  # G = 17 > 16
    assert call_attn(hd, m, Hq=64, Hkv=2) == E.HPC_ERR_UNSUPPORTED  # G = 32 > 16
    assert call_attn(hd, m, Hq=10, Hkv=4) == E.HPC_ERR_UNSUPPORTED  # Hq % Hkv != 0
    assert call_attn(hd, m, q=FAKE + 8) == E.HPC_ERR_ARG  # misaligned Q
    assert call_attn(hd, m, k=FAKE + 2) == E.HPC_ERR_ARG
    assert call_attn(hd, m, num_pages=0) == E.HPC_ERR_ARG
    assert call_attn(hd, m, dtype=7) == E.HPC_ERR_ARG
    assert call_attn(hd, m, dtype=1) == E.HPC_ERR_ARG  # FP8 without q_scale
    assert call_attn(hd, m, sm=float("nan")) == E.HPC_ERR_ARG
    assert call_attn(hd, m, B=5) == E.HPC_ERR_ARG  # map planned for another batch
    m.num_ctas = 0
    assert call_attn(hd, m) == E.HPC_ERR_ARG  # map never planned


def test_combine_argument_checks(hd):
    m = fake_map(hd)
    m.B, m.Hkv, m.num_ctas = 4, 1, 132
    L = hd.lib()
    E = hd.binding
    assert L.hpc_decode_combine(FAKE, FAKE, ctypes.byref(m), 4, 8, 1, 256, FAKE, None) == \
        E.HPC_ERR_UNSUPPORTED
    assert L.hpc_decode_combine(FAKE, FAKE, ctypes.byref(m), 4, 8, 1, 128, FAKE + 4, None) == \
        E.HPC_ERR_ARG
    assert L.hpc_decode_combine(None, FAKE, ctypes.byref(m), 4, 8, 1, 128, FAKE, None) == \
        E.HPC_ERR_ARG
    assert L.hpc_decode_combine(FAKE, FAKE, ctypes.byref(m), 3, 8, 1, 128, FAKE, None) == \
        E.HPC_ERR_ARG


def test_status_strings(hd):
    assert hd.binding.status_string(0) == "ok"
    assert hd.binding.status_string(-3) == "workspace too small"


def test_fused_attention_argument_checks(hd):
    m = fake_map(hd)
    m.B, m.Hkv, m.num_ctas = 4, 1, 132
    L = hd.lib()
    args = [FAKE, None, FAKE, FAKE, 10, 1.0, 1.0, 0, FAKE, 4, FAKE, 4, 8, 1, 128, 0.088,
            ctypes.byref(m), FAKE, FAKE]
    assert L.hpc_decode_attn_combine(*args, None, FAKE, None) == hd.binding.HPC_ERR_ARG
    assert L.hpc_decode_attn_combine(*args, FAKE, None, None) == hd.binding.HPC_ERR_ARG
    assert L.hpc_decode_attn_combine(*args, FAKE, FAKE + 8, None) == hd.binding.HPC_ERR_ARG


def call_rope_norm(hd, qkv=FAKE, stride=1280, N=4, Hq=8, Hkv=1, D=128, B=4, dtype=0,
                   q_scale=None, qout=FAKE, params="default", token_req=None, k_scale=1.0,
                   max_pages=16):
    P = hd.binding.hpc_rope_norm_params
    p = P(1e-6, 1e6, 0, 1, None) if params == "default" else params
    return hd.lib().hpc_rope_norm(qkv, stride, FAKE, FAKE, FAKE, token_req, N, Hq, Hkv, D, FAKE,
                                  max_pages, B, FAKE, FAKE, 10, dtype, k_scale, 1.0, qout,
                                  q_scale, None, None if p is None else ctypes.byref(p), None)


def test_rope_norm_argument_checks(hd):
    E = hd.binding
    P = E.hpc_rope_norm_params
    assert call_rope_norm(hd, N=0) == E.HPC_OK  # nothing to do, nothing launched
    assert call_rope_norm(hd, params=None) == E.HPC_ERR_ARG
    assert call_rope_norm(hd, D=64) == E.HPC_ERR_UNSUPPORTED
    assert call_rope_norm(hd, Hq=12, Hkv=8) == E.HPC_ERR_UNSUPPORTED
    assert call_rope_norm(hd, stride=1272) == E.HPC_ERR_ARG  # shorter than a token's heads
    assert call_rope_norm(hd, stride=1284) == E.HPC_ERR_ARG  # not a multiple of 8 elements
    assert call_rope_norm(hd, qkv=FAKE + 8) == E.HPC_ERR_ARG
    assert call_rope_norm(hd, dtype=1) == E.HPC_ERR_ARG  # FP8 without q_scale_out
    assert call_rope_norm(hd, dtype=1, q_scale=FAKE, k_scale=0.0) == E.HPC_ERR_ARG
    assert call_rope_norm(hd, dtype=5) == E.HPC_ERR_ARG
    assert call_rope_norm(hd, N=5, B=4) == E.HPC_ERR_ARG  # token t is request t: needs N <= B
    assert call_rope_norm(hd, qout=None) == E.HPC_ERR_ARG
    assert call_rope_norm(hd, params=P(-1.0, 1e6, 0, 1, None)) == E.HPC_ERR_ARG
    assert call_rope_norm(hd, params=P(1e-6, 0.0, 0, 1, None)) == E.HPC_ERR_ARG
    assert call_rope_norm(hd, params=P(1e-6, float("inf"), 0, 1, None)) == E.HPC_ERR_ARG
    assert call_rope_norm(hd, params=P(1e-6, 1e6, 2, 1, None)) == E.HPC_ERR_ARG
    assert call_rope_norm(hd, params=P(1e-6, 1e6, 0, 2, None)) == E.HPC_ERR_ARG
    assert call_rope_norm(hd, params=P(1e-6, 1e6, 0, 1, FAKE + 8)) == E.HPC_ERR_ARG  # freq
    # positions must stay exact in fp32: at most 2^24 cache slots per request
    assert call_rope_norm(hd, max_pages=(1 << 18) + 1) == E.HPC_ERR_UNSUPPORTED
    assert call_rope_norm(hd, Hq=400, Hkv=8) == E.HPC_ERR_UNSUPPORTED  # too many head rows
    L = hd.lib()
    assert L.hpc_rope_frequencies(0.0, FAKE, None) == E.HPC_ERR_ARG
    assert L.hpc_rope_frequencies(1e4, None, None) == E.HPC_ERR_ARG
    assert L.hpc_rope_frequencies(1e4, FAKE + 8, None) == E.HPC_ERR_ARG


def test_multi_query_argument_checks(hd):
    m = fake_map(hd)
    m.B, m.Hkv, m.num_ctas = 4, 1, 132
    L = hd.lib()
    E = hd.binding

    def attn(q_len, Hq=8, Hkv=1):
        return L.hpc_decode_attn_mq(FAKE, None, FAKE, FAKE, 10, 1.0, 1.0, 0, FAKE, 4, FAKE, 4,
                                    Hq, Hkv, 128, q_len, 0.088, ctypes.byref(m), FAKE, FAKE, None)

    assert attn(0) == E.HPC_ERR_ARG
    assert attn(3) == E.HPC_ERR_UNSUPPORTED  # 3 x 8 = 24 query rows per KV head > 16
    assert attn(17, Hq=1) == E.HPC_ERR_UNSUPPORTED
    assert L.hpc_decode_combine_mq(FAKE, FAKE, ctypes.byref(m), 4, 8, 1, 128, 0, FAKE,
                                   None) == E.HPC_ERR_ARG
    assert L.hpc_decode_combine_mq(FAKE, FAKE, ctypes.byref(m), 4, 8, 1, 128, 3, FAKE,
                                   None) == E.HPC_ERR_UNSUPPORTED
    assert L.hpc_decode_step_mq(FAKE, None, FAKE, FAKE, 10, 1.0, 1.0, 0, FAKE, 4, FAKE, 4, 8, 1,
                                128, 4, 0.088, 132, 2, 0, ctypes.byref(m), FAKE, FAKE, FAKE, FAKE,
                                None) == E.HPC_ERR_UNSUPPORTED


def test_router_argument_checks(hd):
    L = hd.lib()
    E = hd.binding
    assert L.hpc_router_gemm(FAKE, FAKE, FAKE, 0, 192, 4096, FAKE, None, 0, None, None) == E.HPC_OK
    assert L.hpc_router_gemm(FAKE, FAKE, FAKE, 4, 192, 4000, FAKE, None, 0, None, None) == \
        E.HPC_ERR_UNSUPPORTED  # K not a multiple of 64
    assert L.hpc_router_gemm(FAKE, FAKE, FAKE, 4, 190, 4096, FAKE, None, 0, None, None) == \
        E.HPC_ERR_UNSUPPORTED  # N not a multiple of 16
    assert L.hpc_router_gemm(None, FAKE, FAKE, 4, 192, 4096, FAKE, None, 0, None, None) == \
        E.HPC_ERR_ARG
    assert L.hpc_router_gemm(FAKE + 8, FAKE, FAKE, 4, 192, 4096, FAKE, None, 0, None, None) == \
        E.HPC_ERR_ARG
    assert L.hpc_router_gemm(FAKE, FAKE, FAKE, -1, 192, 4096, FAKE, None, 0, None, None) == \
        E.HPC_ERR_ARG
    assert L.hpc_router_split(None, 192, 4096, FAKE, FAKE, None) == E.HPC_ERR_ARG
    assert L.hpc_router_split(FAKE, 0, 4096, FAKE, FAKE, None) == E.HPC_ERR_ARG
    assert L.hpc_router_workspace_bytes(4, 192, 4000) == -1
    assert L.hpc_router_workspace_bytes(0, 192, 4096) == 0
    plan = (ctypes.c_int32 * 4)()
    assert L.hpc_router_plan(4, 192, 4000, plan) == E.HPC_ERR_UNSUPPORTED
    assert L.hpc_router_plan(4, 192, 4096, None) == E.HPC_ERR_ARG
    assert L.hpc_router_plan(-1, 192, 4096, plan) == E.HPC_ERR_ARG
    assert L.hpc_router_plan(0, 192, 4096, plan) == E.HPC_OK and list(plan) == [0, 0, 0, 0]
    # few tokens: the CUDA-core kernel, two experts per CTA (no device needed)
    assert L.hpc_router_plan(16, 192, 4096, plan) == E.HPC_OK and list(plan) == [0, 0, 0, 96]


def test_prefill_argument_checks(hd):
    L = hd.lib()
    E = hd.binding

    def call(q=FAKE, k=FAKE, v=FAKE, num_pages=100, bt=FAKE, max_pages=8, sl=FAKE, B=2, Hq=8,
             Hkv=2, D=128, q_len=300, sm=0.088, out=FAKE):
        return L.hpc_prefill_attn(q, k, v, num_pages, bt, max_pages, sl, B, Hq, Hkv, D, q_len,
                                  sm, out, None, None)

    assert call(B=0) == E.HPC_OK  # nothing to do, nothing launched
    assert call(D=64) == E.HPC_ERR_UNSUPPORTED
    assert call(Hq=6, Hkv=4) == E.HPC_ERR_UNSUPPORTED
    assert call(q_len=0) == E.HPC_ERR_ARG
    assert call(B=-1) == E.HPC_ERR_ARG
    assert call(num_pages=0) == E.HPC_ERR_ARG
    assert call(max_pages=0) == E.HPC_ERR_ARG
    assert call(q=None) == E.HPC_ERR_ARG
    assert call(out=None) == E.HPC_ERR_ARG
    assert call(sl=None) == E.HPC_ERR_ARG
    assert call(q=FAKE + 8) == E.HPC_ERR_ARG  # not 16-byte aligned
    assert call(k=FAKE + 4) == E.HPC_ERR_ARG
    assert call(sm=float("inf")) == E.HPC_ERR_ARG
    assert call(max_pages=1 << 24) == E.HPC_ERR_UNSUPPORTED  # token index past int32 range


def test_packed_layout(hd):
    E = hd.binding
    total, off = hd.hpc_decode_packed_layout(32, 8, 512, E.HPC_KV_BF16)
    assert off == [0, -1, 32 * 8 * 128 * 2, 32 * 8 * 128 * 2 + 128]
    assert total == off[3] + 32 * 512 * 4
    total, off = hd.hpc_decode_packed_layout(3, 8, 5, E.HPC_KV_FP8_E4M3)
    assert off[0] == 0 and off[1] == 3 * 8 * 128 and off[2] == off[1] + 96
    assert all(o % 16 == 0 for o in off) and total % 16 == 0
    assert off[3] >= off[2] + 3 * 4 and total >= off[3] + 3 * 5 * 4
    L = hd.lib()
    o = (ctypes.c_int64 * 4)()
    assert L.hpc_decode_packed_layout(-1, 8, 5, 0, o) == -1
    assert L.hpc_decode_packed_layout(3, 8, 0, 0, o) == -1
    assert L.hpc_decode_packed_layout(3, 8, 5, 7, o) == -1


def test_packed_step_argument_checks(hd):
    L = hd.lib()
    E = hd.binding
    m = E.hpc_task_map()

    def call(h_in=FAKE, d_in=FAKE, h_out=FAKE, d_out=FAKE, B=4, D=128, unit_done=FAKE):
        return L.hpc_decode_step_host_packed(h_in, d_in, h_out, d_out, FAKE, FAKE, 100, 1.0, 1.0,
                                             0, 8, B, 8, 1, D, 0.088, 132, 2, 0,
                                             ctypes.byref(m), FAKE, FAKE, unit_done, None)

    assert call(h_in=None) == E.HPC_ERR_ARG
    assert call(h_out=None) == E.HPC_ERR_ARG
    # no device output: the kernels store into h_out, which needs the fused
    # combine and a device-mapped pinned host buffer
    assert call(d_out=None, unit_done=None) == E.HPC_ERR_ARG
    assert call(d_out=None) == E.HPC_ERR_ARG  # FAKE is no registered host memory
    assert call(d_in=FAKE + 8) == E.HPC_ERR_ARG  # device staging not 16-byte aligned
    assert call(D=64) == E.HPC_ERR_UNSUPPORTED


def test_selftest_argument_checks(hd):
    L = hd.lib()
    E = hd.binding
    assert L.hpc_selftest_wait_timeout(None, 1000, None) == E.HPC_ERR_ARG
    assert L.hpc_selftest_wait_timeout(FAKE, 0, None) == E.HPC_ERR_ARG
    assert L.hpc_selftest_wait_timeout(FAKE, 1000001, None) == E.HPC_ERR_ARG


def test_noalloc_step_shape_checks_come_first(hd):
    """The allocation-free step rejects what hpc_decode_step rejects, with the
    same status and before it sizes or looks up its built-in scratch; only a
    supported problem too large for the scratch gets HPC_ERR_WORKSPACE."""
    L = hd.lib()
    E = hd.binding

    def call(B=4, Hq=8, Hkv=1, D=128, dtype=0, ctas=132, max_pages=4):
        return L.hpc_decode_step_noalloc(FAKE, None, FAKE, FAKE, 10, 1.0, 1.0, dtype, FAKE,
                                         max_pages, FAKE, B, Hq, Hkv, D, 0.088, ctas, 2, FAKE,
                                         None, None)

    assert call(D=64) == E.HPC_ERR_UNSUPPORTED
    assert call(Hq=17, Hkv=1) == E.HPC_ERR_UNSUPPORTED  # G = 17 > 16
    assert call(Hq=10, Hkv=4) == E.HPC_ERR_UNSUPPORTED
    assert call(B=20000) == E.HPC_ERR_UNSUPPORTED  # above HPC_MAX_BATCH
    assert call(dtype=7) == E.HPC_ERR_ARG
    assert call(B=-1) == E.HPC_ERR_ARG
    assert call(ctas=0) == E.HPC_ERR_ARG
    assert call(max_pages=0) == E.HPC_ERR_ARG
    # supported shapes whose descriptors and partials exceed the 8 MiB array
    assert call(B=16384, Hq=16, Hkv=1) == E.HPC_ERR_WORKSPACE
    assert call(ctas=2 ** 31 - 1) == E.HPC_ERR_WORKSPACE  # sized without wrapping
