"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and rejects invalid arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dg.h")


@pytest.fixture(scope="module")
def lib():
    from expert_gemm_layers_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from expert_gemm_layers_gb300 import build
        build.build()
    return _lib.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    from expert_gemm_layers_gb300 import _lib
    assert set(names) == set(_lib.SIGNATURES), set(names) ^ set(_lib.SIGNATURES)


def test_version_and_empty_error(lib):
    assert b"sm_103a" in lib.dg_version()


def _shape(P, B, T, D, k, eps=1e-5):
    from expert_gemm_layers_gb300._lib import FFNShape
    return FFNShape(P, B, T, D, k, eps)


def test_ffn_shape_validation_without_gpu(lib):
    from expert_gemm_layers_gb300._lib import STATUS_NAMES
    bad = [_shape(3, 1, 16, 128, 2), _shape(2, 1, 16, 100, 2), _shape(0, 1, 16, 128, 2),
           _shape(2, 1, 16, 128, 2, eps=0.0), _shape(2, 1, 16, 8192, 9)]  # last: H = 73728 > 65536
    for sh in bad:
        st = lib.dg_a2a_ffn_fwd(ctypes.byref(sh), *([None] * 10), None, 0, None, 0, 0, None)
        assert STATUS_NAMES[st] in ("DG_ERR_INVALID_ARGUMENT", "DG_ERR_UNSUPPORTED"), (st, lib.dg_last_error())
        assert lib.dg_last_error()
        assert lib.dg_a2a_ffn_saved_bytes(ctypes.byref(sh)) == 0


def test_ffn_saved_and_workspace_sizes(lib):
    sh = _shape(8, 512, 64, 1280, 6)
    rows, H = 64 * 4096, 7680
    saved = lib.dg_a2a_ffn_saved_bytes(ctypes.byref(sh))
    assert saved >= rows * (2 * H * 2 + H * 2 + 16)
    ws = lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), 0)
    assert ws >= 256 + rows * (H * 2 + 2 * H * 2)
    act = 8 * 512 * 64 * 1280 * 2
    assert lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), 1) >= ws + 3 * act     # comp_only buffers
    # the backward takes the forward's flags; the gate flags do not change it
    assert lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), 2) == ws
    assert lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), 4) == ws
    assert lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), 2 | 4) == 0           # exclusive flags
    assert lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), 8) == 0               # unknown flag
    # forward: training needs the error block only; inference holds Z, the statistics and partials
    assert lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 0, 0) == 256
    inf = lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 1, 0)
    assert inf >= 256 + rows * (2 * H * 2 + 16 + H * 2)
    # with the gate fused into the second GEMM (the default), inference needs Hl scratch only when D is
    # wider than one gated column pass (512 columns): the remaining columns come from a plain GEMM on the Hl
    # it stores; the separate pass (flag 4) always needs it
    assert lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 1, 4) == inf
    assert lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 1, 2) == inf
    narrow = _shape(2, 4, 16, 512, 2)
    rows_n, H_n = 16 * 8, 1024
    inf_n = lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(narrow), 1, 4)
    assert lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(narrow), 1, 0) <= inf_n - rows_n * H_n * 2
    assert lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 1, 2 | 4) == 0         # exclusive flags
    assert lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 0, 1) >= 256 + 2 * act
    assert lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 0, 8) == 0             # unknown flag


def _aligned(buf):
    return ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256


def test_null_pointer_rejected(lib):
    sh = _shape(2, 4, 16, 128, 2)
    st = lib.dg_a2a_ffn_fwd(ctypes.byref(sh), *([None] * 10), None, 0, None, 0, 0, None)
    assert st == 1 and b"NULL" in lib.dg_last_error()


def test_ffn_flags_and_error_block_checked_before_the_device(lib):
    from expert_gemm_layers_gb300._lib import STATUS_NAMES
    sh = _shape(2, 4, 16, 128, 2)
    buf = ctypes.create_string_buffer(12 << 16)
    p = [_aligned(buf) + (i << 16) for i in range(11)]   # distinct, non-overlapping stand-ins
    args = [ctypes.byref(sh)] + p[:10]
    # an unknown flag, and the two gate flags together
    st = lib.dg_a2a_ffn_fwd(*args, None, 0, p[10], 256, 8, None)
    assert STATUS_NAMES[st] == "DG_ERR_INVALID_ARGUMENT" and b"flags" in lib.dg_last_error()
    st = lib.dg_a2a_ffn_fwd(*args, None, 0, p[10], 256, 2 | 4, None)
    assert STATUS_NAMES[st] == "DG_ERR_INVALID_ARGUMENT" and b"exclude" in lib.dg_last_error()
    # no workspace at all: the error block is missing
    st = lib.dg_a2a_ffn_fwd(*args, None, 0, None, 0, 0, None)
    assert STATUS_NAMES[st] == "DG_ERR_WORKSPACE" and b"error block" in lib.dg_last_error()
    # a workspace smaller than its query
    st = lib.dg_a2a_ffn_fwd(*args, None, 0, p[10], 128, 0, None)
    assert STATUS_NAMES[st] == "DG_ERR_WORKSPACE"
    # backward: a requested gradient whose input is missing (d_inputs needs w1)
    bw = [ctypes.byref(sh), p[0], None] + p[2:9]        # w1 = NULL
    st = lib.dg_a2a_ffn_bwd(*bw, p[9], 1 << 12, p[10], p[1], None, None, None, None, None, None, None, None,
                            None, 0, 0, None)
    assert STATUS_NAMES[st] == "DG_ERR_INVALID_ARGUMENT" and b"w1" in lib.dg_last_error()
    # backward: the forward's flags, checked the same way
    st = lib.dg_a2a_ffn_bwd(ctypes.byref(sh), *p[:9], p[9], 1 << 12, p[10], *([None] * 9), None, 0, 8, None)
    assert STATUS_NAMES[st] == "DG_ERR_INVALID_ARGUMENT" and b"flags" in lib.dg_last_error()
    st = lib.dg_a2a_ffn_bwd(ctypes.byref(sh), *p[:9], p[9], 1 << 12, p[10], *([None] * 9), None, 0, 2 | 4, None)
    assert STATUS_NAMES[st] == "DG_ERR_INVALID_ARGUMENT" and b"exclude" in lib.dg_last_error()


def test_error_block_query_functions(lib):
    assert lib.dg_gemm_fp8_workspace_bytes(4096, 4096, 4096) == 256
    assert lib.dg_tp_linear_workspace_bytes(8192, 4096, 6144) == 256
    from expert_gemm_layers_gb300._lib import STATUS_NAMES
    assert STATUS_NAMES[lib.dg_workspace_init(None, 0, None)] == "DG_ERR_WORKSPACE"
    buf = ctypes.create_string_buffer(512)
    assert STATUS_NAMES[lib.dg_debug_wait_timeout(_aligned(buf) + 8, 256, 1000, None)] == "DG_ERR_INVALID_ARGUMENT"


def test_gemm_fp8_validation_without_gpu(lib):
    assert lib.dg_gemm_fp8(-1, 8, 16, None, None, None, None, 1.0, 0.0, None, 0, None) == 1
    assert lib.dg_gemm_fp8(8, 8, 17, None, None, None, None, 1.0, 0.0, None, 0, None) == 1     # K % 16
    assert lib.dg_gemm_fp8(8, 12, 16, None, None, None, None, 1.0, 0.0, None, 0, None) == 1    # N % 8
    assert lib.dg_gemm_fp8(0, 8, 16, None, None, None, None, 1.0, 0.0, None, 0, None) == 0     # empty: no-op
    buf = ctypes.create_string_buffer(8192)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    ws = p + 4096
    assert lib.dg_gemm_fp8(8, 8, 16, p, p, None, p, 1.0, 1.0, ws, 256, None) == 1               # C NULL, beta != 0
    assert lib.dg_gemm_fp8(8, 8, 16, p, p + 1024, None, p, 1.0, 0.0, ws, 256, None) == 1         # D overlaps A
    assert lib.dg_gemm_fp8(8, 8, 16, p, p + 512, None, p + 1024, 1.0, 0.0, None, 0, None) == 6   # no error block
    assert lib.dg_gemm_fp8(8, 8, 16, p, p + 512, None, p + 1024, 1.0, 0.0, ws, 64, None) == 6    # too small


def test_tp_swiglu_validation_without_gpu(lib):
    assert lib.dg_tp_swiglu(100, 64, 128, 8, 1, *([None] * 5), 0, None) == 1          # S % W
    assert lib.dg_tp_swiglu(64, 64, 100, 8, 1, *([None] * 5), 0, None) == 1           # ffn % W
    assert lib.dg_tp_swiglu_workspace_bytes(8192, 4096, 14336, 8, 1) == 256 + 8192 * 14336 * 2


def test_tp_swiglu_noalloc_size_limits_without_gpu(lib):
    from expert_gemm_layers_gb300._lib import STATUS_NAMES
    buf = ctypes.create_string_buffer(4096)
    p = [_aligned(buf) + 256 * i for i in range(4)]
    # d beyond 2^31-1 (with S = W = 8, bsz = 1): refused before any device call
    d = (1 << 31) + 8
    assert STATUS_NAMES[lib.dg_tp_swiglu_noalloc(8, d, 64, 8, 1, *p, None)] == "DG_ERR_UNSUPPORTED"
    assert b"2^31" in lib.dg_last_error()
    # S * bsz beyond 2^31-1 although each is below it
    assert STATUS_NAMES[lib.dg_tp_swiglu_noalloc(1 << 30, 64, 64, 8, 4, *p, None)] == "DG_ERR_UNSUPPORTED"
    # h one shard row above the 32 MiB scratch: S*bsz*ffn*2 = (2048 + 8) * 8192 * 2
    assert STATUS_NAMES[lib.dg_tp_swiglu_noalloc(2056, 64, 8192, 8, 1, *p, None)] == "DG_ERR_UNSUPPORTED"
    assert b"scratch" in lib.dg_last_error()


def test_trace_without_launches(lib):
    from expert_gemm_layers_gb300 import trace_begin, trace_end
    trace_begin()
    assert trace_end() == []
