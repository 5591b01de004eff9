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
        st = lib.dg_a2a_ffn_fwd(ctypes.byref(sh), *([None] * 10), None, 0, None)
        assert STATUS_NAMES[st] in ("DG_ERR_INVALID_ARGUMENT", "DG_ERR_UNSUPPORTED"), (st, lib.dg_last_error())
        assert lib.dg_last_error()
        assert lib.dg_a2a_ffn_saved_bytes(ctypes.byref(sh)) == 0


def test_ffn_saved_and_workspace_sizes(lib):
    sh = _shape(8, 512, 64, 1280, 6)
    rows, H = 64 * 4096, 7680
    saved = lib.dg_a2a_ffn_saved_bytes(ctypes.byref(sh))
    assert saved >= rows * (2 * H * 2 + H * 2 + 16)
    ws = lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh))
    assert ws >= rows * (H * 2 + 2 * H * 2)


def test_null_pointer_rejected(lib):
    sh = _shape(2, 4, 16, 128, 2)
    st = lib.dg_a2a_ffn_fwd(ctypes.byref(sh), *([None] * 10), None, 0, None)
    assert st == 1 and b"NULL" in lib.dg_last_error()


def test_gemm_fp8_validation_without_gpu(lib):
    assert lib.dg_gemm_fp8(-1, 8, 16, None, None, None, None, 1.0, 0.0, None) == 1
    assert lib.dg_gemm_fp8(8, 8, 17, None, None, None, None, 1.0, 0.0, None) == 1     # K % 16
    assert lib.dg_gemm_fp8(8, 12, 16, None, None, None, None, 1.0, 0.0, None) == 1    # N % 8
    assert lib.dg_gemm_fp8(0, 8, 16, None, None, None, None, 1.0, 0.0, None) == 0     # empty: no-op
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    assert lib.dg_gemm_fp8(8, 8, 16, p, p, None, p, 1.0, 1.0, None) == 1               # C NULL, beta != 0
    assert lib.dg_gemm_fp8(8, 8, 16, p, p + 1024, None, p, 1.0, 0.0, None) == 1         # D overlaps A


def test_tp_swiglu_validation_without_gpu(lib):
    assert lib.dg_tp_swiglu(100, 64, 128, 8, 1, *([None] * 5), 0, None) == 1          # S % W
    assert lib.dg_tp_swiglu(64, 64, 100, 8, 1, *([None] * 5), 0, None) == 1           # ffn % W
    assert lib.dg_tp_swiglu_workspace_bytes(8192, 4096, 14336, 8, 1) == 8192 * 14336 * 2


def test_trace_without_launches(lib):
    from expert_gemm_layers_gb300 import trace_begin, trace_end
    trace_begin()
    assert trace_end() == []
