"""ctypes binding of libdg (the C ABI declared in include/dg.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  If the library is not built, every call raises: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdg.so")

DG_OK = 0
STATUS_NAMES = {
    0: "DG_OK", 1: "DG_ERR_INVALID_ARGUMENT", 2: "DG_ERR_UNSUPPORTED", 3: "DG_ERR_CUDA",
    4: "DG_ERR_TIMEOUT", 5: "DG_ERR_DEVICE_CHECK", 6: "DG_ERR_WORKSPACE",
}

# Every symbol the header declares, with (restype, argtypes).
_vp, _i32, _i64, _f32, _sz, _u32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                    ctypes.c_size_t, ctypes.c_uint32)


class FFNShape(ctypes.Structure):
    """dg_ffn_shape: P ranks, local batch B, T tokens, model dim D, expansion k, LayerNorm eps."""
    _fields_ = [("P", ctypes.c_int32), ("B", ctypes.c_int32), ("T", ctypes.c_int32),
                ("D", ctypes.c_int32), ("k", ctypes.c_int32), ("eps", ctypes.c_float)]


_PSHAPE = ctypes.POINTER(FFNShape)


class TraceEntry(ctypes.Structure):
    """dg_trace_entry: one kernel name aggregated over its launches."""
    _fields_ = [("name", ctypes.c_char * 40), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]

DG_ERROR_BLOCK_BYTES = 256
DG_FFN_COMP_ONLY = 1
DG_FFN_FUSED_GATE = 2
DG_FFN_SEPARATE_GATE = 4

SIGNATURES = {
    "dg_last_error": (ctypes.c_char_p, []),
    "dg_version": (ctypes.c_char_p, []),
    "dg_workspace_init": (ctypes.c_int, [_vp, _sz, _vp]),
    "dg_check_device_error": (ctypes.c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)]),
    "dg_debug_wait_timeout": (ctypes.c_int, [_vp, _sz, _u32, _vp]),
    "dg_gemm_fp8_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "dg_gemm_fp8": (ctypes.c_int, [_i64, _i64, _i64, _vp, _vp, _vp, _vp, _f32, _f32, _vp, _sz, _vp]),
    "dg_a2a_ffn_saved_bytes": (_sz, [_PSHAPE]),
    "dg_a2a_ffn_fwd_workspace_bytes": (_sz, [_PSHAPE, _i32, _u32]),
    "dg_a2a_ffn_fwd": (ctypes.c_int, [_PSHAPE] + [_vp] * 10 + [_vp, _sz, _vp, _sz, _u32, _vp]),
    "dg_a2a_ffn_bwd_workspace_bytes": (_sz, [_PSHAPE, _u32]),
    "dg_a2a_ffn_bwd": (ctypes.c_int, [_PSHAPE] + [_vp] * 9 + [_vp, _sz, _vp] + [_vp] * 9 + [_vp, _sz, _u32, _vp]),
    "dg_a2a_dispatch": (ctypes.c_int, [_i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "dg_a2a_combine": (ctypes.c_int, [_i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "dg_tp_swiglu_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32, _i32]),
    "dg_tp_swiglu": (ctypes.c_int, [_i64, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dg_tp_swiglu_bwd_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32, _i32]),
    "dg_tp_swiglu_bwd": (ctypes.c_int, [_i64, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                        _vp]),
    "dg_a2a_ffn_fp8_weights_bytes": (_sz, [_PSHAPE]),
    "dg_a2a_ffn_fp8_workspace_bytes": (_sz, [_PSHAPE]),
    "dg_a2a_ffn_fp8_pack_weights": (ctypes.c_int, [_PSHAPE, _vp, _vp, _vp, _sz, _vp]),
    "dg_a2a_ffn_fwd_fp8": (ctypes.c_int, [_PSHAPE, _vp, _vp, _sz, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dg_tp_linear_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "dg_tp_linear_fwd": (ctypes.c_int, [_i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dg_tp_linear_bwd": (ctypes.c_int, [_i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dg_tp_swiglu_noalloc": (ctypes.c_int, [_i64, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "dg_trace_begin": (ctypes.c_int, []),
    "dg_trace_begin_only": (ctypes.c_int, [ctypes.c_char_p]),
    "dg_trace_end": (ctypes.c_int32, [ctypes.POINTER(TraceEntry), ctypes.c_int32]),
}

_lock = threading.Lock()
_lib = None


class DGError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def load():
    """Load libdg.so (once); raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m expert_gemm_layers_gb300.build` "
                    "(or __graft_entry__.build()); there is no fallback implementation")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def check(status: int) -> None:
    if status != DG_OK:
        msg = load().dg_last_error().decode(errors="replace")
        raise DGError(status, msg)
