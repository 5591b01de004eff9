"""dg_tp_swiglu_noalloc, the allocation-free SwiGLU entry point, called through
the C ABI: its output must match dg_tp_swiglu's (the workspace-taking entry
point) on two calls in a row, and requests larger than its built-in scratch
must be refused before anything is enqueued.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test."""
import ctypes

import pytest
import torch

from expert_gemm_layers_gb300 import _lib, synth, tp_swiglu
from _compare import TOL_BF16, err_max

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
SCRATCH_BYTES = 32 << 20


def _noalloc(x, w13, w2, y):
    lib = _lib.load()
    W, bsz, sl, d = x.shape
    ffn = w2.shape[1]
    st = lib.dg_tp_swiglu_noalloc(W * sl, d, ffn, W, bsz, ctypes.c_void_p(x.data_ptr()),
                                  ctypes.c_void_p(w13.data_ptr()), ctypes.c_void_p(w2.data_ptr()),
                                  ctypes.c_void_p(y.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, lib.dg_last_error().decode()


@pytest.mark.parametrize("S,d,ffn,W", [(1024, 512, 2048, 8), (320, 136, 576, 8),
                                       (2048, 64, 8192, 8)])   # last: h is exactly the 32 MiB scratch
def test_noalloc_matches_workspace_entry_point_twice(S, d, ffn, W):
    x, w13, w2 = synth.tp_swiglu_inputs(S, d, ffn, W, seed=S + ffn, device=DEV)
    ref = tp_swiglu(x, w13, w2)
    for _ in range(2):
        y = torch.full_like(x, float("nan"))
        st, msg = _noalloc(x, w13, w2, y)
        assert st == 0, msg
        torch.cuda.synchronize()
        assert err_max(y, ref) <= TOL_BF16
        assert torch.equal(y, ref)            # same kernels, same order: identical bits
    # no failure recorded in the library's own error word (the one this call uses)
    from expert_gemm_layers_gb300 import device_status
    assert device_status(builtin=True)[0] == 0


@pytest.mark.parametrize("S", [4096, 2048 + 8])     # 64 MiB, and one shard row (8 rows) above 32 MiB
def test_noalloc_rejects_requests_beyond_its_scratch(S):
    d, ffn, W = 64, 8192, 8
    assert S * ffn * 2 > SCRATCH_BYTES
    x = torch.zeros((W, 1, S // W, d), dtype=torch.bfloat16, device=DEV)
    w13 = torch.zeros((W, 2 * ffn // W, d), dtype=torch.bfloat16, device=DEV)
    w2 = torch.zeros((d, ffn), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros_like(x)
    st, msg = _noalloc(x, w13, w2, y)
    assert _lib.STATUS_NAMES[st] == "DG_ERR_UNSUPPORTED"
    assert "scratch" in msg
