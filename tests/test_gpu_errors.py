"""The failure path on the GPU, without faulting it: a bounded wait that
nothing satisfies expires and records DG_ERR_TIMEOUT in the error block of
the workspace it was given; later kernels given that workspace skip their
work until the status is read, while calls with another workspace -- on
another stream -- are not affected."""
import pytest
import torch

import expert_gemm_layers_gb300 as dg
from expert_gemm_layers_gb300 import alloc_workspace, debug_wait_timeout, device_status, gemm_fp8, synth

pytestmark = pytest.mark.gpu
DG_ERR_TIMEOUT = 4
DEV = torch.device("cuda")


def test_bounded_wait_expires_and_reports():
    ws = alloc_workspace(256, DEV)
    assert device_status(workspace=ws)[0] == 0
    debug_wait_timeout(20_000, workspace=ws)       # 20 ms
    st, code = device_status(workspace=ws)
    assert st == DG_ERR_TIMEOUT
    assert code & 0xFF == 0x7F
    assert device_status(workspace=ws)[0] == 0     # read-and-clear


def test_kernels_skip_work_while_their_workspace_holds_an_error():
    A, B, C = synth.fp8_gemm_inputs(128, 256, 128, seed=3, device=DEV)
    D = torch.full((128, 256), 7.0, dtype=torch.bfloat16, device=DEV)
    ws = alloc_workspace(256, DEV)
    debug_wait_timeout(10_000, workspace=ws)
    gemm_fp8(A, B, C, 0.5, 1.0, out=D, ws=ws)
    torch.cuda.synchronize()
    assert torch.all(D == 7.0)                     # untouched: the kernel returned early
    assert device_status(workspace=ws)[0] == DG_ERR_TIMEOUT
    gemm_fp8(A, B, C, 0.5, 1.0, out=D, ws=ws)
    torch.cuda.synchronize()
    assert not torch.all(D == 7.0)
    assert device_status(workspace=ws)[0] == 0


def test_a_failure_on_one_stream_leaves_another_streams_calls_alone():
    A, B, C = synth.fp8_gemm_inputs(128, 256, 128, seed=4, device=DEV)
    ref = gemm_fp8(A, B, C, 0.5, 1.0)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ws1, ws2 = alloc_workspace(256, DEV), alloc_workspace(256, DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        debug_wait_timeout(20_000, workspace=ws1)
    D = torch.full((128, 256), 7.0, dtype=torch.bfloat16, device=DEV)
    with torch.cuda.stream(s2):
        gemm_fp8(A, B, C, 0.5, 1.0, out=D, ws=ws2)
    torch.cuda.synchronize()
    assert torch.equal(D, ref)                     # written although stream 1 holds a timeout
    with torch.cuda.stream(s2):
        assert device_status(workspace=ws2)[0] == 0
    with torch.cuda.stream(s1):
        assert device_status(workspace=ws1)[0] == DG_ERR_TIMEOUT
        assert device_status(workspace=ws1)[0] == 0


def test_streams_get_their_own_default_error_blocks():
    s1 = torch.cuda.Stream()
    with torch.cuda.stream(s1):
        b1 = dg.error_block(DEV)
    b0 = dg.error_block(DEV)
    assert b0.data_ptr() != b1.data_ptr()
    assert device_status(builtin=True)[0] == 0      # the library's own word: only the no-alloc call writes it
