"""The failure path on the GPU, without faulting it: a bounded wait that
nothing satisfies expires, records DG_ERR_TIMEOUT in the error word, and
the library's kernels then skip their work until the status is read."""
import pytest
import torch

from expert_gemm_layers_gb300 import debug_wait_timeout, device_status, gemm_fp8, synth

pytestmark = pytest.mark.gpu
DG_ERR_TIMEOUT = 4


def test_bounded_wait_expires_and_reports():
    assert device_status()[0] == 0
    debug_wait_timeout(20_000)                 # 20 ms
    st, code = device_status()
    assert st == DG_ERR_TIMEOUT
    assert code & 0xFF == 0x7F
    assert device_status()[0] == 0             # read-and-clear


def test_kernels_skip_work_while_error_is_pending():
    dev = torch.device("cuda")
    A, B, C = synth.fp8_gemm_inputs(128, 256, 128, seed=3, device=dev)
    D = torch.full((128, 256), 7.0, dtype=torch.bfloat16, device=dev)
    debug_wait_timeout(10_000)
    gemm_fp8(A, B, C, 0.5, 1.0, out=D)
    torch.cuda.synchronize()
    assert torch.all(D == 7.0)                 # untouched: the kernel returned early
    assert device_status()[0] == DG_ERR_TIMEOUT
    gemm_fp8(A, B, C, 0.5, 1.0, out=D)
    torch.cuda.synchronize()
    assert not torch.all(D == 7.0)
    assert device_status()[0] == 0
