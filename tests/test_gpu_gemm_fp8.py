"""FP8 GEMM parity: libdg's tcgen05 kernel against the fp64 oracle.

Closed forms are compared bit for bit; random inputs within the FP8
tolerance (5e-2 normwise max-relative), plus a tighter check that the error
stays at the level of one bf16 rounding.
"""
import numpy as np
import pytest
import torch

import oracle as O
from expert_gemm_layers_gb300 import gemm_fp8, synth
from _compare import TOL_FP8, assert_close, err_max, to_f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _run(A, B, C, alpha, beta):
    dev = torch.device("cuda")
    D = gemm_fp8(A.to(dev), B.to(dev), None if C is None else C.to(dev), alpha, beta)
    torch.cuda.synchronize()
    return D.cpu()


def test_identity_closed_form_bit_exact():
    # B = I, beta = 0: D = bf16(0.5 * A) exactly (half of an e4m3 value is a bf16 value)
    M, K = 300, 256
    A, _, _ = synth.fp8_gemm_inputs(M, K, K, seed=5)
    B = synth.to_e4m3(torch.eye(K))
    D = _run(A, B, None, 0.5, 0.0)
    expect = 0.5 * O.e4m3_to_f64(synth.bits(A))
    assert np.array_equal(to_f64(D), expect)


def test_alpha_zero_gives_c_bit_exact():
    A, B, C = synth.fp8_gemm_inputs(130, 264, 64, seed=6)
    D = _run(A, B, C, 0.0, 1.0)
    assert np.array_equal(to_f64(D), O.bf16_to_f64(synth.bits(C)))


def test_k_zero_gives_beta_c():
    C = torch.randn(64, 32, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    A = torch.empty((64, 0), dtype=torch.float8_e4m3fn)
    B = torch.empty((32, 0), dtype=torch.float8_e4m3fn)
    D = _run(A, B, C, 0.5, 1.0)
    assert np.array_equal(to_f64(D), O.bf16_to_f64(synth.bits(C)))


def test_small_integers_exact():
    g = torch.Generator().manual_seed(2)
    M, N, K = 256, 512, 384
    A = synth.to_e4m3(torch.randint(-2, 3, (M, K), generator=g).float())
    B = synth.to_e4m3(torch.randint(-2, 3, (N, K), generator=g).float())
    D = _run(A, B, None, 1.0, 0.0)
    ref = O.gemm_fp8(synth.bits(A), synth.bits(B), None, 1.0, 0.0)
    # integer sums (|s| <= 1536) are exact in fp32; the one rounding is RNE to bf16,
    # which torch's own conversion of the exact value reproduces
    expect = torch.from_numpy(ref).to(torch.bfloat16)
    assert torch.equal(D, expect)


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 128),      # one tile
    (1, 8, 16),           # degenerate
    (257, 520, 80),       # ragged M, N and K (K not a multiple of the 128-wide K block)
    (640, 768, 1024),     # several tiles per CTA
    (96, 4096, 512),      # wide
])
def test_random_parity(M, N, K):
    A, B, C = synth.fp8_gemm_inputs(M, N, K, seed=M + N + K)
    D = _run(A, B, C, 0.5, 1.0)
    ref = O.gemm_fp8(synth.bits(A), synth.bits(B), synth.bits(C), 0.5, 1.0)
    e = assert_close(D, ref, TOL_FP8, f"gemm_fp8 {M}x{N}x{K}")
    assert e < 1e-2          # one bf16 rounding of the result dominates


def test_no_c_path_alpha_only():
    A, B, _ = synth.fp8_gemm_inputs(200, 136, 256, seed=9, with_c=False)
    D = _run(A, B, None, 0.25, 0.0)
    ref = O.gemm_fp8(synth.bits(A), synth.bits(B), None, 0.25, 0.0)
    assert_close(D, ref, TOL_FP8, "gemm_fp8 no C")


def test_full_size_4096():
    # the FP8 GEMM workload at its full size, all 16.8M outputs compared
    M = N = K = 4096
    dev = torch.device("cuda")
    A, B, C = synth.fp8_gemm_inputs(M, N, K, seed=1, device=dev)
    D = gemm_fp8(A, B, C, 0.5, 1.0)
    torch.cuda.synchronize()
    ref = O.gemm_fp8(synth.bits(A), synth.bits(B), synth.bits(C), 0.5, 1.0)
    e = assert_close(D, ref, TOL_FP8, "gemm_fp8 4096^3")
    assert e < 1e-2


def test_deterministic_reruns():
    A, B, C = synth.fp8_gemm_inputs(384, 512, 512, seed=11)
    d1, d2 = _run(A, B, C, 0.5, 1.0), _run(A, B, C, 0.5, 1.0)
    assert torch.equal(d1, d2)


def test_tile_widths_both_run():
    # Small problems take 224-column tiles; at 19456 x 4864 (76 x 19 tiles of
    # 256 columns) the 256-column tiles need fewer column steps per CTA pair.
    from expert_gemm_layers_gb300 import trace_begin, trace_end
    names = []
    for M, N, K in [(512, 1024, 256), (19456, 4864, 128)]:
        A, B, C = synth.fp8_gemm_inputs(M, N, K, seed=M + K, device=DEV)
        trace_begin()
        D = gemm_fp8(A, B, C, 0.5, 1.0)
        torch.cuda.synchronize()
        names += [e["name"] for e in trace_end()]
        rows = np.random.default_rng(M).choice(M, size=48, replace=False)
        ref = O.gemm_fp8(synth.bits(A), synth.bits(B), synth.bits(C), 0.5, 1.0, rows=rows)
        assert_close(D[torch.from_numpy(rows).to(DEV)], ref, TOL_FP8, f"gemm_fp8 {M}x{N}x{K}")
    assert names == ["gemm_fp8_n224", "gemm_fp8"], names
