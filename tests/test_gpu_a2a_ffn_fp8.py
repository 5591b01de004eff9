"""A2A FFN forward with e4m3 GEMMs: libdg against the fp64 oracle of the same
quantised layer (per-row activation scales, per-column weight scales).

The e4m3 codes and scales of the weights and of the input rows are compared bit
for bit (both sides take the code decision in binary32); the layer output within
the FP8 tolerance."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from expert_gemm_layers_gb300 import (FFN_PARAM_NAMES, _lib, a2a_ffn_forward_fp8, a2a_ffn_fp8_pack_weights,
                                      synth)
from _compare import TOL_FP8, assert_close, err_max

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")

SHAPES = [
    (2, 4, 16, 128, 2),     # the tiny workload (H=256)
    (2, 3, 4, 144, 3),      # ragged: D=144, H=432, 2H=864 (N % 256 != 0), K % 128 != 0
    (4, 40, 16, 64, 2),     # M=160 rows: two row tiles, the second ragged
    (1, 5, 16, 128, 6),     # one rank
    (2, 2, 4, 1024, 8),     # H=8192, the widest e4m3 Hl row
]


def _inputs(P, B, T, D, k, seed):
    t = synth.ffn_inputs(P, B, T, D, k, seed=seed, device=DEV, norm_affine="random")
    return t["inputs"], {n: t[n] for n in FFN_PARAM_NAMES}


def _round256(n):
    return (n + 255) // 256 * 256


def test_packed_weights_bit_exact():
    P, B, T, D, k = 2, 3, 4, 144, 3
    H, L = D * k, T // P
    x, params = _inputs(P, B, T, D, k, seed=31)
    packed = a2a_ffn_fp8_pack_weights(params, P, B, T, D)
    torch.cuda.synchronize()
    pk = packed.cpu().numpy()
    w1 = O.bf16_to_f64(synth.bits(params["w1"])).reshape(T, D, 2 * H)
    wo = O.bf16_to_f64(synth.bits(params["wout"])).reshape(T, H, D)
    off_s1 = _round256(T * 2 * H * D)
    off_woq = _round256(off_s1 + T * 2 * H * 4)
    off_so = _round256(off_woq + T * D * H)
    w1q = pk[:T * 2 * H * D].reshape(T, 2 * H, D)
    s1 = pk[off_s1:off_s1 + T * 2 * H * 4].view(np.float32).reshape(T, 2 * H)
    woq = pk[off_woq:off_woq + T * D * H].reshape(T, D, H)
    so = pk[off_so:off_so + T * D * 4].view(np.float32).reshape(T, D)
    for t in range(T):
        q, s = O.quantize_e4m3(w1[t], axis=0)            # per column of [D, 2H]
        assert np.array_equal(w1q[t], q.T) and np.array_equal(s1[t], s), t
        q, s = O.quantize_e4m3(wo[t], axis=0)            # per column of [H, D]
        assert np.array_equal(woq[t], q.T) and np.array_equal(so[t], s), t


def test_input_codes_bit_exact():
    P, B, T, D, k = 2, 3, 4, 144, 3
    M = P * B
    x, params = _inputs(P, B, T, D, k, seed=32)
    packed = a2a_ffn_fp8_pack_weights(params, P, B, T, D)
    lib = _lib.load()
    nbytes = lib.dg_a2a_ffn_fp8_workspace_bytes(ctypes.byref(_lib.FFNShape(P, B, T, D, k, 1e-5)))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    a2a_ffn_forward_fp8(x, params, packed, workspace=ws)
    torch.cuda.synchronize()
    w = ws.cpu().numpy()[256:]          # past the error block
    rows = P * B * T
    q, s = O.quantize_e4m3(O.bf16_to_f64(synth.bits(x)).reshape(rows, D), axis=1)
    assert np.array_equal(w[:rows * D].reshape(rows, D), q)
    off = _round256(rows * D)
    got_s = w[off:off + rows * 4].view(np.float32).reshape(T, M)
    # oracle rows are input rows (s, b, t); the library keeps the scale at t*M + s*B + b
    assert np.array_equal(got_s, s.reshape(M, T).T)


@pytest.mark.parametrize("P,B,T,D,k", SHAPES)
def test_forward_small_full(P, B, T, D, k):
    x, params = _inputs(P, B, T, D, k, seed=33 + D)
    packed = a2a_ffn_fp8_pack_weights(params, P, B, T, D)
    out = a2a_ffn_forward_fp8(x, params, packed)
    torch.cuda.synchronize()
    xb, pb = synth.bits(x), {n: synth.bits(v) for n, v in params.items()}
    sh = O.FFNShape(P, B, T, D, k)
    assert_close(out, O.ffn_forward_fp8(sh, xb, pb), TOL_FP8, f"fp8 forward {P,B,T,D,k}")
    # against the exact (unquantised) layer: e4m3 precision
    assert err_max(out, O.ffn_forward(sh, xb, pb)) < 0.15


def test_forward_full_size_rows():
    # P=8, B=512, T=64, D=1280, k=6: 64 seeded rows of each of 4 seeded token positions
    P, B, T, D, k = 8, 512, 64, 1280, 6
    x, params = _inputs(P, B, T, D, k, seed=42)
    packed = a2a_ffn_fp8_pack_weights(params, P, B, T, D)
    out = a2a_ffn_forward_fp8(x, params, packed)
    torch.cuda.synchronize()
    rng = np.random.default_rng(44)
    ts = rng.choice(T, size=4, replace=False)
    sbs = [rng.choice(P * B, size=64, replace=False) for _ in ts]
    rows = np.concatenate([sb * T + t for t, sb in zip(ts, sbs)])       # flat (s*B + b)*T + t
    xb, pb = synth.bits(x), {n: synth.bits(v) for n, v in params.items()}
    ref = O.ffn_forward_fp8_rows(O.FFNShape(P, B, T, D, k), xb, pb, rows)
    got = out.reshape(-1, D)[torch.from_numpy(rows).to(DEV)]
    assert_close(got, ref, TOL_FP8, "fp8 forward full size (256 rows)")


def test_forward_fp8_close_to_bf16_path():
    from expert_gemm_layers_gb300 import a2a_ffn_forward
    P, B, T, D, k = 2, 4, 16, 128, 2
    x, params = _inputs(P, B, T, D, k, seed=34)
    packed = a2a_ffn_fp8_pack_weights(params, P, B, T, D)
    out8 = a2a_ffn_forward_fp8(x, params, packed)
    out16, _ = a2a_ffn_forward(x, params)
    torch.cuda.synchronize()
    assert err_max(out8, out16) < 0.15
