"""Pins of the CPU oracle to facts outside itself.

Each test ties one oracle function to something it does not compute itself:
an independent library's conversion tables, the exchange example printed on
the A2A-FFN project page, closed forms, invariants, brute force on tiny
inputs written as plain scalar loops, finite differences, or torch float64
library routines (layer_norm, silu, autograd).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
from expert_gemm_layers_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# decoders: exhaustive against torch's own dtype conversions
# --------------------------------------------------------------------------

def test_bf16_decode_exhaustive():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_to_f64(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_exhaustive():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2                       # s.1111.111 only
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.nanmax(ours) == 448.0 and np.nanmin(ours) == -448.0


def test_e4m3_rounding_of_generator_saturates():
    x = torch.tensor([1000.0, -1000.0, 448.0, 0.0, 1.0 + 1.0 / 16])
    b = synth.bits(synth.to_e4m3(x))
    vals = O.e4m3_to_f64(b)
    assert list(vals[:4]) == [448.0, -448.0, 448.0, 0.0]
    assert vals[4] == 1.0                          # tie 1+1/16 rounds to even (1.0)


# --------------------------------------------------------------------------
# FP8 GEMM
# --------------------------------------------------------------------------

def _e4m3_bits(vals):
    return synth.bits(synth.to_e4m3(torch.tensor(vals, dtype=torch.float32)))


def test_gemm_fp8_identity_closed_form():
    # B = I (N = K), beta = 0  =>  D = alpha * A, exactly
    rng = np.random.default_rng(0)
    M, K = 37, 48
    A = _e4m3_bits(rng.standard_normal((M, K)))
    B = _e4m3_bits(np.eye(K))
    D = O.gemm_fp8(A, B, None, 0.5, 0.0)
    assert np.array_equal(D, 0.5 * O.e4m3_to_f64(A))


def test_gemm_fp8_alpha_zero_gives_beta_c():
    g = torch.Generator().manual_seed(3)
    A = _e4m3_bits(torch.randn(9, 32, generator=g).numpy())
    B = _e4m3_bits(torch.randn(11, 32, generator=g).numpy())
    C = synth.bits(torch.randn(9, 11, generator=g).to(torch.bfloat16))
    D = O.gemm_fp8(A, B, C, 0.0, 1.0)
    assert np.array_equal(D, O.bf16_to_f64(C))


def test_gemm_fp8_small_integers_exact():
    rng = np.random.default_rng(1)
    M, N, K = 5, 7, 64
    a = rng.integers(-2, 3, size=(M, K)).astype(np.float64)
    b = rng.integers(-2, 3, size=(N, K)).astype(np.float64)
    D = O.gemm_fp8(_e4m3_bits(a), _e4m3_bits(b), None, 1.0, 0.0)
    for i in range(M):
        for j in range(N):
            assert D[i, j] == sum(int(a[i, kk]) * int(b[j, kk]) for kk in range(K))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 9, 33), (33, 2, 16)])
def test_gemm_fp8_brute_force(M, N, K):
    g = torch.Generator().manual_seed(M * 100 + N * 10 + K)
    A = _e4m3_bits(torch.randn(M, K, generator=g).numpy())
    B = _e4m3_bits(torch.randn(N, K, generator=g).numpy())
    C = synth.bits(torch.randn(M, N, generator=g).to(torch.bfloat16))
    alpha, beta = 0.5, 1.0
    D = O.gemm_fp8(A, B, C, alpha, beta)
    a, b, c = O.e4m3_to_f64(A), O.e4m3_to_f64(B), O.bf16_to_f64(C)
    for i in range(M):
        for j in range(N):
            s = 0.0
            for kk in range(K):
                s += float(a[i, kk]) * float(b[j, kk])      # B row j, i.e. (A @ B^T)
            assert D[i, j] == pytest.approx(alpha * s + beta * float(c[i, j]), rel=1e-13, abs=1e-13)
    # row subset reproduces the full result
    rows = [M - 1, 0]
    assert np.array_equal(O.gemm_fp8(A, B, C, alpha, beta, rows=rows), D[rows])


# --------------------------------------------------------------------------
# A2A exchange
# --------------------------------------------------------------------------

def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals.setdefault(key, []).append([int(v) for v in rest])
    return vals


def test_exchange_example_from_page():
    g = _read_golden("a2a_exchange_P2_B1_T2_D1.txt")
    P, B, T, D = g["P"][0][0], g["B"][0][0], g["T"][0][0], g["D"][0][0]
    x = np.zeros((P, B, T, D), dtype=np.int64)
    for rank, *v in g["input"]:
        x[rank] = np.array(v).reshape(B, T, D)
    X = O.a2a_dispatch(x)
    assert X.shape == (P, P * B, T // P, D)
    for rank, *v in g["dispatched"]:
        assert X[rank].reshape(-1).tolist() == v
        assert X[rank].shape == (2, 1, 1)
    # identity local compute: combine reconstructs the rank inputs
    assert np.array_equal(O.a2a_combine(X, B), x)


@pytest.mark.parametrize("P,B,T,D", [(2, 4, 16, 3), (8, 3, 64, 2), (4, 1, 16, 1), (1, 5, 16, 2)])
def test_dispatch_combine_round_trip_and_index_maps(P, B, T, D):
    x = np.arange(P * B * T * D).reshape(P, B, T, D)
    X = O.a2a_dispatch(x)
    assert np.array_equal(O.a2a_combine(X, B), x)
    L = T // P
    flat = x.reshape(P * B * T, D)
    for r, n, l in itertools.product(range(P), range(P * B), range(L)):
        assert np.array_equal(X[r, n, l], flat[O.dispatch_source_row(P, B, T, r, n, l)])
    Y = X.reshape(P * P * B * L, D)
    out = O.a2a_combine(X, B)
    for s, b, t in itertools.product(range(P), range(B), range(T)):
        assert np.array_equal(out[s, b, t], Y[O.combine_source_row(P, B, T, s, b, t)])


def test_dispatch_matches_torch_chunk_cat():
    # A2A(x, split_dim=1, concat_dim=0) written with torch.chunk / torch.cat
    P, B, T, D = 4, 3, 16, 5
    x = torch.arange(P * B * T * D).reshape(P, B, T, D)
    recv = [torch.cat([torch.chunk(x[s], P, dim=1)[r] for s in range(P)], dim=0) for r in range(P)]
    assert np.array_equal(O.a2a_dispatch(x.numpy()), torch.stack(recv).numpy())


# --------------------------------------------------------------------------
# LayerNorm / silu
# --------------------------------------------------------------------------

def test_layer_norm_invariants():
    rng = np.random.default_rng(5)
    z = rng.standard_normal((6, 300)) * 3.0 + 2.0
    eps = 1e-5
    y = O.layer_norm(z, np.ones(300), np.zeros(300), eps)
    var = z.var(axis=1)
    assert np.allclose(y.mean(axis=1), 0.0, atol=1e-12)
    assert np.allclose(y.var(axis=1), var / (var + eps), rtol=1e-12)
    const = np.full((2, 64), 7.25)
    beta = rng.standard_normal(64)
    assert np.array_equal(O.layer_norm(const, rng.standard_normal(64), beta, eps), np.broadcast_to(beta, (2, 64)))


def test_layer_norm_and_silu_match_torch_float64():
    rng = np.random.default_rng(6)
    z = rng.standard_normal((5, 96))
    gam, bet = rng.standard_normal(96), rng.standard_normal(96)
    ref = F.layer_norm(torch.from_numpy(z), (96,), torch.from_numpy(gam), torch.from_numpy(bet), eps=1e-5)
    assert np.allclose(O.layer_norm(z, gam, bet, 1e-5), ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(O.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-15)
    assert O.silu(np.array([0.0]))[0] == 0.0


# --------------------------------------------------------------------------
# FFN forward
# --------------------------------------------------------------------------

def _ffn_bits(sh, seed=11, norm_affine="random"):
    t = synth.ffn_inputs(sh.P, sh.B, sh.T, sh.D, sh.k, seed=seed, norm_affine=norm_affine)
    return t, {k: synth.bits(v) for k, v in t.items()}


def test_ffn_closed_form_constant_halves():
    # w1 = 0 and constant b1 halves make U and G constant rows, so
    # LN_x(U) = beta_x and LN_g(G) = beta_g exactly; with beta_x = 1 and
    # beta_g = c:  Hl = silu(c) and Y[n] = silu(c) * colsum(wout) + bout.
    sh = O.FFNShape(2, 3, 4, 8, 2)
    t, b = _ffn_bits(sh)
    H = sh.H
    t["w1"].zero_()
    t["b1"][..., :H] = 0.75
    t["b1"][..., H:] = -1.5
    t["nx_b"].fill_(1.0)
    c = 0.625
    t["ng_b"].fill_(c)
    b = {k: synth.bits(v) for k, v in t.items()}
    out = O.ffn_forward(sh, b["inputs"], b)
    silu_c = c / (1.0 + math.exp(-c))
    wout = O.bf16_to_f64(b["wout"]).reshape(sh.P, sh.L, H, sh.D)
    bout = O.bf16_to_f64(b["bout"]).reshape(sh.P, sh.L, sh.D)
    for s, bb, tt in itertools.product(range(sh.P), range(sh.B), range(sh.T)):
        r, l = divmod(tt, sh.L)
        expect = silu_c * wout[r, l].sum(axis=0) + bout[r, l]
        assert np.allclose(out[s, bb, tt], expect, rtol=1e-13, atol=1e-13)


def test_ffn_forward_brute_force_scalar_loops():
    # tiny shape, every step written as plain scalar loops
    sh = O.FFNShape(2, 1, 2, 4, 1)     # H = 4, L = 1
    t, b = _ffn_bits(sh, seed=21)
    f = {k: O.bf16_to_f64(v) for k, v in b.items()}
    P, B, T, D, H, L = sh.P, sh.B, sh.T, sh.D, sh.H, sh.L
    x = f["inputs"].reshape(P, B, T, D)
    w1 = f["w1"].reshape(P, L, D, 2 * H)
    b1 = f["b1"].reshape(P, L, 2 * H)
    wo = f["wout"].reshape(P, L, H, D)
    bo = f["bout"].reshape(P, L, D)
    out = O.ffn_forward(sh, b["inputs"], b)
    for s in range(P):
        for bb in range(B):
            for tt in range(T):
                r, l = tt // L, tt % L
                xin = [float(v) for v in x[s, bb, tt]]
                z = [sum(xin[d] * w1[r, l, d, j] for d in range(D)) + b1[r, l, j] for j in range(2 * H)]

                def ln(v, gam, bet):
                    m = sum(v) / len(v)
                    var = sum((vi - m) ** 2 for vi in v) / len(v)
                    return [(vi - m) / math.sqrt(var + 1e-5) * gam[i] + bet[i] for i, vi in enumerate(v)]
                a = ln(z[:H], f["nx_w"].reshape(P, H)[r], f["nx_b"].reshape(P, H)[r])
                g = ln(z[H:], f["ng_w"].reshape(P, H)[r], f["ng_b"].reshape(P, H)[r])
                h = [a[i] * (g[i] / (1.0 + math.exp(-g[i]))) for i in range(H)]
                y = [sum(h[i] * wo[r, l, i, e] for i in range(H)) + bo[r, l, e] for e in range(D)]
                assert np.allclose(out[s, bb, tt], y, rtol=1e-12, atol=1e-12)


def _torch_ffn_forward(sh, f64):
    """Independent float64 formulation: torch.chunk A2A, bmm, F.layer_norm, F.silu."""
    P, B, T, D, H, L = sh.P, sh.B, sh.T, sh.D, sh.H, sh.L
    x = f64["inputs"].reshape(P, B, T, D)
    outs_local = []
    for r in range(P):
        Xr = torch.cat([torch.chunk(x[s], P, dim=1)[r] for s in range(P)], dim=0)     # [PB, L, D]
        Z = torch.bmm(Xr.transpose(0, 1), f64["w1"][r]) + f64["b1"][r][:, None, :]    # [L, PB, 2H]
        U, G = torch.chunk(Z, 2, dim=-1)
        a = F.layer_norm(U, (H,), f64["nx_w"][r], f64["nx_b"][r], eps=sh.eps)
        s_ = F.layer_norm(G, (H,), f64["ng_w"][r], f64["ng_b"][r], eps=sh.eps)
        Hl = a * F.silu(s_)
        Y = torch.bmm(Hl, f64["wout"][r]) + f64["bout"][r][:, None, :]              # [L, PB, D]
        outs_local.append(Y.transpose(0, 1))                                           # [PB, L, D]
    out = [torch.cat([torch.chunk(outs_local[r], P, dim=0)[s] for r in range(P)], dim=1) for s in range(P)]
    return torch.stack(out)


def _f64_tensors(sh, b, dY_bits=None):
    shapes = dict(inputs=(sh.P, sh.B, sh.T, sh.D), w1=(sh.P, sh.L, sh.D, 2 * sh.H),
                  b1=(sh.P, sh.L, 2 * sh.H), wout=(sh.P, sh.L, sh.H, sh.D), bout=(sh.P, sh.L, sh.D),
                  nx_w=(sh.P, sh.H), nx_b=(sh.P, sh.H), ng_w=(sh.P, sh.H), ng_b=(sh.P, sh.H))
    return {k: torch.from_numpy(O.bf16_to_f64(b[k]).reshape(s)) for k, s in shapes.items()}


@pytest.mark.parametrize("P,B,T,D,k", [(2, 4, 16, 16, 2), (4, 2, 16, 8, 3), (1, 3, 16, 8, 6)])
def test_ffn_forward_matches_torch_formulation(P, B, T, D, k):
    sh = O.FFNShape(P, B, T, D, k)
    _, b = _ffn_bits(sh, seed=P * 7 + k)
    ours = O.ffn_forward(sh, b["inputs"], b)
    ref = _torch_ffn_forward(sh, _f64_tensors(sh, b)).numpy()
    assert np.allclose(ours, ref, rtol=1e-11, atol=1e-11)
    rows = np.random.default_rng(0).choice(P * B * T, size=min(17, P * B * T), replace=False)
    sub = O.ffn_forward_rows(sh, b["inputs"], b, rows)
    assert np.allclose(sub, ours.reshape(-1, D)[rows], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# FFN backward
# --------------------------------------------------------------------------

def test_ffn_backward_finite_differences():
    sh = O.FFNShape(2, 1, 2, 4, 2)
    _, b = _ffn_bits(sh, seed=31)
    f = {k: v.numpy().copy() for k, v in _f64_tensors(sh, b).items()}
    rng = np.random.default_rng(2)
    dY = rng.standard_normal(f["inputs"].shape)

    def params(ff):
        return dict(w1=ff["w1"], b1=ff["b1"], wout=ff["wout"], bout=ff["bout"],
                    nxw=ff["nx_w"], nxb=ff["nx_b"], ngw=ff["ng_w"], ngb=ff["ng_b"])

    def loss(ff):
        return float((O.ffn_forward(sh, ff["inputs"], params(ff), decoded=True) * dY).sum())

    g = O.ffn_backward(sh, f["inputs"], params(f), dY, decoded=True)
    names = dict(inputs="d_inputs", w1="dw1", b1="db1", wout="dwout", bout="dbout",
                 nx_w="dnx_w", nx_b="dnx_b", ng_w="dng_w", ng_b="dng_b")
    h = 1e-6
    for key, gkey in names.items():
        flat = f[key].reshape(-1)
        ana = g[gkey].reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = loss(f)
            flat[i] = old - h
            lm = loss(f)
            flat[i] = old
            num = (lp - lm) / (2 * h)
            assert abs(num - ana[i]) <= 1e-6 * max(1.0, abs(num)), (key, i, num, ana[i])


def test_ffn_backward_matches_torch_autograd():
    sh = O.FFNShape(2, 3, 16, 8, 2)
    _, b = _ffn_bits(sh, seed=41)
    t = _f64_tensors(sh, b)
    for v in t.values():
        v.requires_grad_(True)
    dY = torch.randn(t["inputs"].shape, dtype=torch.float64, generator=torch.Generator().manual_seed(9))
    out = _torch_ffn_forward(sh, t)
    out.backward(dY)
    prm = dict(w1=t["w1"].detach().numpy(), b1=t["b1"].detach().numpy(), wout=t["wout"].detach().numpy(),
               bout=t["bout"].detach().numpy(), nxw=t["nx_w"].detach().numpy(), nxb=t["nx_b"].detach().numpy(),
               ngw=t["ng_w"].detach().numpy(), ngb=t["ng_b"].detach().numpy())
    g = O.ffn_backward(sh, t["inputs"].detach().numpy(), prm, dY.numpy(), decoded=True)
    pairs = dict(inputs="d_inputs", w1="dw1", b1="db1", wout="dwout", bout="dbout",
                 nx_w="dnx_w", nx_b="dnx_b", ng_w="dng_w", ng_b="dng_b")
    for key, gkey in pairs.items():
        assert np.allclose(g[gkey], t[key].grad.numpy(), rtol=1e-10, atol=1e-10), key


def test_ffn_backward_subset_functions_match_full():
    sh = O.FFNShape(2, 3, 16, 8, 2)
    _, b = _ffn_bits(sh, seed=51)
    dY = synth.bits(synth.ffn_grad_output(sh.P, sh.B, sh.T, sh.D, seed=52))
    full = O.ffn_backward(sh, b["inputs"], b, dY)
    rows = [0, 5, 77, sh.P * sh.B * sh.T - 1]
    dx = O.ffn_backward_dx_rows(sh, b["inputs"], b, dY, rows)
    assert np.allclose(dx, full["d_inputs"].reshape(-1, sh.D)[rows], rtol=1e-12, atol=1e-12)
    for t in (0, 13):
        o = O.ffn_backward_problem(sh, b["inputs"], b, dY, t)
        r, l = divmod(t, sh.L)
        for key in ("dw1", "db1", "dwout", "dbout"):
            assert np.allclose(o[key], full[key][r, l], rtol=1e-12, atol=1e-12), key
    nr = O.ffn_backward_norm_rank(sh, b["inputs"], b, dY, 1)
    for key in ("dnx_w", "dnx_b", "dng_w", "dng_b"):
        assert np.allclose(nr[key], full[key][1], rtol=1e-12, atol=1e-12), key


def test_ffn_norm_rank_helper_matches_full_backward():
    # the norm-only helper behind ffn_backward_norm_rank against the full backward of each problem
    sh = O.FFNShape(4, 2, 16, 8, 3)
    _, b = _ffn_bits(sh, seed=61)
    dY = synth.bits(synth.ffn_grad_output(sh.P, sh.B, sh.T, sh.D, seed=62))
    full = O.ffn_backward(sh, b["inputs"], b, dY)
    for r in (0, 3):
        nr = O.ffn_backward_norm_rank(sh, b["inputs"], b, dY, r)
        for key in ("dnx_w", "dnx_b", "dng_w", "dng_b"):
            assert np.allclose(nr[key], full[key][r], rtol=1e-12, atol=1e-12), key


# --------------------------------------------------------------------------
# comp_only (no exchange)
# --------------------------------------------------------------------------

def test_comp_only_is_the_layer_when_one_rank():
    # with P = 1 both exchanges are the identity, so both modes are the same map
    sh = O.FFNShape(1, 3, 8, 8, 2)
    _, b = _ffn_bits(sh, seed=71)
    dY = synth.bits(synth.ffn_grad_output(sh.P, sh.B, sh.T, sh.D, seed=72))
    assert np.array_equal(O.ffn_forward_comp_only(sh, b["inputs"], b), O.ffn_forward(sh, b["inputs"], b))
    g1, g2 = O.ffn_backward_comp_only(sh, b["inputs"], b, dY), O.ffn_backward(sh, b["inputs"], b, dY)
    for key in g2:
        assert np.array_equal(g1[key], g2[key]), key


def test_comp_only_closed_form_uses_own_rank_and_slice():
    # constant halves (as in the exchange closed form): output row (r, b, t) is
    # silu(c) * colsum(wout[r, t % L]) + bout[r, t % L] -- rank r's own problem
    sh = O.FFNShape(2, 3, 8, 8, 2)
    t, _ = _ffn_bits(sh, seed=73)
    H = sh.H
    t["w1"].zero_()
    t["b1"][..., :H] = 0.5
    t["b1"][..., H:] = 2.0
    t["nx_b"].fill_(1.0)
    c = -0.875
    t["ng_b"].fill_(c)
    b = {k: synth.bits(v) for k, v in t.items()}
    out = O.ffn_forward_comp_only(sh, b["inputs"], b)
    silu_c = c / (1.0 + math.exp(-c))
    wout = O.bf16_to_f64(b["wout"]).reshape(sh.P, sh.L, H, sh.D)
    bout = O.bf16_to_f64(b["bout"]).reshape(sh.P, sh.L, sh.D)
    for r, bb, tt in itertools.product(range(sh.P), range(sh.B), range(sh.T)):
        l = tt % sh.L
        expect = silu_c * wout[r, l].sum(axis=0) + bout[r, l]
        assert np.allclose(out[r, bb, tt], expect, rtol=1e-13, atol=1e-13)


def test_comp_only_forward_brute_force_scalar_loops():
    sh = O.FFNShape(2, 2, 4, 4, 1)     # H = 4, L = 2
    _, b = _ffn_bits(sh, seed=74)
    f = {k: O.bf16_to_f64(v) for k, v in b.items()}
    P, B, T, D, H, L = sh.P, sh.B, sh.T, sh.D, sh.H, sh.L
    x = f["inputs"].reshape(P, B, T, D)
    w1, b1 = f["w1"].reshape(P, L, D, 2 * H), f["b1"].reshape(P, L, 2 * H)
    wo, bo = f["wout"].reshape(P, L, H, D), f["bout"].reshape(P, L, D)
    out = O.ffn_forward_comp_only(sh, b["inputs"], b)
    for r in range(P):
        for bb in range(B):
            for tt in range(T):
                l = tt % L                       # slice of token tt = p*L + l in the [B, P, L, D] view
                xin = [float(v) for v in x[r, bb, tt]]
                z = [sum(xin[d] * w1[r, l, d, j] for d in range(D)) + b1[r, l, j] for j in range(2 * H)]

                def ln(v, gam, bet):
                    m = sum(v) / len(v)
                    var = sum((vi - m) ** 2 for vi in v) / len(v)
                    return [(vi - m) / math.sqrt(var + 1e-5) * gam[i] + bet[i] for i, vi in enumerate(v)]
                a = ln(z[:H], f["nx_w"].reshape(P, H)[r], f["nx_b"].reshape(P, H)[r])
                g = ln(z[H:], f["ng_w"].reshape(P, H)[r], f["ng_b"].reshape(P, H)[r])
                h = [a[i] * (g[i] / (1.0 + math.exp(-g[i]))) for i in range(H)]
                y = [sum(h[i] * wo[r, l, i, e] for i in range(H)) + bo[r, l, e] for e in range(D)]
                assert np.allclose(out[r, bb, tt], y, rtol=1e-12, atol=1e-12)


def _torch_ffn_comp_only(sh, f64):
    """Independent float64 formulation of comp_only: torch view/reshape, bmm, F.layer_norm, F.silu."""
    P, B, T, D, H, L = sh.P, sh.B, sh.T, sh.D, sh.H, sh.L
    outs = []
    for r in range(P):
        Xr = f64["inputs"][r].view(B, P, L, D).reshape(B * P, L, D)
        Z = torch.bmm(Xr.transpose(0, 1), f64["w1"][r]) + f64["b1"][r][:, None, :]
        U, G = torch.chunk(Z, 2, dim=-1)
        a = F.layer_norm(U, (H,), f64["nx_w"][r], f64["nx_b"][r], eps=sh.eps)
        s_ = F.layer_norm(G, (H,), f64["ng_w"][r], f64["ng_b"][r], eps=sh.eps)
        Y = torch.bmm(a * F.silu(s_), f64["wout"][r]) + f64["bout"][r][:, None, :]
        outs.append(Y.transpose(0, 1).reshape(B, P, L, D).reshape(B, T, D))
    return torch.stack(outs)


def test_comp_only_matches_torch_formulation_and_autograd():
    sh = O.FFNShape(4, 2, 16, 8, 2)
    _, b = _ffn_bits(sh, seed=75)
    t = _f64_tensors(sh, b)
    for v in t.values():
        v.requires_grad_(True)
    out = _torch_ffn_comp_only(sh, t)
    assert np.allclose(O.ffn_forward_comp_only(sh, b["inputs"], b), out.detach().numpy(), rtol=1e-11, atol=1e-11)
    dY = torch.randn(out.shape, dtype=torch.float64, generator=torch.Generator().manual_seed(76))
    out.backward(dY)
    prm = dict(w1=t["w1"].detach().numpy(), b1=t["b1"].detach().numpy(), wout=t["wout"].detach().numpy(),
               bout=t["bout"].detach().numpy(), nxw=t["nx_w"].detach().numpy(), nxb=t["nx_b"].detach().numpy(),
               ngw=t["ng_w"].detach().numpy(), ngb=t["ng_b"].detach().numpy())
    g = O.ffn_backward_comp_only(sh, t["inputs"].detach().numpy(), prm, dY.numpy(), decoded=True)
    pairs = dict(inputs="d_inputs", w1="dw1", b1="db1", wout="dwout", bout="dbout",
                 nx_w="dnx_w", nx_b="dnx_b", ng_w="dng_w", ng_b="dng_b")
    for key, gkey in pairs.items():
        assert np.allclose(g[gkey], t[key].grad.numpy(), rtol=1e-10, atol=1e-10), key


def test_comp_only_backward_finite_differences():
    sh = O.FFNShape(2, 1, 4, 4, 1)
    _, b = _ffn_bits(sh, seed=77)
    f = {k: v.numpy().copy() for k, v in _f64_tensors(sh, b).items()}
    dY = np.random.default_rng(78).standard_normal(f["inputs"].shape)

    def params(ff):
        return dict(w1=ff["w1"], b1=ff["b1"], wout=ff["wout"], bout=ff["bout"],
                    nxw=ff["nx_w"], nxb=ff["nx_b"], ngw=ff["ng_w"], ngb=ff["ng_b"])

    def loss(ff):
        return float((O.ffn_forward_comp_only(sh, ff["inputs"], params(ff), decoded=True) * dY).sum())

    g = O.ffn_backward_comp_only(sh, f["inputs"], params(f), dY, decoded=True)
    names = dict(inputs="d_inputs", w1="dw1", b1="db1", wout="dwout", bout="dbout",
                 nx_w="dnx_w", nx_b="dnx_b", ng_w="dng_w", ng_b="dng_b")
    h = 1e-6
    for key, gkey in names.items():
        flat = f[key].reshape(-1)
        ana = g[gkey].reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = loss(f)
            flat[i] = old - h
            lm = loss(f)
            flat[i] = old
            num = (lp - lm) / (2 * h)
            assert abs(num - ana[i]) <= 1e-6 * max(1.0, abs(num)), (key, i, num, ana[i])


# --------------------------------------------------------------------------
# TP SwiGLU
# --------------------------------------------------------------------------

def test_tp_swiglu_hand_computed():
    # W = 2 shards, F = 1 column each, d = 2, one token.  x = [1, 2].
    # shard 0: w1 row [1, 0], w3 row [0, 1]  -> a = 1, b = 2,  h = 2*silu(1)
    # shard 1: w1 row [0, 1], w3 row [1, 1]  -> a = 2, b = 3,  h = 3*silu(2)
    # w2 [d=2, ffn=2] = [[1, 0], [1, -1]] -> y = [h0, h0 - h1]
    x = np.array([[[[1.0, 2.0]]], [[[0.0, 0.0]]]])          # [W=2, bsz=1, S/W=1, d=2]
    w13 = np.array([[[1.0, 0.0], [0.0, 1.0]], [[0.0, 1.0], [1.0, 1.0]]])
    w2 = np.array([[1.0, 0.0], [1.0, -1.0]])
    y = O.tp_swiglu(x, w13, w2, W=2, decoded=True)
    s1 = 1.0 / (1.0 + math.exp(-1.0))
    s2 = 2.0 / (1.0 + math.exp(-2.0))
    h0, h1 = 2.0 * s1, 3.0 * s2
    assert y.shape == (2, 1, 1, 2)
    assert y[0, 0, 0, 0] == pytest.approx(h0, rel=1e-15)
    assert y[0, 0, 0, 1] == pytest.approx(h0 - h1, rel=1e-15)
    assert np.array_equal(y[1, 0, 0], [0.0, 0.0])            # silu(0) * 0 = 0


def test_tp_swiglu_shard_count_invariance_and_rows():
    # The same unsharded weights split over W = 1, 2, 4 shards give the same Y
    # (the shards partition the ffn columns; their partials sum to the product).
    rng = np.random.default_rng(8)
    d, ffn, S = 8, 16, 8
    w1 = rng.standard_normal((ffn, d)) / 3
    w3 = rng.standard_normal((ffn, d)) / 3
    w2 = rng.standard_normal((d, ffn)) / 4
    x_full = rng.standard_normal((S, d))
    ys = []
    for W in (1, 2, 4):
        F_ = ffn // W
        w13 = np.stack([np.concatenate([w1[s * F_:(s + 1) * F_], w3[s * F_:(s + 1) * F_]]) for s in range(W)])
        ys.append(O.tp_swiglu(x_full.reshape(W, 1, S // W, d), w13, w2, W=W, decoded=True).reshape(S, d))
    assert np.allclose(ys[0], ys[1], rtol=1e-12, atol=1e-12)
    assert np.allclose(ys[0], ys[2], rtol=1e-12, atol=1e-12)
    # unsharded textbook SwiGLU via torch float64 library ops
    ref = (F.silu(torch.from_numpy(x_full) @ torch.from_numpy(w1).T)
           * (torch.from_numpy(x_full) @ torch.from_numpy(w3).T)) @ torch.from_numpy(w2).T
    assert np.allclose(ys[0], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_tp_swiglu_batch_order_and_row_subset():
    x, w13, w2 = synth.tp_swiglu_inputs(32, 16, 24, 4, bsz=2, seed=3)
    xb, wb, w2b = synth.bits(x), synth.bits(w13), synth.bits(w2)
    y = O.tp_swiglu(xb, wb, w2b, W=4)
    assert y.shape == (4, 2, 8, 16)
    rows = [0, 9, 63]
    sub = O.tp_swiglu_rows(xb, wb, w2b, 4, rows)
    assert np.allclose(sub, y.reshape(-1, 16)[rows], rtol=1e-12, atol=1e-12)
    # every output row is the pair applied to the same row of the input
    one = O.tp_swiglu(xb[:, :1], wb, w2b, W=4)
    assert np.allclose(one[:, 0], y[:, 0], rtol=1e-12, atol=1e-12)


def test_oracle_is_not_imported_by_the_product_package():
    pkg = os.path.join(os.path.dirname(GOLDEN), "..", "expert_gemm_layers_gb300")
    for root, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                src = open(os.path.join(root, fn)).read()
                assert "import oracle" not in src and "from oracle" not in src, fn


# --------------------------------------------------------------------------
# TP SwiGLU backward
# --------------------------------------------------------------------------

def _tp_tiny(seed, W=2, bsz=1, sl=2, d=3, F=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((W, bsz, sl, d))
    w13 = rng.standard_normal((W, 2 * F, d)) / 2
    w2 = rng.standard_normal((d, W * F)) / 2
    dy = rng.standard_normal((W, bsz, sl, d))
    return x, w13, w2, dy


def test_tp_swiglu_backward_finite_differences():
    x, w13, w2, dy = _tp_tiny(3, bsz=2)
    g = O.tp_swiglu_backward(x, w13, w2, dy, W=2, decoded=True)

    def loss():
        return float((O.tp_swiglu(x, w13, w2, W=2, decoded=True) * dy).sum())
    h = 1e-6
    for arr, ga in ((x, g["dx"]), (w13, g["dw13"]), (w2, g["dw2"])):
        flat, gf = arr.reshape(-1), ga.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = loss()
            flat[i] = old - h
            lm = loss()
            flat[i] = old
            num = (lp - lm) / (2 * h)
            assert abs(num - gf[i]) <= 1e-6 * max(1.0, abs(num)), (i, num, gf[i])


def test_tp_swiglu_backward_matches_torch_autograd_and_subsets():
    W, Fs, d, S = 4, 6, 8, 16
    rng = np.random.default_rng(12)
    x = torch.from_numpy(rng.standard_normal((W, 1, S // W, d))).requires_grad_(True)
    w1 = torch.from_numpy(rng.standard_normal((W * Fs, d)) / 3).requires_grad_(True)
    w3 = torch.from_numpy(rng.standard_normal((W * Fs, d)) / 3).requires_grad_(True)
    w2 = torch.from_numpy(rng.standard_normal((d, W * Fs)) / 3).requires_grad_(True)
    dy = torch.from_numpy(rng.standard_normal((W, 1, S // W, d)))
    # textbook unsharded SwiGLU with torch library ops
    X = x.reshape(S, d)
    y = (F.silu(X @ w1.T) * (X @ w3.T)) @ w2.T
    y.reshape(W, 1, S // W, d).backward(dy)
    w13 = torch.stack([torch.cat([w1[s * Fs:(s + 1) * Fs], w3[s * Fs:(s + 1) * Fs]]) for s in range(W)])
    g = O.tp_swiglu_backward(x.detach().numpy(), w13.detach().numpy(), w2.detach().numpy(), dy.numpy(), W=W,
                             decoded=True)
    assert np.allclose(g["dx"], x.grad.numpy(), rtol=1e-10, atol=1e-10)
    assert np.allclose(g["dw2"], w2.grad.numpy(), rtol=1e-10, atol=1e-10)
    dw1 = np.concatenate([g["dw13"][s, :Fs] for s in range(W)])
    dw3 = np.concatenate([g["dw13"][s, Fs:] for s in range(W)])
    assert np.allclose(dw1, w1.grad.numpy(), rtol=1e-10, atol=1e-10)
    assert np.allclose(dw3, w3.grad.numpy(), rtol=1e-10, atol=1e-10)
    # bit-pattern subsets agree with the full result
    xb, w13b, w2b, dyb = (synth.bits(torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16))
                          for a in (x.detach().numpy(), w13.detach().numpy(), w2.detach().numpy(), dy.numpy()))
    full = O.tp_swiglu_backward(xb, w13b, w2b, dyb, W=W)
    rows = [0, 5, S - 1]
    assert np.allclose(O.tp_swiglu_backward_rows(xb, w13b, w2b, dyb, W, rows), full["dx"].reshape(-1, d)[rows],
                       rtol=1e-12, atol=1e-12)
    cols = [0, 7, W * Fs - 1]
    wc = O.tp_swiglu_backward_weight_cols(xb, w13b, w2b, dyb, W, cols)
    assert np.allclose(wc["dw2"], full["dw2"][:, cols], rtol=1e-12, atol=1e-12)
    for j, c in enumerate(cols):
        s_, cc = divmod(c, Fs)
        assert np.allclose(wc["dw1"][j], full["dw13"][s_, cc], rtol=1e-12, atol=1e-12)
        assert np.allclose(wc["dw3"][j], full["dw13"][s_, Fs + cc], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ attention projections

def test_allgather_linear_hand_computed():
    # W = 2 ranks, bsz = 1, one token each, in = 2, out = 2 (one feature per rank)
    x = np.array([[[[1.0, 2.0]]], [[[3.0, -1.0]]]])            # [W, bsz, S/W, in]
    w = np.array([[1.0, 1.0], [2.0, -1.0]])                    # [out, in]
    b = np.array([0.5, -0.5])
    y = O.allgather_linear(x, w, b, W=2, decoded=True)         # [W, rows, out/W]
    # gathered rows: (1, 2), (3, -1); rank 0 owns feature 0: x0+x1+0.5, rank 1 feature 1: 2x0-x1-0.5
    assert np.array_equal(y[0, :, 0], [3.5, 2.5])
    assert np.array_equal(y[1, :, 0], [-0.5, 6.5])


def test_linear_reduce_scatter_hand_computed():
    # rank 0 holds input feature 0, rank 1 feature 1, for both gathered rows
    a = np.array([[[1.0], [3.0]], [[2.0], [-1.0]]])            # [W, rows, in/W]
    w = np.array([[1.0, 1.0], [2.0, -1.0]])
    b = np.array([0.5, -0.5])
    y = O.linear_reduce_scatter(a, w, b, W=2, bsz=1, decoded=True)   # [W, bsz, S/W, out]
    assert np.array_equal(y[0, 0, 0], [3.5, -0.5])
    assert np.array_equal(y[1, 0, 0], [2.5, 6.5])


@pytest.mark.parametrize("W,bsz", [(1, 1), (2, 3), (4, 2)])
def test_attention_projections_match_unsharded_torch_linear(W, bsz):
    rng = np.random.default_rng(W * 10 + bsz)
    S, din, dout = 8, 16, 24
    x = rng.standard_normal((W, bsz, S // W, din))
    wq = rng.standard_normal((dout, din))
    bq = rng.standard_normal(dout)
    wo = rng.standard_normal((din, dout))
    bo = rng.standard_normal(din)
    # column-parallel: concatenating the ranks' feature blocks gives the unsharded linear
    # of the gathered rows (rank, seq_local, batch)
    X = torch.from_numpy(x).permute(0, 2, 1, 3).reshape(-1, din)
    ref = F.linear(X, torch.from_numpy(wq), torch.from_numpy(bq)).numpy()
    y = O.allgather_linear(x, wq, bq, W=W, decoded=True)
    assert np.allclose(np.concatenate(list(y), axis=1), ref, rtol=1e-12, atol=1e-12)
    # row-parallel on the column-parallel output: the unsharded composition, scattered back
    z = O.linear_reduce_scatter(y, wo, bo, W=W, bsz=bsz, decoded=True)
    ref2 = F.linear(torch.from_numpy(ref), torch.from_numpy(wo), torch.from_numpy(bo))
    ref2 = ref2.reshape(W, S // W, bsz, din).permute(0, 2, 1, 3).numpy()
    assert np.allclose(z, ref2, rtol=1e-11, atol=1e-11)


def test_attention_projection_backward_finite_differences():
    rng = np.random.default_rng(5)
    W, bsz, sl, din, dout = 2, 2, 2, 3, 4
    x = rng.standard_normal((W, bsz, sl, din))
    w = rng.standard_normal((dout, din))
    b = rng.standard_normal(dout)
    dy = rng.standard_normal((W, W * sl * bsz, dout // W))
    g = O.allgather_linear_backward(x, w, dy, W=W, decoded=True)

    def loss_col():
        return float((O.allgather_linear(x, w, b, W=W, decoded=True) * dy).sum())
    a = rng.standard_normal((W, W * sl * bsz, 2))              # 2 input features per rank
    wo = rng.standard_normal((dout, 2 * W))
    bo = rng.standard_normal(dout)
    dz = rng.standard_normal((W, bsz, sl, dout))
    g2 = O.linear_reduce_scatter_backward(a, wo, dz, W=W, decoded=True)

    def loss_row():
        return float((O.linear_reduce_scatter(a, wo, bo, W=W, bsz=bsz, decoded=True) * dz).sum())
    h = 1e-6
    for loss, pairs in ((loss_col, ((x, g["dx"]), (w, g["d_weight"]), (b, g["d_bias"]))),
                        (loss_row, ((a, g2["da"]), (wo, g2["d_weight"]), (bo, g2["d_bias"])))):
        for arr, ga in pairs:
            flat, gf = arr.reshape(-1), ga.reshape(-1)
            for i in range(flat.size):
                old = flat[i]
                flat[i] = old + h
                lp = loss()
                flat[i] = old - h
                lm = loss()
                flat[i] = old
                num = (lp - lm) / (2 * h)
                assert abs(num - gf[i]) <= 1e-6 * max(1.0, abs(num)), (i, num, gf[i])


def test_attention_projection_backward_matches_torch_autograd():
    rng = np.random.default_rng(9)
    W, bsz, S, din, dout = 4, 2, 8, 16, 12
    x = torch.from_numpy(rng.standard_normal((W, bsz, S // W, din))).requires_grad_(True)
    w = torch.from_numpy(rng.standard_normal((dout, din))).requires_grad_(True)
    b = torch.from_numpy(rng.standard_normal(dout)).requires_grad_(True)
    X = x.permute(0, 2, 1, 3).reshape(-1, din)
    y = F.linear(X, w, b)
    dy = torch.from_numpy(rng.standard_normal(y.shape))
    y.backward(dy)
    F_ = dout // W
    dy_ranks = np.stack([dy.numpy()[:, s * F_:(s + 1) * F_] for s in range(W)])
    g = O.allgather_linear_backward(x.detach().numpy(), w.detach().numpy(), dy_ranks, W=W, decoded=True)
    assert np.allclose(g["dx"], x.grad.numpy(), rtol=1e-11, atol=1e-11)
    assert np.allclose(g["d_weight"], w.grad.numpy(), rtol=1e-11, atol=1e-11)
    assert np.allclose(g["d_bias"], b.grad.numpy(), rtol=1e-11, atol=1e-11)
    # row-parallel: the input is the ranks' feature blocks of an unsharded activation
    A = torch.from_numpy(rng.standard_normal((W * S // W * bsz, din))).requires_grad_(True)
    wo = torch.from_numpy(rng.standard_normal((dout, din))).requires_grad_(True)
    bo = torch.from_numpy(rng.standard_normal(dout)).requires_grad_(True)
    z = F.linear(A, wo, bo)
    dz = torch.from_numpy(rng.standard_normal(z.shape))
    z.backward(dz)
    K = din // W
    a_ranks = np.stack([A.detach().numpy()[:, s * K:(s + 1) * K] for s in range(W)])
    dz_shards = dz.numpy().reshape(W, S // W, bsz, dout).transpose(0, 2, 1, 3)
    g2 = O.linear_reduce_scatter_backward(a_ranks, wo.detach().numpy(), dz_shards, W=W, decoded=True)
    assert np.allclose(np.concatenate(list(g2["da"]), axis=1), A.grad.numpy(), rtol=1e-11, atol=1e-11)
    assert np.allclose(g2["d_weight"], wo.grad.numpy(), rtol=1e-11, atol=1e-11)
    assert np.allclose(g2["d_bias"], bo.grad.numpy(), rtol=1e-11, atol=1e-11)


# ------------------------------------------------------------------ FP8 inside the FFN

def test_e4m3_rne_identity_ties_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7f, 0xff)], dtype=np.uint8)
    vals = O.e4m3_to_f64(codes)
    assert np.array_equal(O.e4m3_rne(vals), codes)                  # every value encodes to itself
    pos = O.e4m3_to_f64(np.arange(0, 0x7f, dtype=np.uint8))
    mid = (pos[:-1] + pos[1:]) / 2                                    # exact midpoints (binary)
    got = O.e4m3_rne(mid)
    lo, hi = np.arange(0, 0x7e), np.arange(1, 0x7f)
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, hi))         # ties to the even code
    assert np.array_equal(O.e4m3_rne(np.nextafter(mid, np.inf)), hi)  # just above: the upper value
    assert np.array_equal(O.e4m3_rne(np.nextafter(mid, -np.inf)), lo)
    assert list(O.e4m3_rne(np.array([449.0, 1e9, np.inf, -1e9, -np.inf]))) == [0x7e, 0x7e, 0x7e, 0xfe, 0xfe]


def test_e4m3_rne_matches_torch_cast():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_rne(x)
    same = (got == ref) | ((got & 0x7f) == 0) & ((ref & 0x7f) == 0)  # +-0 may differ in sign only
    assert same.all()


def test_quantize_e4m3_scales_and_error_bound():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((64, 300)) * np.exp(rng.uniform(-3, 3, (64, 1)))).astype(np.float32)
    x[5] = 0.0
    q, s = O.quantize_e4m3(x, axis=1)
    assert s[5] == 1.0 and not q[5].any()
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(s[np.arange(64) != 5], (amax / np.float32(448))[np.arange(64) != 5])
    # the largest magnitude of every row lands on +-448 (within the binary32 division)
    assert (np.abs(O.e4m3_to_f64(q)).max(axis=1)[np.arange(64) != 5] == 448).all()
    dq = O.e4m3_to_f64(q) * s.astype(np.float64)[:, None]
    bound = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s[:, None] + 1e-7 * np.abs(x)
    assert (np.abs(dq - x) <= bound).all()
    qc, sc = O.quantize_e4m3(x.T.copy(), axis=0)                      # per column of the transpose
    assert np.array_equal(qc, q.T) and np.array_equal(sc, s)


def test_ffn_forward_fp8_closed_form():
    # The constant-halves setup of the bf16 closed form: Hl = silu(c) on every row, so the
    # row's amax quantises it to 448 * scale exactly; wout chosen on the e4m3 grid times
    # 2^-6 with +-448 * 2^-6 in every column quantises exactly too, hence
    # Y[n] = silu(c) * colsum(wout) + bout as in the bf16 path.
    sh = O.FFNShape(2, 3, 4, 8, 2)
    t, b = _ffn_bits(sh)
    H = sh.H
    t["w1"].zero_()
    t["b1"][..., :H] = 0.75
    t["b1"][..., H:] = -1.5
    t["nx_b"].fill_(1.0)
    c = 0.625
    t["ng_b"].fill_(c)
    rng = np.random.default_rng(8)
    grid = O.e4m3_to_f64(rng.integers(0, 0x7f, size=t["wout"].shape).astype(np.uint8))
    grid = grid * rng.choice([-1.0, 1.0], size=grid.shape)
    grid[..., 0, :] = 448.0
    t["wout"] = torch.from_numpy(grid * 2.0 ** -6).to(torch.bfloat16)
    b = {k: synth.bits(v) for k, v in t.items()}
    out = O.ffn_forward_fp8(sh, b["inputs"], b)
    silu_c = c / (1.0 + math.exp(-c))
    hq, hs = O.quantize_e4m3(np.full((1, H), silu_c, dtype=np.float32), axis=1)
    silu_q = O.e4m3_to_f64(hq)[0, 0] * float(hs[0])                  # silu(c) after binary32 rounding
    wout = O.bf16_to_f64(b["wout"]).reshape(sh.P, sh.L, H, sh.D)
    bout = O.bf16_to_f64(b["bout"]).reshape(sh.P, sh.L, sh.D)
    for s, bb, tt in itertools.product(range(sh.P), range(sh.B), range(sh.T)):
        r, l = divmod(tt, sh.L)
        expect = silu_q * wout[r, l].sum(axis=0) + bout[r, l]
        assert np.allclose(out[s, bb, tt], expect, rtol=1e-13, atol=1e-13)


def test_ffn_forward_fp8_matches_torch_formulation():
    # independent restatement: torch float8 casts for the codes, torch float64 for the rest
    sh = O.FFNShape(2, 4, 8, 32, 2)
    t, b = _ffn_bits(sh, seed=21)
    P, B, T, D, H, L = sh.P, sh.B, sh.T, sh.D, sh.H, sh.L
    f64 = {k: torch.from_numpy(O.bf16_to_f64(v)) for k, v in b.items()}

    def q(x32, dim):
        # torch's float32 division on the CPU is not correctly rounded, so the
        # two quotients are taken in numpy binary32; torch casts to e4m3
        amax = x32.abs().amax(dim=dim, keepdim=True).numpy()
        nz = amax > 0
        a = np.where(nz, amax, np.float32(1)).astype(np.float32)
        s = torch.from_numpy(np.where(nz, a / np.float32(448), np.float32(1)).astype(np.float32))
        inv = torch.from_numpy(np.where(nz, np.float32(448) / a, np.float32(1)).astype(np.float32))
        codes = (x32 * inv).to(torch.float8_e4m3fn)
        return codes.to(torch.float64) * s.to(torch.float64)

    x = q(f64["inputs"].to(torch.float32).reshape(-1, D), 1).reshape(P, B, T, D)
    out = torch.zeros(P, B, T, D, dtype=torch.float64)
    w1 = f64["w1"].reshape(P, L, D, 2 * H)
    wo = f64["wout"].reshape(P, L, H, D)
    for r in range(P):
        for l in range(L):
            tt = r * L + l
            X = x[:, :, tt].reshape(P * B, D)
            Z = X @ q(w1[r, l].to(torch.float32), 0) + f64["b1"].reshape(P, L, -1)[r, l]
            a = F.layer_norm(Z[:, :H], (H,), f64["nx_w"].reshape(P, H)[r], f64["nx_b"].reshape(P, H)[r], sh.eps)
            g = F.layer_norm(Z[:, H:], (H,), f64["ng_w"].reshape(P, H)[r], f64["ng_b"].reshape(P, H)[r], sh.eps)
            Hl = a * F.silu(g)
            Y = q(Hl.to(torch.float32), 1) @ q(wo[r, l].to(torch.float32), 0) + f64["bout"].reshape(P, L, D)[r, l]
            out[:, :, tt] = Y.reshape(P, B, D)
    got = O.ffn_forward_fp8(sh, b["inputs"], b)
    assert np.allclose(got, out.numpy(), rtol=1e-10, atol=1e-10)
    # and the quantised layer stays within e4m3 precision of the exact one
    ref = O.ffn_forward(sh, b["inputs"], b)
    assert np.abs(got - ref).max() / np.abs(ref).max() < 0.15


def test_ffn_forward_fp8_rows_match_full():
    sh = O.FFNShape(2, 3, 8, 32, 3)
    t, b = _ffn_bits(sh, seed=22)
    full = O.ffn_forward_fp8(sh, b["inputs"], b).reshape(-1, sh.D)
    rows = np.array([0, 5, 17, 18, 31, sh.P * sh.B * sh.T - 1])
    assert np.allclose(O.ffn_forward_fp8_rows(sh, b["inputs"], b, rows), full[rows], rtol=1e-13, atol=1e-13)
