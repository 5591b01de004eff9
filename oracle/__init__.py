"""Plain fp64 CPU oracle for the dg hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and ``--impl reference`` arm) may call it.  It shares no
code, table or constant with the CUDA library under
``expert_gemm_layers_gb300/``.

Every function works on numpy float64 after an exact decode of the stored bit
patterns (bf16 as uint16, e4m3 as uint8).  Nothing is rounded in between: Z,
Hl, a/b/h and all partial sums stay fp64.  numpy's float64 ``matmul`` is the
only library primitive used for the contractions; no step is blocked, fused
or reordered beyond what the definitions below state.

Sources (web pages, cited by title and section):

* "Pytorch Op for blackwell distributed gemm" (pytorch-distributed-gemm
  README), sections "Usage" and "Limitations & Important Notes": the FP8 GEMM
  ``alpha * (A @ B^T) + beta * C`` with A [M,K], row-major B [N,K], C [M,N],
  elements ``cutlass::float_e4m3_t``.
* The A2A-FFN project statement (problems/p04), sections "Interface, layout,
  and parameters" and "Computation and communication example": the
  dispatch / GEMM1 / LayerNorm-gate / GEMM2 / combine layer and its exchange
  example; "Cross-node tests and correctness" for the gradient check.
* "Add dist GEMM attention and FFN backend" (torchtitan PR #4044), sections
  "Structure" and "Row ordering": the SwiGLU column/row-parallel pair, the
  attention projections (column-parallel AllGatherLinear, row-parallel
  LinearReduceScatter) and the (rank, batch, seq_local) order of gathered rows.

Readings where the pages are silent are listed in the module docstrings of the
functions concerned (U = first half of Z, biased variance, silu(x) = x*sigmoid(x),
one [H] LayerNorm weight/bias pair per rank shared by its L slices).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(exhaustive decode tables, the exchange example, closed forms, LayerNorm
invariants, finite differences and brute force).  None is "parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = [
    "bf16_to_f64", "e4m3_to_f64", "gemm_fp8",
    "a2a_dispatch", "a2a_combine", "dispatch_source_row", "combine_source_row",
    "layer_norm", "silu", "FFNShape", "ffn_forward", "ffn_forward_rows",
    "ffn_problem_backward", "ffn_backward", "ffn_backward_dx_rows",
    "ffn_backward_problem", "ffn_backward_norm_rank", "ffn_forward_comp_only", "ffn_backward_comp_only",
    "tp_swiglu", "tp_swiglu_rows", "tp_swiglu_backward", "tp_swiglu_backward_rows",
    "tp_swiglu_backward_weight_cols",
]


# ---------------------------------------------------------------------------
# Exact decoders of the stored bit patterns
# ---------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly.

    bf16 is the upper half of an IEEE binary32, so the value is the float32
    whose high 16 bits are the pattern; float32 -> float64 is exact.
    """
    b = np.ascontiguousarray(bits).view(np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _e4m3_value(code: int) -> float:
    """Value of one OCP E4M3FN code (the element type cutlass::float_e4m3_t).

    Layout s.eeee.mmm, exponent bias 7, subnormals at exponent field 0, no
    infinities, the two codes s.1111.111 are NaN, largest finite 448.
    """
    s = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_to_f64(bits) -> np.ndarray:
    """e4m3 bit patterns (uint8) -> float64, exactly (table of the 256 codes)."""
    b = np.ascontiguousarray(bits).view(np.uint8)
    return _E4M3_TABLE[b]


# ---------------------------------------------------------------------------
# (a) FP8 GEMM  D = alpha * (A @ B^T) + beta * C
# ---------------------------------------------------------------------------

def gemm_fp8(A_bits, B_bits, C_bits, alpha: float, beta: float, rows=None) -> np.ndarray:
    """D = alpha * (A @ B^T) + beta * C in fp64.

    A: e4m3 [M, K]; B: e4m3 [N, K] row-major (the transposed operand of
    torch.matmul); C: bf16 [M, N] or None when beta == 0.  ``rows`` selects a
    subset of output rows (each output row depends only on its row of A and C).
    Returns float64 [len(rows), N] (or [M, N]).
    """
    A = np.asarray(A_bits)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        A = A[rows]
    a = e4m3_to_f64(A)
    b = e4m3_to_f64(np.asarray(B_bits))
    acc = a @ b.T
    out = float(alpha) * acc
    if beta != 0.0:
        C = np.asarray(C_bits)
        if rows is not None:
            C = C[rows]
        out = out + float(beta) * bf16_to_f64(C)
    return out


# ---------------------------------------------------------------------------
# (b) All-to-all expert-parallel FFN layer
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class FFNShape:
    """P ranks, local batch B, T tokens, model dim D, expansion k (H = D*k, L = T/P)."""
    P: int
    B: int
    T: int
    D: int
    k: int
    eps: float = 1e-5

    @property
    def H(self) -> int:
        return self.D * self.k

    @property
    def L(self) -> int:
        if self.T % self.P:
            raise ValueError("T must be divisible by P")
        return self.T // self.P

    @property
    def M(self) -> int:
        return self.P * self.B


def a2a_dispatch(x: np.ndarray) -> np.ndarray:
    """Dispatch ``A2A(inputs, split_dim=1, concat_dim=0)`` over all ranks at once.

    x: [P (source rank s), B, T, ...].  Every source rank splits its token axis
    into P slices of L tokens; rank r receives slice r of every source and
    concatenates them along the batch axis in source-rank order, so
    result[r] = concat_s x[s][:, r*L:(r+1)*L]  -> [P, P*B, L, ...].
    Works on any dtype, so it also moves bit patterns unchanged.
    """
    P, B, T = x.shape[0], x.shape[1], x.shape[2]
    L = T // P
    return np.stack([
        np.concatenate([x[s][:, r * L:(r + 1) * L] for s in range(P)], axis=0)
        for r in range(P)
    ])


def a2a_combine(y: np.ndarray, B: int) -> np.ndarray:
    """Combine ``A2A(Ylocal, split_dim=0, concat_dim=1)``: the inverse exchange.

    y: [P (rank r), P*B, L, ...].  Rank r splits its rows into P chunks of B
    (chunk s belongs to source rank s); rank s concatenates the chunks it gets
    from r = 0..P-1 along the token axis -> result[s] = [B, P*L, ...].
    """
    P = y.shape[0]
    return np.stack([
        np.concatenate([y[r][s * B:(s + 1) * B] for r in range(P)], axis=1)
        for s in range(P)
    ])


def dispatch_source_row(P: int, B: int, T: int, r: int, n: int, l: int) -> int:
    """Flat row index into inputs [P,B,T] that dispatch sends to Xlocal[r][n, l]."""
    L = T // P
    s, b = divmod(n, B)
    return (s * B + b) * T + r * L + l


def combine_source_row(P: int, B: int, T: int, s: int, b: int, t: int) -> int:
    """Flat row index into Ylocal [P, P*B, L] that combine sends to output[s][b, t]."""
    L = T // P
    r, l = divmod(t, L)
    return (r * (P * B) + s * B + b) * L + l


def layer_norm(z: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float) -> np.ndarray:
    """LN(z) = ((z - mean(z)) / sqrt(mean((z - mean(z))^2) + eps)) * gamma + beta.

    Over the last axis; biased variance; eps inside the square root.
    """
    mu = z.mean(axis=-1, keepdims=True)
    c = z - mu
    var = (c * c).mean(axis=-1, keepdims=True)
    return c / np.sqrt(var + eps) * gamma + beta


def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x * sigmoid(x) = x / (1 + exp(-x)) (not defined on the pages)."""
    return x / (1.0 + np.exp(-x))


def _ffn_problem_forward(X, w1, b1, wout, bout, nxw, nxb, ngw, ngb, eps, H):
    """One (rank, slice) problem: rows X [n, D] -> (Z, Hl, Y) in fp64."""
    Z = X @ w1 + b1
    U, G = Z[:, :H], Z[:, H:]
    Hl = layer_norm(U, nxw, nxb, eps) * silu(layer_norm(G, ngw, ngb, eps))
    Y = Hl @ wout + bout
    return Z, Hl, Y


def _decode_ffn_params(sh: FFNShape, prm: dict) -> dict:
    P, L, D, H = sh.P, sh.L, sh.D, sh.H
    f = bf16_to_f64
    return dict(
        w1=f(prm["w1"]).reshape(P, L, D, 2 * H),
        b1=f(prm["b1"]).reshape(P, L, 2 * H),
        wout=f(prm["wout"]).reshape(P, L, H, D),
        bout=f(prm["bout"]).reshape(P, L, D),
        nxw=f(prm["nx_w"]).reshape(P, H), nxb=f(prm["nx_b"]).reshape(P, H),
        ngw=f(prm["ng_w"]).reshape(P, H), ngb=f(prm["ng_b"]).reshape(P, H),
    )


def ffn_forward(sh: FFNShape, inputs, prm: dict, intermediates: bool = False,
                decoded: bool = False):
    """The whole layer for all ranks, in the page's order (dense_v2 + bmm path).

    inputs: bf16 bits [P, B, T, D] (or float64 when ``decoded``); prm holds
    bf16 bits of w1 [P,L,D,2H], b1 [P,L,2H], wout [P,L,H,D], bout [P,L,D],
    nx_w/nx_b/ng_w/ng_b [P,H].  Steps: Xlocal = dispatch(inputs);
    Z[n,l] = Xlocal[n,l] @ w1[l] + b1[l]; (U, G) = halves of Z;
    Hl = LN_x(U) * silu(LN_gate(G)); Ylocal[n,l] = Hl[n,l] @ wout[l] + bout[l];
    output = combine(Ylocal).  Returns float64 output [P,B,T,D] (and Z, Hl
    as [P, P*B, L, *] when ``intermediates``).
    """
    P, B, L, D, H = sh.P, sh.B, sh.L, sh.D, sh.H
    x = np.asarray(inputs, dtype=np.float64) if decoded else bf16_to_f64(inputs)
    x = x.reshape(P, B, sh.T, D)
    p = prm if decoded else _decode_ffn_params(sh, prm)
    X = a2a_dispatch(x)                                  # [P, P*B, L, D]
    Y = np.empty((P, P * B, L, D))
    Zs = np.empty((P, P * B, L, 2 * H)) if intermediates else None
    Hs = np.empty((P, P * B, L, H)) if intermediates else None
    for r in range(P):
        for l in range(L):
            Z, Hl, Yl = _ffn_problem_forward(
                X[r, :, l, :], p["w1"][r, l], p["b1"][r, l], p["wout"][r, l], p["bout"][r, l],
                p["nxw"][r], p["nxb"][r], p["ngw"][r], p["ngb"][r], sh.eps, H)
            Y[r, :, l, :] = Yl
            if intermediates:
                Zs[r, :, l, :] = Z
                Hs[r, :, l, :] = Hl
    out = a2a_combine(Y, B)                              # [P, B, T, D]
    if intermediates:
        return out, Zs, Hs
    return out


def ffn_forward_rows(sh: FFNShape, inputs_bits, prm: dict, out_rows) -> np.ndarray:
    """Selected rows of the layer's output, each computed exactly as ffn_forward does.

    out_rows: flat indices into output [P,B,T] (row (s,b,t) -> (s*B+b)*T+t).
    Each output row (s,b,t) is Ylocal[r][n,l] with r,l = divmod(t, L) and
    n = s*B+b (combine), whose input row is inputs[s][b, r*L+l] (dispatch);
    rows sharing a problem (r,l) are batched through the same weights.
    Returns float64 [len(out_rows), D].
    """
    P, B, T, L, D, H = sh.P, sh.B, sh.T, sh.L, sh.D, sh.H
    out_rows = np.asarray(out_rows, dtype=np.int64)
    x_all = np.asarray(inputs_bits).reshape(P * B * T, D)
    w1 = np.asarray(prm["w1"]).reshape(P, L, D, 2 * H)
    b1 = np.asarray(prm["b1"]).reshape(P, L, 2 * H)
    wout = np.asarray(prm["wout"]).reshape(P, L, H, D)
    bout = np.asarray(prm["bout"]).reshape(P, L, D)
    nxw = bf16_to_f64(prm["nx_w"]).reshape(P, H)
    nxb = bf16_to_f64(prm["nx_b"]).reshape(P, H)
    ngw = bf16_to_f64(prm["ng_w"]).reshape(P, H)
    ngb = bf16_to_f64(prm["ng_b"]).reshape(P, H)
    result = np.empty((len(out_rows), D))
    sbt = np.stack(np.unravel_index(out_rows, (P, B, T)), axis=1)
    problems = {}
    for i, (s, b, t) in enumerate(sbt):
        r, l = divmod(int(t), L)
        problems.setdefault((r, l), []).append((i, int(s) * B + int(b)))
    for (r, l), items in problems.items():
        idx = np.array([i for i, _ in items])
        src = [dispatch_source_row(P, B, T, r, n, l) for _, n in items]
        X = bf16_to_f64(x_all[src])
        _, _, Yl = _ffn_problem_forward(
            X, bf16_to_f64(w1[r, l]), bf16_to_f64(b1[r, l]), bf16_to_f64(wout[r, l]),
            bf16_to_f64(bout[r, l]), nxw[r], nxb[r], ngw[r], ngb[r], sh.eps, H)
        result[idx] = Yl
    return result


def _layer_norm_backward(dy_hat_aff, z, gamma, eps):
    """Gradient of LN w.r.t. its input z, given dL/d(LN output).

    With c = z - mean, rstd = 1/sqrt(mean(c^2)+eps), xhat = c*rstd and
    dxhat = dL/dy * gamma:  dz = rstd * (dxhat - mean(dxhat) - xhat*mean(dxhat*xhat)).
    Returns (dz, xhat).
    """
    mu = z.mean(axis=-1, keepdims=True)
    c = z - mu
    rstd = 1.0 / np.sqrt((c * c).mean(axis=-1, keepdims=True) + eps)
    xhat = c * rstd
    dxhat = dy_hat_aff * gamma
    dz = rstd * (dxhat - dxhat.mean(axis=-1, keepdims=True)
                 - xhat * (dxhat * xhat).mean(axis=-1, keepdims=True))
    return dz, xhat


def ffn_problem_backward(X, dY, w1, b1, wout, bout, nxw, nxb, ngw, ngb, eps, H):
    """Backward of one (rank, slice) problem for the rows given, in fp64.

    Forward: Z = X w1 + b1; U,G = halves; a = LN_x(U); s = LN_g(G);
    Hl = a * silu(s); Y = Hl wout + bout.  Backward, by the chain rule:
    dHl = dY wout^T; da = dHl*silu(s); ds = dHl*a*silu'(s) with
    silu'(s) = sig(s)*(1 + s*(1-sig(s))); LN backward for each half;
    dZ = [dU, dG]; dX = dZ w1^T; dw1 = X^T dZ; db1 = sum_n dZ;
    dwout = Hl^T dY; dbout = sum_n dY; dgamma_x = sum_n da*xhat_u,
    dbeta_x = sum_n da (and the same for the gate half with ds).
    """
    Z = X @ w1 + b1
    U, G = Z[:, :H], Z[:, H:]
    a = layer_norm(U, nxw, nxb, eps)
    s = layer_norm(G, ngw, ngb, eps)
    sig = 1.0 / (1.0 + np.exp(-s))
    q = s * sig
    Hl = a * q
    dHl = dY @ wout.T
    da = dHl * q
    ds = dHl * a * (sig * (1.0 + s * (1.0 - sig)))
    dU, xu = _layer_norm_backward(da, U, nxw, eps)
    dG, xg = _layer_norm_backward(ds, G, ngw, eps)
    dZ = np.concatenate([dU, dG], axis=1)
    return dict(
        dX=dZ @ w1.T, dw1=X.T @ dZ, db1=dZ.sum(axis=0),
        dwout=Hl.T @ dY, dbout=dY.sum(axis=0),
        dnx_w=(da * xu).sum(axis=0), dnx_b=da.sum(axis=0),
        dng_w=(ds * xg).sum(axis=0), dng_b=ds.sum(axis=0),
    )


def ffn_backward(sh: FFNShape, inputs, prm: dict, dY, decoded: bool = False) -> dict:
    """All gradients of the layer (inputs and every parameter), float64.

    The adjoint of combine is dispatch and the adjoint of dispatch is combine,
    so dYlocal = dispatch(dY) and d_inputs = combine(dXlocal).  Norm weight
    gradients of rank r sum over its rows n and its L slices.
    """
    P, B, L, D, H = sh.P, sh.B, sh.L, sh.D, sh.H
    x = np.asarray(inputs, dtype=np.float64) if decoded else bf16_to_f64(inputs)
    dy = np.asarray(dY, dtype=np.float64) if decoded else bf16_to_f64(dY)
    p = prm if decoded else _decode_ffn_params(sh, prm)
    X = a2a_dispatch(x.reshape(P, B, sh.T, D))
    dYl = a2a_dispatch(dy.reshape(P, B, sh.T, D))
    dXl = np.empty_like(X)
    g = dict(dw1=np.empty((P, L, D, 2 * H)), db1=np.empty((P, L, 2 * H)),
             dwout=np.empty((P, L, H, D)), dbout=np.empty((P, L, D)),
             dnx_w=np.zeros((P, H)), dnx_b=np.zeros((P, H)),
             dng_w=np.zeros((P, H)), dng_b=np.zeros((P, H)))
    for r in range(P):
        for l in range(L):
            o = ffn_problem_backward(
                X[r, :, l, :], dYl[r, :, l, :], p["w1"][r, l], p["b1"][r, l],
                p["wout"][r, l], p["bout"][r, l], p["nxw"][r], p["nxb"][r],
                p["ngw"][r], p["ngb"][r], sh.eps, H)
            dXl[r, :, l, :] = o["dX"]
            for key in ("dw1", "db1", "dwout", "dbout"):
                g[key][r, l] = o[key]
            for key in ("dnx_w", "dnx_b", "dng_w", "dng_b"):
                g[key][r] += o[key]
    g["d_inputs"] = a2a_combine(dXl, B)
    return g


def _problem_rows(sh: FFNShape, x_all, r, l, ns):
    P, B, T = sh.P, sh.B, sh.T
    return [dispatch_source_row(P, B, T, r, n, l) for n in ns]


def _problem_params(sh: FFNShape, prm: dict, r: int, l: int) -> dict:
    P, L, D, H = sh.P, sh.L, sh.D, sh.H
    f = bf16_to_f64
    return dict(
        w1=f(np.asarray(prm["w1"]).reshape(P, L, D, 2 * H)[r, l]),
        b1=f(np.asarray(prm["b1"]).reshape(P, L, 2 * H)[r, l]),
        wout=f(np.asarray(prm["wout"]).reshape(P, L, H, D)[r, l]),
        bout=f(np.asarray(prm["bout"]).reshape(P, L, D)[r, l]),
        nxw=f(np.asarray(prm["nx_w"]).reshape(P, H)[r]),
        nxb=f(np.asarray(prm["nx_b"]).reshape(P, H)[r]),
        ngw=f(np.asarray(prm["ng_w"]).reshape(P, H)[r]),
        ngb=f(np.asarray(prm["ng_b"]).reshape(P, H)[r]),
    )


def _run_problem(sh, inputs_bits, prm, dY_bits, r, l, ns):
    P, B, T, D, H = sh.P, sh.B, sh.T, sh.D, sh.H
    x_all = np.asarray(inputs_bits).reshape(P * B * T, D)
    dy_all = np.asarray(dY_bits).reshape(P * B * T, D)
    src = _problem_rows(sh, x_all, r, l, ns)
    p = _problem_params(sh, prm, r, l)
    return ffn_problem_backward(
        bf16_to_f64(x_all[src]), bf16_to_f64(dy_all[src]), p["w1"], p["b1"], p["wout"],
        p["bout"], p["nxw"], p["nxb"], p["ngw"], p["ngb"], sh.eps, H)


def ffn_backward_dx_rows(sh: FFNShape, inputs_bits, prm: dict, dY_bits, in_rows) -> np.ndarray:
    """Selected rows of d_inputs (flat (s*B+b)*T+t); each row depends only on itself."""
    P, B, T, L = sh.P, sh.B, sh.T, sh.L
    in_rows = np.asarray(in_rows, dtype=np.int64)
    out = np.empty((len(in_rows), sh.D))
    sbt = np.stack(np.unravel_index(in_rows, (P, B, T)), axis=1)
    problems = {}
    for i, (s, b, t) in enumerate(sbt):
        r, l = divmod(int(t), L)
        problems.setdefault((r, l), []).append((i, int(s) * B + int(b)))
    for (r, l), items in problems.items():
        o = _run_problem(sh, inputs_bits, prm, dY_bits, r, l, [n for _, n in items])
        out[[i for i, _ in items]] = o["dX"]
    return out


def ffn_backward_problem(sh: FFNShape, inputs_bits, prm: dict, dY_bits, t: int) -> dict:
    """Full gradients owned by token position t = r*L + l: dw1[t], db1[t], dwout[t],
    dbout[t], plus this slice's contribution to rank r's norm gradients."""
    r, l = divmod(int(t), sh.L)
    return _run_problem(sh, inputs_bits, prm, dY_bits, r, l, range(sh.M))


def _problem_norm_grads(X, dY, w1, b1, wout, nxw, nxb, ngw, ngb, eps, H):
    """The LayerNorm weight/bias gradients of one (rank, slice) problem alone.

    The same chain rule as ffn_problem_backward, stopped where these four
    gradients are complete: Z = X w1 + b1, a = LN_x(U), s = LN_g(G),
    dHl = dY wout^T, da = dHl*silu(s), ds = dHl*a*silu'(s); then
    dgamma_x = sum_n da*xhat_u, dbeta_x = sum_n da, and the same with ds and
    xhat_g (xhat the normalised half before the affine).
    """
    Z = X @ w1 + b1
    U, G = Z[:, :H], Z[:, H:]
    a = layer_norm(U, nxw, nxb, eps)
    s = layer_norm(G, ngw, ngb, eps)
    sig = 1.0 / (1.0 + np.exp(-s))
    dHl = dY @ wout.T
    da = dHl * (s * sig)
    ds = dHl * a * (sig * (1.0 + s * (1.0 - sig)))
    xu = layer_norm(U, 1.0, 0.0, eps)
    xg = layer_norm(G, 1.0, 0.0, eps)
    return dict(dnx_w=(da * xu).sum(axis=0), dnx_b=da.sum(axis=0),
                dng_w=(ds * xg).sum(axis=0), dng_b=ds.sum(axis=0))


def ffn_backward_norm_rank(sh: FFNShape, inputs_bits, prm: dict, dY_bits, r: int) -> dict:
    """Rank r's LayerNorm weight/bias gradients: sums over its L slices and all rows."""
    P, B, T, D, H = sh.P, sh.B, sh.T, sh.D, sh.H
    x_all = np.asarray(inputs_bits).reshape(P * B * T, D)
    dy_all = np.asarray(dY_bits).reshape(P * B * T, D)
    acc = None
    for l in range(sh.L):
        src = _problem_rows(sh, x_all, r, l, range(sh.M))
        p = _problem_params(sh, prm, r, l)
        part = _problem_norm_grads(bf16_to_f64(x_all[src]), bf16_to_f64(dy_all[src]), p["w1"], p["b1"], p["wout"],
                                   p["nxw"], p["nxb"], p["ngw"], p["ngb"], sh.eps, H)
        acc = part if acc is None else {k: acc[k] + part[k] for k in acc}
    return acc


# ---------------------------------------------------------------------------
# comp_only: the layer without the exchange
# ---------------------------------------------------------------------------
#
# The project statement's forward_ffn(ffn, inputs, *, comp_only=False)
# ("Interface, layout, and parameters") names a compute-only mode without
# defining it.  Reading: no exchange -- rank r's own inputs [B, T, D] are
# viewed as [B, P, L, D] (token t = p*L + l), i.e. [B*P, L, D] with row
# n = b*P + p, and slice l of that view goes through rank r's problem l
# (w1[r][l], ..., the rank's norm_x / norm_gate); the result is viewed back
# to [B, T, D] at the same place.  Every row is still processed on its own.

def _comp_only_view(x_r, sh: FFNShape):
    """[B, T, D] -> [B*P, L, D] (row n = b*P + p holds token t = p*L + l)."""
    return x_r.reshape(sh.B, sh.P, sh.L, -1).reshape(sh.B * sh.P, sh.L, -1)


def _comp_only_unview(y_r, sh: FFNShape):
    """[B*P, L, D] -> [B, T, D], the inverse of _comp_only_view."""
    return y_r.reshape(sh.B, sh.P, sh.L, -1).reshape(sh.B, sh.T, -1)


def ffn_forward_comp_only(sh: FFNShape, inputs, prm: dict, decoded: bool = False) -> np.ndarray:
    """The layer in comp_only mode (no exchange), float64 [P, B, T, D]."""
    P, L, D, H = sh.P, sh.L, sh.D, sh.H
    x = np.asarray(inputs, dtype=np.float64) if decoded else bf16_to_f64(inputs)
    x = x.reshape(P, sh.B, sh.T, D)
    p = prm if decoded else _decode_ffn_params(sh, prm)
    out = np.empty_like(x)
    for r in range(P):
        Xr = _comp_only_view(x[r], sh)
        Yr = np.empty_like(Xr)
        for l in range(L):
            _, _, Yr[:, l, :] = _ffn_problem_forward(
                Xr[:, l, :], p["w1"][r, l], p["b1"][r, l], p["wout"][r, l], p["bout"][r, l],
                p["nxw"][r], p["nxb"][r], p["ngw"][r], p["ngb"][r], sh.eps, H)
        out[r] = _comp_only_unview(Yr, sh)
    return out


def ffn_backward_comp_only(sh: FFNShape, inputs, prm: dict, dY, decoded: bool = False) -> dict:
    """All gradients of the comp_only layer, float64 (keys as ffn_backward)."""
    P, L, D, H = sh.P, sh.L, sh.D, sh.H
    x = np.asarray(inputs, dtype=np.float64) if decoded else bf16_to_f64(inputs)
    dy = np.asarray(dY, dtype=np.float64) if decoded else bf16_to_f64(dY)
    x = x.reshape(P, sh.B, sh.T, D)
    dy = dy.reshape(P, sh.B, sh.T, D)
    p = prm if decoded else _decode_ffn_params(sh, prm)
    g = dict(d_inputs=np.empty_like(x), dw1=np.empty((P, L, D, 2 * H)), db1=np.empty((P, L, 2 * H)),
             dwout=np.empty((P, L, H, D)), dbout=np.empty((P, L, D)),
             dnx_w=np.zeros((P, H)), dnx_b=np.zeros((P, H)), dng_w=np.zeros((P, H)), dng_b=np.zeros((P, H)))
    for r in range(P):
        Xr, dYr = _comp_only_view(x[r], sh), _comp_only_view(dy[r], sh)
        dXr = np.empty_like(Xr)
        for l in range(L):
            o = ffn_problem_backward(Xr[:, l, :], dYr[:, l, :], p["w1"][r, l], p["b1"][r, l], p["wout"][r, l],
                                     p["bout"][r, l], p["nxw"][r], p["nxb"][r], p["ngw"][r], p["ngb"][r],
                                     sh.eps, H)
            dXr[:, l, :] = o["dX"]
            for key in ("dw1", "db1", "dwout", "dbout"):
                g[key][r, l] = o[key]
            for key in ("dnx_w", "dnx_b", "dng_w", "dng_b"):
                g[key][r] += o[key]
        g["d_inputs"][r] = _comp_only_unview(dXr, sh)
    return g


# ---------------------------------------------------------------------------
# (c) TP SwiGLU column/row-parallel pair
# ---------------------------------------------------------------------------

def _swiglu_shards(x_rows, w13, w2, W):
    """Y = sum_s h_s @ w2_s^T with h_s = silu(X w1_s^T) * (X w3_s^T).

    w13: [W, 2F, d] where rows [0,F) of shard s are w1_s and rows [F,2F) are
    w3_s (the packed column-parallel pair); w2: [d, ffn] stock layout whose
    column block s*F..(s+1)*F is shard s of the row-parallel projection.
    """
    F = w13.shape[1] // 2
    Y = np.zeros((x_rows.shape[0], w2.shape[0]))
    for s in range(W):
        a = x_rows @ w13[s, :F].T
        b = x_rows @ w13[s, F:].T
        h = silu(a) * b
        Y += h @ w2[:, s * F:(s + 1) * F].T          # partial of shard s, then the sum
    return Y


def tp_swiglu(x_shards, w13, w2, W: int, bsz: int = 1, decoded: bool = False) -> np.ndarray:
    """The SwiGLU pair over W tensor-parallel shards, all shards summed.

    x_shards: [W, bsz, S/W, d] (sequence shards of each rank).  All-gather
    concatenates whole per-rank blocks, i.e. rows in (rank, batch, seq_local)
    order; the forward puts the sequence outermost before flattening, so the
    GEMM rows are (rank, seq_local, batch).  Each shard computes its
    column-parallel GEMM pair and its row-parallel partial; the partials are
    summed (reduce) and the rows split back into W sequence shards (scatter),
    undoing the flattening.  Returns float64 y_shards [W, bsz, S/W, d].
    """
    xs = np.asarray(x_shards)
    Wn, b_, sl, d = xs.shape
    f = (lambda a: np.asarray(a, dtype=np.float64)) if decoded else bf16_to_f64
    x = f(xs)
    # gather with the sequence outermost: rows (rank, seq_local, batch)
    X = x.transpose(0, 2, 1, 3).reshape(Wn * sl * b_, d)
    Y = _swiglu_shards(X, f(w13), f(w2), W)
    # scatter: rank w owns rows [w*sl*b_, (w+1)*sl*b_), viewed [sl, b_, d] -> [b_, sl, d]
    return Y.reshape(Wn, sl, b_, -1).transpose(0, 2, 1, 3)


def tp_swiglu_rows(x_shards_bits, w13_bits, w2_bits, W: int, rows) -> np.ndarray:
    """Selected output rows (flat indices into y_shards [W*bsz*S/W]) of tp_swiglu.

    The layer is row-local (each token row passes through the same pair of
    projections), so a row of y_shards is the pair applied to the same row of
    x_shards.
    """
    xs = np.asarray(x_shards_bits)
    d = xs.shape[-1]
    X = bf16_to_f64(xs.reshape(-1, d)[np.asarray(rows, dtype=np.int64)])
    return _swiglu_shards(X, bf16_to_f64(w13_bits), bf16_to_f64(w2_bits), W)


def _swiglu_shard_backward(X, dY, w13s, w2s):
    """Gradients of one shard's pair, Y_s = (silu(X w1_s^T) * (X w3_s^T)) w2_s^T.

    The row-parallel sum passes dY unchanged to every shard's partial.  With
    a = X w1^T, b = X w3^T, sig = sigmoid(a), h = a*sig*b:
      dh = dY w2_s;  dw2_s = dY^T h;
      da = dh * b * (sig + a*sig*(1 - sig));  db = dh * a * sig;
      dw1_s = da^T X;  dw3_s = db^T X;  dX_s = [da | db] [w1_s ; w3_s]
    (one concatenated product for both column-parallel projections).
    """
    F = w13s.shape[0] // 2
    w1, w3 = w13s[:F], w13s[F:]
    a = X @ w1.T
    b = X @ w3.T
    sig = 1.0 / (1.0 + np.exp(-a))
    h = a * sig * b
    dh = dY @ w2s
    da = dh * b * (sig + a * sig * (1.0 - sig))
    db = dh * a * sig
    dab = np.concatenate([da, db], axis=1)
    return dict(dX=dab @ w13s, dw13=dab.T @ X, dw2=dY.T @ h)


def tp_swiglu_backward(x_shards, w13, w2, dy_shards, W: int, decoded: bool = False) -> dict:
    """Gradients of tp_swiglu w.r.t. x_shards, w13 and w2 (float64).

    Rows are gathered exactly as in the forward (rank, seq_local, batch);
    each shard's gradients follow _swiglu_shard_backward; dX sums the
    shards' contributions (the transpose of the all-gather is a
    reduce-scatter), then is scattered back to [W, bsz, S/W, d].
    """
    xs = np.asarray(x_shards)
    Wn, b_, sl, d = xs.shape
    f = (lambda a: np.asarray(a, dtype=np.float64)) if decoded else bf16_to_f64
    X = f(xs).transpose(0, 2, 1, 3).reshape(Wn * sl * b_, d)
    dY = f(np.asarray(dy_shards)).transpose(0, 2, 1, 3).reshape(Wn * sl * b_, d)
    w13f, w2f = f(w13), f(w2)
    F = w13f.shape[1] // 2
    dX = np.zeros_like(X)
    dw13 = np.empty_like(w13f)
    dw2 = np.empty_like(w2f)
    for s in range(W):
        o = _swiglu_shard_backward(X, dY, w13f[s], w2f[:, s * F:(s + 1) * F])
        dX += o["dX"]
        dw13[s] = o["dw13"]
        dw2[:, s * F:(s + 1) * F] = o["dw2"]
    dx = dX.reshape(Wn, sl, b_, d).transpose(0, 2, 1, 3)
    return dict(dx=dx, dw13=dw13, dw2=dw2)


def tp_swiglu_backward_rows(x_shards_bits, w13_bits, w2_bits, dy_shards_bits, W: int, rows) -> np.ndarray:
    """Selected rows (flat, memory order of x_shards) of dx: row-local like the forward."""
    xs = np.asarray(x_shards_bits)
    d = xs.shape[-1]
    r = np.asarray(rows, dtype=np.int64)
    X = bf16_to_f64(xs.reshape(-1, d)[r])
    dY = bf16_to_f64(np.asarray(dy_shards_bits).reshape(-1, d)[r])
    w13f, w2f = bf16_to_f64(w13_bits), bf16_to_f64(w2_bits)
    F = w13f.shape[1] // 2
    dX = np.zeros_like(X)
    for s in range(W):
        dX += _swiglu_shard_backward(X, dY, w13f[s], w2f[:, s * F:(s + 1) * F])["dX"]
    return dX


def tp_swiglu_backward_weight_cols(x_shards_bits, w13_bits, w2_bits, dy_shards_bits, W: int, cols) -> dict:
    """dw2[:, j] and the rows j of w1_s / w3_s gradients for selected ffn columns j.

    Column j = s*F + c of the ffn axis belongs to shard s; its weight
    gradients need a[:, c], b[:, c] over all rows only, so a column subset is
    exact.  Returns dw2 [d, len(cols)], dw1 [len(cols), d], dw3 [len(cols), d].
    """
    xs = np.asarray(x_shards_bits)
    d = xs.shape[-1]
    X = bf16_to_f64(xs.reshape(-1, d))
    dY = bf16_to_f64(np.asarray(dy_shards_bits).reshape(-1, d))
    w13f, w2f = bf16_to_f64(w13_bits), bf16_to_f64(w2_bits)
    F = w13f.shape[1] // 2
    cols = np.asarray(cols, dtype=np.int64)
    s_idx, c_idx = np.divmod(cols, F)
    w1 = w13f[s_idx, c_idx]          # [n, d]
    w3 = w13f[s_idx, F + c_idx]
    a = X @ w1.T
    b = X @ w3.T
    sig = 1.0 / (1.0 + np.exp(-a))
    h = a * sig * b
    dh = dY @ w2f[:, cols]
    da = dh * b * (sig + a * sig * (1.0 - sig))
    db = dh * a * sig
    return dict(dw2=dY.T @ h, dw1=da.T @ X, dw3=db.T @ X)


# --------------------------------------------------------------------------
# Attention projections: the column-parallel AllGatherLinear (the fused QKV
# projection) and the row-parallel LinearReduceScatter (the output projection
# wo), "Add dist GEMM attention and FFN backend" (torchtitan PR #4044),
# sections "Structure" and "Row ordering".  Both keep the stock parameter
# layout: weight [out, in]; the column-parallel shard s is the row block
# [s*out/W, (s+1)*out/W) of the weight (and of the bias), the row-parallel
# shard s is the column block [s*in/W, (s+1)*in/W).
# --------------------------------------------------------------------------

def _gather_rows(x_shards):
    """All-gather of sequence shards [W, bsz, S/W, f] -> rows (rank, seq_local, batch)."""
    Wn, b_, sl, f = x_shards.shape
    return x_shards.transpose(0, 2, 1, 3).reshape(Wn * sl * b_, f)


def _scatter_rows(Y, Wn, b_):
    """Inverse of _gather_rows: rows (rank, seq_local, batch) -> [W, bsz, S/W, f]."""
    sl = Y.shape[0] // (Wn * b_)
    return Y.reshape(Wn, sl, b_, -1).transpose(0, 2, 1, 3)


def allgather_linear(x_shards, weight, bias, W: int, decoded: bool = False) -> np.ndarray:
    """Column-parallel linear over W shards: every rank gathers all sequence
    shards and multiplies by its own block of output features.

    x_shards [W, bsz, S/W, in]; weight [out, in]; bias [out] or None.
    Returns float64 [W, S*bsz, out/W]: rank s's output Y_s = X W_s^T + b_s,
    rows in gathered order (rank, seq_local, batch).
    """
    f = (lambda a: np.asarray(a, dtype=np.float64)) if decoded else bf16_to_f64
    X = _gather_rows(f(np.asarray(x_shards)))
    Wt = f(np.asarray(weight))
    bt = None if bias is None else f(np.asarray(bias))
    F = Wt.shape[0] // W
    out = []
    for s in range(W):
        Ys = X @ Wt[s * F:(s + 1) * F].T
        if bt is not None:
            Ys = Ys + bt[s * F:(s + 1) * F]
        out.append(Ys)
    return np.stack(out)


def linear_reduce_scatter(a_ranks, weight, bias, W: int, bsz: int = 1, decoded: bool = False) -> np.ndarray:
    """Row-parallel linear over W shards: each rank multiplies its block of
    input features by its block of weight columns, the partial products are
    summed (reduce) and the rows split back into sequence shards (scatter).

    a_ranks [W, S*bsz, in/W] (rank s's input features for all gathered rows,
    in gathered order); weight [out, in]; bias [out] or None, added once to the
    sum.  Returns float64 y_shards [W, bsz, S/W, out].
    """
    f = (lambda a: np.asarray(a, dtype=np.float64)) if decoded else bf16_to_f64
    A = f(np.asarray(a_ranks))
    Wt = f(np.asarray(weight))
    K = A.shape[2]
    Y = np.zeros((A.shape[1], Wt.shape[0]))
    for s in range(W):
        Y += A[s] @ Wt[:, s * K:(s + 1) * K].T        # partial of shard s, then the sum
    if bias is not None:
        Y = Y + f(np.asarray(bias))
    return _scatter_rows(Y, W, bsz)


def allgather_linear_backward(x_shards, weight, dy_ranks, W: int, decoded: bool = False) -> dict:
    """Gradients of allgather_linear given dY_s [W, S*bsz, out/W].

    Per rank: dW_s = dY_s^T X, db_s = sum over rows of dY_s, and the rank's
    share of dX, dY_s W_s; the shares are summed (the transpose of the
    all-gather is a reduce-scatter) and scattered to [W, bsz, S/W, in].
    Returns dx_shards, d_weight [out, in], d_bias [out].
    """
    f = (lambda a: np.asarray(a, dtype=np.float64)) if decoded else bf16_to_f64
    xs = f(np.asarray(x_shards))
    Wn, b_ = xs.shape[0], xs.shape[1]
    X = _gather_rows(xs)
    Wt = f(np.asarray(weight))
    dY = f(np.asarray(dy_ranks))
    F = Wt.shape[0] // W
    dX = np.zeros_like(X)
    dW = np.zeros_like(Wt)
    db = np.zeros(Wt.shape[0])
    for s in range(W):
        dX += dY[s] @ Wt[s * F:(s + 1) * F]
        dW[s * F:(s + 1) * F] = dY[s].T @ X
        db[s * F:(s + 1) * F] = dY[s].sum(axis=0)
    return dict(dx=_scatter_rows(dX, Wn, b_), d_weight=dW, d_bias=db)


def linear_reduce_scatter_backward(a_ranks, weight, dy_shards, W: int, decoded: bool = False) -> dict:
    """Gradients of linear_reduce_scatter given dy_shards [W, bsz, S/W, out].

    dY is all-gathered back to rows in gathered order (the transpose of the
    reduce-scatter); each rank gets dA_s = dY W_s (its block of weight
    columns) and dW_s = dY^T A_s; d_bias = sum over rows of dY.
    Returns da_ranks [W, S*bsz, in/W], d_weight [out, in], d_bias [out].
    """
    f = (lambda a: np.asarray(a, dtype=np.float64)) if decoded else bf16_to_f64
    A = f(np.asarray(a_ranks))
    Wt = f(np.asarray(weight))
    dY = _gather_rows(f(np.asarray(dy_shards)))
    K = A.shape[2]
    dA = np.stack([dY @ Wt[:, s * K:(s + 1) * K] for s in range(W)])
    dW = np.concatenate([dY.T @ A[s] for s in range(W)], axis=1)
    return dict(da=dA, d_weight=dW, d_bias=dY.sum(axis=0))


# --------------------------------------------------------------------------
# FP8 GEMMs inside the A2A FFN (forward).  The project statement lists
# optional FP8 paths for the layer ("Public checks and instructor coverage")
# without a recipe; the reading taken here: GEMM1 and GEMM2 run on e4m3
# operands with fp32 accumulation; activations (the dispatched input rows and
# Hl) carry one scale per row, weights one scale per output column; a scale is
# amax / 448 (1 for an all-zero vector) and a code is the e4m3 value nearest to
# x * (448 / amax), ties to the even code, saturating at +-448.  The code
# decision is taken in binary32 (amax, the quotient 448 / amax and the product
# are binary32 operations), as on the GPU.  Everything after the decoded codes
# is fp64.
# --------------------------------------------------------------------------

_E4M3_MAX = 448.0
# non-negative finite e4m3 values in code order (codes 0x00..0x7e are increasing)
_E4M3_POS_VALUES = _E4M3_TABLE[:0x7f]


def e4m3_rne(x) -> np.ndarray:
    """Codes (uint8) of the e4m3 values nearest to x: ties to the even code,
    magnitudes above 448 (and infinities) saturate to +-448, NaN gives 0x7f."""
    v = np.asarray(x, dtype=np.float64)
    a = np.abs(v)
    sat = np.minimum(np.nan_to_num(a, nan=0.0, posinf=_E4M3_MAX), _E4M3_MAX)
    hi = np.searchsorted(_E4M3_POS_VALUES, sat, side="left")    # first value >= |x|
    hi = np.minimum(hi, 0x7e)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_POS_VALUES[hi] - sat
    d_lo = sat - _E4M3_POS_VALUES[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(_E4M3_POS_VALUES[hi] == sat, hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    code = np.where(np.signbit(v), code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(np.isnan(v), np.uint8(0x7f), code).astype(np.uint8)


def quantize_e4m3(x, axis: int):
    """e4m3 codes and binary32 scales of x (binary32 values) with one scale per
    slice along `axis` (axis=1: per row of a [rows, K] matrix; axis=0: per
    column of a [K, N] matrix).  code = e4m3_rne(x * inv), inv = 448 / amax,
    scale = amax / 448 (inv = scale = 1 for an all-zero slice)."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=axis)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1.0)).astype(np.float32)
    scale = np.where(nz, safe / np.float32(_E4M3_MAX), np.float32(1.0)).astype(np.float32)
    inv = np.where(nz, np.float32(_E4M3_MAX) / safe, np.float32(1.0)).astype(np.float32)
    iv = inv[:, None] if axis == 1 else inv[None, :]
    return e4m3_rne((x32 * iv).astype(np.float32)), scale


def ffn_forward_fp8(sh: FFNShape, inputs, prm: dict, decoded: bool = False) -> np.ndarray:
    """The A2A FFN forward with both GEMMs on e4m3 operands (see above).

    Same dispatch / LayerNorm-gate / combine as ffn_forward; Z and Hl stay
    fp64 apart from the quantisation of Hl (per row, from its binary32 value)
    before GEMM2.  Returns float64 output [P, B, T, D].
    """
    f = (lambda a: np.asarray(a, dtype=np.float64)) if decoded else bf16_to_f64
    x = f(np.asarray(inputs))                                  # [P, B, T, D]
    p = {k: f(np.asarray(v)) for k, v in prm.items()}
    P, B, T, D, H, L = sh.P, sh.B, sh.T, sh.D, sh.H, sh.L
    # per-row quantisation of every input token row (s, b, t)
    xq, sx = quantize_e4m3(x.reshape(-1, D), axis=1)
    xd = (e4m3_to_f64(xq) * sx.astype(np.float64)[:, None]).reshape(P, B, T, D)
    out = np.zeros((P, B, T, D))
    for r in range(P):
        for l in range(L):
            t = r * L + l
            X = xd[:, :, t, :].reshape(P * B, D)               # dispatched rows n = s*B + b
            w1q, s1 = quantize_e4m3(p["w1"][r, l], axis=0)     # [D, 2H], one scale per column
            Z = X @ (e4m3_to_f64(w1q) * s1.astype(np.float64)[None, :]) + p["b1"][r, l]
            a = layer_norm(Z[:, :H], p["nx_w"][r], p["nx_b"][r], sh.eps)
            g = layer_norm(Z[:, H:], p["ng_w"][r], p["ng_b"][r], sh.eps)
            Hl = a * silu(g)
            hq, sh_ = quantize_e4m3(Hl.astype(np.float32), axis=1)
            woq, so = quantize_e4m3(p["wout"][r, l], axis=0)   # [H, D]
            Y = (e4m3_to_f64(hq) * sh_.astype(np.float64)[:, None]) @ \
                (e4m3_to_f64(woq) * so.astype(np.float64)[None, :]) + p["bout"][r, l]
            out[:, :, t, :] = Y.reshape(P, B, D)
    return out


def ffn_forward_fp8_rows(sh: FFNShape, inputs_bits, prm: dict, out_rows) -> np.ndarray:
    """Selected output rows (flat indices into [P, B, T]) of ffn_forward_fp8.

    An output row (s, b, t) needs its own input row (scaled on its own), the
    problem t's weights (scaled per column over the whole weight) and its own
    Hl row (scaled on its own), so a row subset is exact.
    """
    P, B, T, D, H, L = sh.P, sh.B, sh.T, sh.D, sh.H, sh.L
    x = bf16_to_f64(np.asarray(inputs_bits)).reshape(P * B * T, D)
    rows = np.asarray(out_rows, dtype=np.int64)
    res = np.zeros((rows.size, D))
    p = {k: bf16_to_f64(np.asarray(v)) for k, v in prm.items()}
    ts = rows % T
    for t in np.unique(ts):
        r, l = divmod(int(t), L)
        sel = np.nonzero(ts == t)[0]
        xq, sx = quantize_e4m3(x[rows[sel]], axis=1)
        X = e4m3_to_f64(xq) * sx.astype(np.float64)[:, None]
        w1q, s1 = quantize_e4m3(p["w1"][r, l], axis=0)
        Z = X @ (e4m3_to_f64(w1q) * s1.astype(np.float64)[None, :]) + p["b1"][r, l]
        a = layer_norm(Z[:, :H], p["nx_w"][r], p["nx_b"][r], sh.eps)
        g = layer_norm(Z[:, H:], p["ng_w"][r], p["ng_b"][r], sh.eps)
        hq, shs = quantize_e4m3((a * silu(g)).astype(np.float32), axis=1)
        woq, so = quantize_e4m3(p["wout"][r, l], axis=0)
        res[sel] = (e4m3_to_f64(hq) * shs.astype(np.float64)[:, None]) @ \
            (e4m3_to_f64(woq) * so.astype(np.float64)[None, :]) + p["bout"][r, l]
    return res
