"""Torch-facing wrappers of the libdg entry points.

Each function checks dtypes/devices, allocates outputs and scratch with
torch (device memory only) and passes raw pointers plus the current CUDA
stream to the C ABI.  No arithmetic of the layers happens here.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import (DG_ERROR_BLOCK_BYTES, DG_FFN_COMP_ONLY, DG_FFN_FUSED_GATE, DG_FFN_SEPARATE_GATE, FFNShape,
                   TraceEntry, check, load)

__all__ = [
    "gemm_fp8", "ffn_shape", "a2a_ffn_forward", "a2a_ffn_backward", "a2a_ffn_fp8_pack_weights", "a2a_ffn_forward_fp8", "A2AFFN", "a2a_ffn",
    "a2a_dispatch", "a2a_combine", "tp_swiglu", "tp_swiglu_backward", "TPSwiGLU", "tp_swiglu_layer",
    "tp_linear", "tp_linear_backward", "TPLinear", "tp_linear_layer", "device_status", "debug_wait_timeout",
    "FFN_PARAM_NAMES", "trace_begin", "trace_end", "alloc_workspace", "error_block", "DG_FFN_COMP_ONLY",
    "DG_FFN_FUSED_GATE",
    "DG_FFN_SEPARATE_GATE",
]

FFN_PARAM_NAMES = ("w1", "b1", "wout", "bout", "nx_w", "nx_b", "ng_w", "ng_b")


def _stream(dev: torch.device) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_error_blocks: dict = {}


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A workspace of `nbytes` bytes on `device` whose error block (its first
    DG_ERROR_BLOCK_BYTES bytes) is zeroed on the current stream."""
    ws = torch.empty(max(int(nbytes), DG_ERROR_BLOCK_BYTES), dtype=torch.uint8, device=device)
    ws[:DG_ERROR_BLOCK_BYTES].zero_()
    return ws


def error_block(device=None) -> torch.Tensor:
    """The zeroed error block this module gives calls that need no other
    scratch, one per (device, current stream): calls on different streams
    do not share an error word."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    key = (dev.index, _stream(dev))
    blk = _error_blocks.get(key)
    if blk is None:
        with torch.cuda.device(dev):
            blk = torch.zeros(DG_ERROR_BLOCK_BYTES, dtype=torch.uint8, device=dev)
        _error_blocks[key] = blk
    return blk


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


# ------------------------------------------------------------------ FP8 GEMM

def gemm_fp8(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, alpha: float = 1.0,
             beta: float = 0.0, out: torch.Tensor | None = None, ws: torch.Tensor | None = None) -> torch.Tensor:
    """D = alpha * (A @ B^T) + beta * C with A [M,K], B [N,K] in float8_e4m3fn, C/D bf16 [M,N].
    `ws` holds the call's error block (default: this stream's error_block())."""
    lib = load()
    M, K = A.shape
    N = B.shape[0]
    _need(A, "A", torch.float8_e4m3fn, (M, K))
    _need(B, "B", torch.float8_e4m3fn, (N, K), A.device)
    if C is not None:
        _need(C, "C", torch.bfloat16, (M, N), A.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(out, "out", torch.bfloat16, (M, N), A.device)
    if ws is None:
        ws = error_block(A.device)
    with torch.cuda.device(A.device):
        check(lib.dg_gemm_fp8(M, N, K, _ptr(A), _ptr(B), _ptr(C), _ptr(out), float(alpha), float(beta),
                              _ptr(ws), ws.numel(), ctypes.c_void_p(_stream(A.device))))
    return out


# ------------------------------------------------------------------ A2A FFN

def ffn_shape(P: int, B: int, T: int, D: int, k: int, eps: float = 1e-5) -> FFNShape:
    return FFNShape(P, B, T, D, k, eps)


def _ffn_param_shapes(P, B, T, D, k):
    H, L = D * k, T // P
    return dict(inputs=(P, B, T, D), w1=(P, L, D, 2 * H), b1=(P, L, 2 * H), wout=(P, L, H, D),
                bout=(P, L, D), nx_w=(P, H), nx_b=(P, H), ng_w=(P, H), ng_b=(P, H))


def a2a_ffn_forward(inputs: torch.Tensor, params: dict, eps: float = 1e-5, saved: torch.Tensor | None = None,
                    out: torch.Tensor | None = None, inference: bool = False, flags: int = 0,
                    ws: torch.Tensor | None = None):
    """The A2A FFN layer for all P ranks at once.

    inputs [P,B,T,D] bf16; params: w1 [P,L,D,2H], b1 [P,L,2H], wout [P,L,H,D],
    bout [P,L,D], nx_w/nx_b/ng_w/ng_b [P,H] (bf16), where k = 2H/(2D) is read
    from w1.  Returns (output [P,B,T,D], saved) where `saved` is the opaque
    byte buffer the backward needs (None with inference=True: nothing is
    kept).  flags: DG_FFN_COMP_ONLY; DG_FFN_SEPARATE_GATE (the gate as a
    separate pass instead of inside GEMM2) or DG_FFN_FUSED_GATE (the default).
    """
    lib = load()
    P, B, T, D = inputs.shape
    k = params["w1"].shape[-1] // (2 * D)
    shapes = _ffn_param_shapes(P, B, T, D, k)
    dev = inputs.device
    _need(inputs, "inputs", torch.bfloat16, shapes["inputs"])
    for name in FFN_PARAM_NAMES:
        _need(params[name], name, torch.bfloat16, shapes[name], dev)
    sh = FFNShape(P, B, T, D, k, eps)
    nbytes = lib.dg_a2a_ffn_saved_bytes(ctypes.byref(sh))
    wsb = lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), int(inference), int(flags))
    if nbytes == 0 or wsb == 0:
        check(lib.dg_a2a_ffn_fwd(ctypes.byref(sh), *([None] * 10), None, 0, None, 0, int(flags), None))
    if saved is None and not inference:
        saved = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if inference:
        saved = None
    if ws is None:
        ws = error_block(dev) if wsb <= DG_ERROR_BLOCK_BYTES else alloc_workspace(wsb, dev)
    if out is None:
        out = torch.empty(shapes["inputs"], dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, shapes["inputs"], dev)
    with torch.cuda.device(dev):
        check(lib.dg_a2a_ffn_fwd(ctypes.byref(sh), _ptr(inputs), *[_ptr(params[n]) for n in FFN_PARAM_NAMES],
                                 _ptr(out), _ptr(saved), 0 if saved is None else saved.numel(), _ptr(ws),
                                 ws.numel(), int(flags), ctypes.c_void_p(_stream(dev))))
    return out, saved


def a2a_ffn_fp8_pack_weights(params: dict, P: int, B: int, T: int, D: int, eps: float = 1e-5,
                             packed: torch.Tensor | None = None) -> torch.Tensor:
    """e4m3 copy of w1 and wout (per output column scales) for a2a_ffn_forward_fp8."""
    lib = load()
    k = params["w1"].shape[-1] // (2 * D)
    shapes = _ffn_param_shapes(P, B, T, D, k)
    dev = params["w1"].device
    _need(params["w1"], "w1", torch.bfloat16, shapes["w1"], dev)
    _need(params["wout"], "wout", torch.bfloat16, shapes["wout"], dev)
    sh = FFNShape(P, B, T, D, k, eps)
    nbytes = lib.dg_a2a_ffn_fp8_weights_bytes(ctypes.byref(sh))
    if nbytes == 0:
        check(lib.dg_a2a_ffn_fp8_pack_weights(ctypes.byref(sh), None, None, None, 0, None))
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        check(lib.dg_a2a_ffn_fp8_pack_weights(ctypes.byref(sh), _ptr(params["w1"]), _ptr(params["wout"]), _ptr(packed),
                                              packed.numel(), ctypes.c_void_p(_stream(dev))))
    return packed


def a2a_ffn_forward_fp8(inputs: torch.Tensor, params: dict, packed: torch.Tensor, eps: float = 1e-5,
                        workspace: torch.Tensor | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    """The A2A FFN forward with both GEMMs on e4m3 operands (inference).

    `packed` comes from a2a_ffn_fp8_pack_weights; b1, bout and the LayerNorm
    parameters are taken from `params` (bf16).  Returns output [P,B,T,D] bf16."""
    lib = load()
    P, B, T, D = inputs.shape
    k = params["w1"].shape[-1] // (2 * D)
    shapes = _ffn_param_shapes(P, B, T, D, k)
    dev = inputs.device
    _need(inputs, "inputs", torch.bfloat16, shapes["inputs"])
    names = ("b1", "bout", "nx_w", "nx_b", "ng_w", "ng_b")
    for name in names:
        _need(params[name], name, torch.bfloat16, shapes[name], dev)
    sh = FFNShape(P, B, T, D, k, eps)
    nbytes = lib.dg_a2a_ffn_fp8_workspace_bytes(ctypes.byref(sh))
    if nbytes == 0:
        check(lib.dg_a2a_ffn_fwd_fp8(ctypes.byref(sh), *([None] * 3), *([None] * 7), None, 0, None))
    if workspace is None:
        workspace = alloc_workspace(nbytes, dev)
    if out is None:
        out = torch.empty(shapes["inputs"], dtype=torch.bfloat16, device=dev)
    with torch.cuda.device(dev):
        check(lib.dg_a2a_ffn_fwd_fp8(ctypes.byref(sh), _ptr(inputs), _ptr(packed), packed.numel(),
                                     *[_ptr(params[n]) for n in names], _ptr(out), _ptr(workspace), workspace.numel(),
                                     ctypes.c_void_p(_stream(dev))))
    return out


def a2a_ffn_backward(inputs: torch.Tensor, params: dict, saved: torch.Tensor, dY: torch.Tensor,
                     eps: float = 1e-5, workspace: torch.Tensor | None = None, grads: dict | None = None,
                     flags: int = 0, need: tuple | None = None) -> dict:
    """Gradients of the layer w.r.t. inputs and every parameter (overwritten, bf16).

    Returns a dict with keys "inputs" and the names in FFN_PARAM_NAMES.  With
    `need` (a subset of those keys) only those gradients are computed (the
    others are None and their work is skipped); `grads` may hold None entries
    for the same effect.  flags: those given to the forward (DG_FFN_COMP_ONLY
    applies; the gate flags are accepted and leave the backward unchanged).
    """
    lib = load()
    P, B, T, D = inputs.shape
    k = params["w1"].shape[-1] // (2 * D)
    shapes = _ffn_param_shapes(P, B, T, D, k)
    dev = inputs.device
    _need(dY, "dY", torch.bfloat16, shapes["inputs"], dev)
    sh = FFNShape(P, B, T, D, k, eps)
    wsb = lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), int(flags))
    if workspace is None:
        workspace = alloc_workspace(wsb, dev)
    names = ("inputs",) + FFN_PARAM_NAMES
    if grads is None:
        grads = {name: (torch.empty(shapes[name], dtype=torch.bfloat16, device=dev)
                        if need is None or name in need else None) for name in names}
    g = grads
    with torch.cuda.device(dev):
        check(lib.dg_a2a_ffn_bwd(
            ctypes.byref(sh), _ptr(inputs), *[_ptr(params[n]) for n in FFN_PARAM_NAMES],
            _ptr(saved), 0 if saved is None else saved.numel(), _ptr(dY),
            _ptr(g.get("inputs")), _ptr(g.get("w1")), _ptr(g.get("b1")), _ptr(g.get("wout")), _ptr(g.get("bout")),
            _ptr(g.get("nx_w")), _ptr(g.get("nx_b")), _ptr(g.get("ng_w")), _ptr(g.get("ng_b")),
            _ptr(workspace), workspace.numel(), int(flags), ctypes.c_void_p(_stream(dev))))
    return grads


class A2AFFN(torch.autograd.Function):
    """Autograd wrapper: gradients reach the input and all eight parameters."""

    @staticmethod
    def forward(ctx, inputs, w1, b1, wout, bout, nx_w, nx_b, ng_w, ng_b, eps):
        params = dict(w1=w1, b1=b1, wout=wout, bout=bout, nx_w=nx_w, nx_b=nx_b, ng_w=ng_w, ng_b=ng_b)
        out, saved = a2a_ffn_forward(inputs, params, eps)
        ctx.save_for_backward(inputs, w1, b1, wout, bout, nx_w, nx_b, ng_w, ng_b, saved)
        ctx.eps = eps
        return out

    @staticmethod
    def backward(ctx, dY):
        inputs, w1, b1, wout, bout, nx_w, nx_b, ng_w, ng_b, saved = ctx.saved_tensors
        params = dict(w1=w1, b1=b1, wout=wout, bout=bout, nx_w=nx_w, nx_b=nx_b, ng_w=ng_w, ng_b=ng_b)
        names = ("inputs",) + FFN_PARAM_NAMES
        need = tuple(n for n, want in zip(names, ctx.needs_input_grad[:9]) if want)
        g = a2a_ffn_backward(inputs, params, saved, dY.contiguous(), ctx.eps, need=need)
        return tuple(g[n] for n in names) + (None,)


def a2a_ffn(inputs, params: dict, eps: float = 1e-5):
    """Differentiable A2A FFN layer (see A2AFFN)."""
    return A2AFFN.apply(inputs, *[params[n] for n in FFN_PARAM_NAMES], eps)


def a2a_dispatch(inputs: torch.Tensor) -> torch.Tensor:
    """inputs [P,B,T,D] -> dispatched [P, P*B, T/P, D] (explicit permutation copy)."""
    lib = load()
    P, B, T, D = inputs.shape
    _need(inputs, "inputs", torch.bfloat16)
    out = torch.empty((P, P * B, T // P, D), dtype=torch.bfloat16, device=inputs.device)
    with torch.cuda.device(inputs.device):
        check(lib.dg_a2a_dispatch(P, B, T, D, _ptr(inputs), _ptr(out), ctypes.c_void_p(_stream(inputs.device))))
    return out


def a2a_combine(ylocal: torch.Tensor, B: int) -> torch.Tensor:
    """ylocal [P, P*B, L, D] -> output [P, B, P*L, D] (explicit permutation copy)."""
    lib = load()
    P, PB, L, D = ylocal.shape
    _need(ylocal, "ylocal", torch.bfloat16)
    out = torch.empty((P, B, P * L, D), dtype=torch.bfloat16, device=ylocal.device)
    with torch.cuda.device(ylocal.device):
        check(lib.dg_a2a_combine(P, B, P * L, D, _ptr(ylocal), _ptr(out), ctypes.c_void_p(_stream(ylocal.device))))
    return out


# ------------------------------------------------------------------ TP SwiGLU

def tp_swiglu(x_shards: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor,
              workspace: torch.Tensor | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    """SwiGLU pair over W shards: x_shards [W, bsz, S/W, d] (or [W, S/W, d]),
    w13 [W, 2F, d] (rows [w1_s; w3_s]), w2 [d, W*F].  Returns y_shards like x_shards."""
    lib = load()
    squeeze = x_shards.dim() == 3
    xs = x_shards.unsqueeze(1) if squeeze else x_shards
    W, bsz, sl, d = xs.shape
    ffn = w2.shape[1]
    dev = x_shards.device
    _need(x_shards, "x_shards", torch.bfloat16)
    _need(w13, "w13", torch.bfloat16, (W, 2 * (ffn // W), d), dev)
    _need(w2, "w2", torch.bfloat16, (d, ffn), dev)
    S = W * sl
    wsb = lib.dg_tp_swiglu_workspace_bytes(S, d, ffn, W, bsz)
    if workspace is None:
        workspace = alloc_workspace(wsb, dev)
    if out is None:
        out = torch.empty_like(x_shards)
    with torch.cuda.device(dev):
        check(lib.dg_tp_swiglu(S, d, ffn, W, bsz, _ptr(x_shards), _ptr(w13), _ptr(w2), _ptr(out),
                               _ptr(workspace), workspace.numel(), ctypes.c_void_p(_stream(dev))))
    return out


def tp_swiglu_backward(x_shards: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor, dy_shards: torch.Tensor,
                       workspace: torch.Tensor | None = None, grads: dict | None = None) -> dict:
    """Gradients of tp_swiglu given dy_shards (layout of y_shards): dict with
    "x" (like x_shards), "w13" [W, 2F, d] and "w2" [d, W*F]."""
    lib = load()
    squeeze = x_shards.dim() == 3
    xs = x_shards.unsqueeze(1) if squeeze else x_shards
    W, bsz, sl, d = xs.shape
    ffn = w2.shape[1]
    dev = x_shards.device
    _need(x_shards, "x_shards", torch.bfloat16)
    _need(w13, "w13", torch.bfloat16, (W, 2 * (ffn // W), d), dev)
    _need(w2, "w2", torch.bfloat16, (d, ffn), dev)
    _need(dy_shards, "dy_shards", torch.bfloat16, tuple(x_shards.shape), dev)
    S = W * sl
    wsb = lib.dg_tp_swiglu_bwd_workspace_bytes(S, d, ffn, W, bsz)
    if workspace is None:
        workspace = alloc_workspace(wsb, dev)
    if grads is None:
        grads = dict(x=torch.empty_like(x_shards), w13=torch.empty_like(w13), w2=torch.empty_like(w2))
    with torch.cuda.device(dev):
        check(lib.dg_tp_swiglu_bwd(S, d, ffn, W, bsz, _ptr(x_shards), _ptr(w13), _ptr(w2), _ptr(dy_shards),
                                   _ptr(grads["x"]), _ptr(grads["w13"]), _ptr(grads["w2"]), _ptr(workspace),
                                   workspace.numel(), ctypes.c_void_p(_stream(dev))))
    return grads


class TPSwiGLU(torch.autograd.Function):
    """Autograd wrapper of the SwiGLU pair; the backward recomputes [a|b] from x."""

    @staticmethod
    def forward(ctx, x_shards, w13, w2):
        ctx.save_for_backward(x_shards, w13, w2)
        return tp_swiglu(x_shards, w13, w2)

    @staticmethod
    def backward(ctx, dy):
        x_shards, w13, w2 = ctx.saved_tensors
        g = tp_swiglu_backward(x_shards, w13, w2, dy.contiguous())
        return g["x"], g["w13"], g["w2"]


def tp_swiglu_layer(x_shards, w13, w2):
    """Differentiable SwiGLU pair (see TPSwiGLU)."""
    return TPSwiGLU.apply(x_shards, w13, w2)


# ------------------------------------------------------------------ attention projections

def tp_linear(x: torch.Tensor, weight: torch.Tensor, bias: torch.Tensor | None = None,
              out: torch.Tensor | None = None) -> torch.Tensor:
    """y = x @ weight^T (+ bias) over all tensor-parallel shards at once.

    The column-parallel all-gather linear (fused QKV) and the row-parallel
    linear reduce-scatter (wo) in the stock layout: x [..., in] (e.g. sequence
    shards [W, bsz, S/W, in]), weight [out, in], bias [out]; rank s's block is
    a column block of the output (column parallel) or of x and weight (row
    parallel).  Returns [..., out] with the rows of x in place."""
    lib = load()
    in_f = x.shape[-1]
    out_f = weight.shape[0]
    dev = x.device
    _need(x, "x", torch.bfloat16)
    _need(weight, "weight", torch.bfloat16, (out_f, in_f), dev)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, (out_f,), dev)
    rows = x.numel() // in_f
    if out is None:
        out = torch.empty((*x.shape[:-1], out_f), dtype=torch.bfloat16, device=dev)
    ws = error_block(dev)
    with torch.cuda.device(dev):
        check(lib.dg_tp_linear_fwd(rows, in_f, out_f, _ptr(x), _ptr(weight),
                                   None if bias is None else _ptr(bias), _ptr(out), _ptr(ws), ws.numel(),
                                   ctypes.c_void_p(_stream(dev))))
    return out


def tp_linear_backward(x: torch.Tensor, weight: torch.Tensor, dy: torch.Tensor, need_dx: bool = True,
                       need_dw: bool = True, need_db: bool = False) -> dict:
    """Gradients of tp_linear: "x" = dy weight, "weight" = dy^T x, "bias" = column sums of dy."""
    lib = load()
    in_f = x.shape[-1]
    out_f = weight.shape[0]
    dev = x.device
    _need(x, "x", torch.bfloat16)
    _need(weight, "weight", torch.bfloat16, (out_f, in_f), dev)
    _need(dy, "dy", torch.bfloat16, (*x.shape[:-1], out_f), dev)
    rows = x.numel() // in_f
    g = {}
    g["x"] = torch.empty_like(x) if need_dx else None
    g["weight"] = torch.empty_like(weight) if need_dw else None
    g["bias"] = torch.empty(out_f, dtype=torch.bfloat16, device=dev) if need_db else None
    p = lambda t: None if t is None else _ptr(t)
    ws = error_block(dev)
    with torch.cuda.device(dev):
        check(lib.dg_tp_linear_bwd(rows, in_f, out_f, _ptr(x), _ptr(weight), _ptr(dy), p(g["x"]), p(g["weight"]),
                                   p(g["bias"]), _ptr(ws), ws.numel(), ctypes.c_void_p(_stream(dev))))
    return g


class TPLinear(torch.autograd.Function):
    """Autograd wrapper of tp_linear (gradients for x, weight and bias)."""

    @staticmethod
    def forward(ctx, x, weight, bias):
        ctx.save_for_backward(x, weight)
        ctx.has_bias = bias is not None
        return tp_linear(x, weight, bias)

    @staticmethod
    def backward(ctx, dy):
        x, weight = ctx.saved_tensors
        g = tp_linear_backward(x, weight, dy.contiguous(), need_dx=ctx.needs_input_grad[0],
                               need_dw=ctx.needs_input_grad[1], need_db=ctx.has_bias and ctx.needs_input_grad[2])
        return g["x"], g["weight"], g["bias"]


def tp_linear_layer(x, weight, bias=None):
    """Differentiable tp_linear (see TPLinear)."""
    return TPLinear.apply(x, weight, bias)


# ------------------------------------------------------------------ diagnostics

def device_status(device=None, workspace: torch.Tensor | None = None, builtin: bool = False):
    """Synchronise the current stream and read/clear an error word: that of
    `workspace`, else this stream's error_block() (builtin=True: the library's
    own word, written only by dg_tp_swiglu_noalloc).  Returns (status, raw code)."""
    lib = load()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if builtin:
        ws = None
    else:
        ws = workspace if workspace is not None else error_block(dev)
    site = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        st = lib.dg_check_device_error(_ptr(ws), ctypes.c_void_p(_stream(dev)), ctypes.byref(site))
    return st, site.value


def debug_wait_timeout(limit_us: int, device=None, workspace: torch.Tensor | None = None) -> None:
    """Expire one bounded wait on purpose; the failure lands in `workspace`'s error block
    (default: this stream's error_block())."""
    lib = load()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    ws = workspace if workspace is not None else error_block(dev)
    with torch.cuda.device(dev):
        check(lib.dg_debug_wait_timeout(_ptr(ws), ws.numel(), int(limit_us), ctypes.c_void_p(_stream(dev))))


def trace_begin(only: str | None = None) -> None:
    """Start recording libdg kernel launches with CUDA events: all of them, or
    only those named `only`."""
    if only:
        check(load().dg_trace_begin_only(only.encode()))
    else:
        check(load().dg_trace_begin())


def trace_end() -> list[dict]:
    """Stop recording; per kernel name: launches, total_ms, flops, bytes (algorithmic)."""
    lib = load()
    buf = (TraceEntry * 64)()
    n = lib.dg_trace_end(buf, 64)
    if n < 0:
        check(3)
    return [dict(name=buf[i].name.decode(), launches=int(buf[i].launches), total_ms=buf[i].total_ms,
                 flops=buf[i].flops, bytes=buf[i].bytes) for i in range(min(n, 64))]
