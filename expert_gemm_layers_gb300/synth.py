"""Seeded synthetic inputs for the three operations.

This module only draws random numbers and stores them in the operations'
storage types; it holds none of the operations' arithmetic.  Both the CUDA
path and the CPU oracle consume the tensors it returns (the oracle through
``bits()``), so the two sides always read identical bytes.

Distributions follow the workloads the pages describe:

* FFN layer (A2A-FFN project statement, "Interface, layout, and parameters";
  "the benchmark generates inputs using --seed 42 and initializes parameters
  with its he-uniform function"): rank r draws from seed + r, in the order
  inputs, w1, b1, wout, bout.  inputs ~ N(0,1); w ~ U(+-sqrt(6/fan_in)) with
  fan_in the contraction length (D for w1, H for wout); biases
  ~ U(+-1/sqrt(fan_in)); LayerNorm gamma = 1, beta = 0 unless
  ``norm_affine="random"`` (tests use random affines so that gamma/beta bugs
  cannot hide).
* FP8 GEMM: A, B ~ N(0,1) rounded to e4m3 (clamp to +-448, then round to
  nearest even); C ~ N(0,1) in bf16.
* TP SwiGLU: X ~ N(0,1); weights ~ U(+-1/sqrt(fan_in)) (fan_in d for the
  packed [w1;w3], ffn for w2).
"""
from __future__ import annotations

import math

import torch

E4M3_MAX = 448.0


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, g, device, dtype):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def _uniform(shape, bound, g, device, dtype):
    t = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return (t * (2.0 * bound) - bound).to(dtype)


def to_e4m3(x: torch.Tensor) -> torch.Tensor:
    """Round float values to e4m3 (OCP E4M3FN) nearest-even with saturation."""
    return x.float().clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)


def fp8_gemm_inputs(M: int, N: int, K: int, seed: int = 1, device="cpu", with_c: bool = True):
    g = _gen(device, seed)
    A = to_e4m3(torch.randn((M, K), generator=g, device=device))
    B = to_e4m3(torch.randn((N, K), generator=g, device=device))
    C = _normal((M, N), g, device, torch.bfloat16) if with_c else None
    return A, B, C


def ffn_inputs(P: int, B: int, T: int, D: int, k: int, seed: int = 42, device="cpu",
               norm_affine: str = "identity"):
    """Inputs and parameters of the A2A FFN layer, stacked over the P ranks.

    Returns a dict of bf16 tensors: inputs [P,B,T,D], w1 [P,L,D,2H],
    b1 [P,L,2H], wout [P,L,H,D], bout [P,L,D], nx_w/nx_b/ng_w/ng_b [P,H].
    """
    if T % P:
        raise ValueError("T must be divisible by P")
    H, L = D * k, T // P
    bf = torch.bfloat16
    out = {key: [] for key in ("inputs", "w1", "b1", "wout", "bout")}
    for r in range(P):
        g = _gen(device, seed + r)
        out["inputs"].append(_normal((B, T, D), g, device, bf))
        out["w1"].append(_uniform((L, D, 2 * H), math.sqrt(6.0 / D), g, device, bf))
        out["b1"].append(_uniform((L, 2 * H), 1.0 / math.sqrt(D), g, device, bf))
        out["wout"].append(_uniform((L, H, D), math.sqrt(6.0 / H), g, device, bf))
        out["bout"].append(_uniform((L, D), 1.0 / math.sqrt(H), g, device, bf))
    res = {key: torch.stack(v) for key, v in out.items()}
    if norm_affine == "identity":
        res["nx_w"] = torch.ones((P, H), device=device, dtype=bf)
        res["nx_b"] = torch.zeros((P, H), device=device, dtype=bf)
        res["ng_w"] = torch.ones((P, H), device=device, dtype=bf)
        res["ng_b"] = torch.zeros((P, H), device=device, dtype=bf)
    elif norm_affine == "random":
        g = _gen(device, seed + 1000)
        res["nx_w"] = _uniform((P, H), 1.0, g, device, torch.float32).add_(1.0).to(bf)
        res["nx_b"] = _uniform((P, H), 0.5, g, device, bf)
        res["ng_w"] = _uniform((P, H), 1.0, g, device, torch.float32).add_(1.0).to(bf)
        res["ng_b"] = _uniform((P, H), 0.5, g, device, bf)
    else:
        raise ValueError(norm_affine)
    return res


def ffn_grad_output(P: int, B: int, T: int, D: int, seed: int = 43, device="cpu"):
    """Upstream gradient dY [P,B,T,D] ~ N(0,1), bf16."""
    return _normal((P, B, T, D), _gen(device, seed), device, torch.bfloat16)


def tp_swiglu_inputs(S: int, d: int, ffn: int, W: int, bsz: int = 1, seed: int = 7, device="cpu"):
    """x_shards [W, bsz, S/W, d]; w13 [W, 2*ffn/W, d] (rows [w1_s; w3_s]); w2 [d, ffn]."""
    if S % W or ffn % W:
        raise ValueError("S and ffn must be divisible by W")
    g = _gen(device, seed)
    bf = torch.bfloat16
    x = _normal((W, bsz, S // W, d), g, device, bf)
    w13 = _uniform((W, 2 * (ffn // W), d), 1.0 / math.sqrt(d), g, device, bf)
    w2 = _uniform((d, ffn), 1.0 / math.sqrt(ffn), g, device, bf)
    return x, w13, w2


def bits(t: torch.Tensor):
    """Raw storage bits of a bf16 (uint16) or e4m3 (uint8) tensor as a numpy array."""
    import numpy as np
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")
