"""TP SwiGLU pair parity: libdg against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from expert_gemm_layers_gb300 import synth, tp_swiglu
from _compare import TOL_BF16, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.mark.parametrize("S,d,ffn,W,bsz", [
    (256, 128, 512, 2, 1),       # one row tile per shard pair
    (8 * 40, 136, 8 * 72, 8, 1),  # ragged: rows 320, d 136 (K % 64 != 0), F 72 (N % 128 != 0)
    (512, 256, 1024, 4, 2),      # bsz 2: rows in (rank, batch, seq_local) order
    (128, 64, 128, 1, 1),        # a single shard
])
def test_small_full(S, d, ffn, W, bsz):
    x, w13, w2 = synth.tp_swiglu_inputs(S, d, ffn, W, bsz=bsz, seed=S + d)
    y = tp_swiglu(x.to(DEV), w13.to(DEV), w2.to(DEV))
    torch.cuda.synchronize()
    ref = O.tp_swiglu(synth.bits(x), synth.bits(w13), synth.bits(w2), W=W)
    assert_close(y, ref, TOL_BF16, f"tp_swiglu {S,d,ffn,W,bsz}")


def test_shard_count_invariance():
    # the same unsharded weights split over W = 1 and W = 4 shards: identical math,
    # so the results agree to bf16 rounding of the reordered K loop
    S, d, ffn = 256, 128, 512
    g = torch.Generator().manual_seed(4)
    x = torch.randn(S, d, generator=g).to(torch.bfloat16)
    w1 = (torch.rand(ffn, d, generator=g) - 0.5).to(torch.bfloat16)
    w3 = (torch.rand(ffn, d, generator=g) - 0.5).to(torch.bfloat16)
    w2 = ((torch.rand(d, ffn, generator=g) - 0.5) / 8).to(torch.bfloat16)
    ys = []
    for W in (1, 4):
        F = ffn // W
        w13 = torch.stack([torch.cat([w1[s * F:(s + 1) * F], w3[s * F:(s + 1) * F]]) for s in range(W)])
        ys.append(tp_swiglu(x.reshape(W, S // W, d).to(DEV), w13.to(DEV), w2.to(DEV)).reshape(S, d).cpu())
    ref = O.tp_swiglu(synth.bits(x.reshape(1, 1, S, d)), synth.bits(torch.cat([w1, w3]).unsqueeze(0)),
                      synth.bits(w2), W=1).reshape(S, d)
    for y in ys:
        assert_close(y, ref, TOL_BF16, "shard invariance")


def test_full_size_row_subset():
    # Llama-3-8B FFN shape: S=8192, d=4096, ffn=14336 over W=8 shards, seed 7
    S, d, ffn, W = 8192, 4096, 14336, 8
    x, w13, w2 = synth.tp_swiglu_inputs(S, d, ffn, W, seed=7, device=DEV)
    y = tp_swiglu(x, w13, w2)
    torch.cuda.synchronize()
    rows = np.random.default_rng(7).choice(S, size=64, replace=False)
    ref = O.tp_swiglu_rows(synth.bits(x), synth.bits(w13), synth.bits(w2), W, rows)
    got = y.reshape(-1, d)[torch.from_numpy(rows).to(DEV)]
    assert_close(got, ref, TOL_BF16, "tp_swiglu full size (64 rows)")


# ------------------------------------------------------------------ backward

def _grads_vs_oracle(x, w13, w2, dy, W, what):
    from expert_gemm_layers_gb300 import tp_swiglu_backward
    g = tp_swiglu_backward(x.to(DEV), w13.to(DEV), w2.to(DEV), dy.to(DEV))
    torch.cuda.synchronize()
    ref = O.tp_swiglu_backward(synth.bits(x), synth.bits(w13), synth.bits(w2), synth.bits(dy), W=W)
    assert_close(g["x"], ref["dx"], TOL_BF16, f"{what} dx")
    assert_close(g["w13"], ref["dw13"], TOL_BF16, f"{what} dw13")
    assert_close(g["w2"], ref["dw2"], TOL_BF16, f"{what} dw2")


@pytest.mark.parametrize("S,d,ffn,W,bsz", [
    (256, 128, 512, 2, 1),
    (8 * 40, 136, 8 * 72, 8, 1),  # ragged rows (K of the weight GEMMs), d and F off the tile grid
    (512, 256, 1024, 4, 2),
    (128, 64, 128, 1, 1),
    (8, 8, 16, 2, 1),             # far below one tile in every dimension
])
def test_backward_small_full(S, d, ffn, W, bsz):
    x, w13, w2 = synth.tp_swiglu_inputs(S, d, ffn, W, bsz=bsz, seed=S + d + 1)
    dy = synth.tp_swiglu_inputs(S, d, ffn, W, bsz=bsz, seed=S + d + 2)[0]
    _grads_vs_oracle(x, w13, w2, dy, W, f"tp_swiglu_bwd {S,d,ffn,W,bsz}")


def test_backward_autograd_matches_direct_call():
    from expert_gemm_layers_gb300 import tp_swiglu_backward, tp_swiglu_layer
    S, d, ffn, W = 256, 128, 512, 4
    x, w13, w2 = synth.tp_swiglu_inputs(S, d, ffn, W, seed=11, device=DEV)
    dy = synth.tp_swiglu_inputs(S, d, ffn, W, seed=12, device=DEV)[0]
    xr, w13r, w2r = (t.clone().requires_grad_(True) for t in (x, w13, w2))
    y = tp_swiglu_layer(xr, w13r, w2r)
    assert torch.equal(y.detach(), tp_swiglu(x, w13, w2))
    y.backward(dy)
    g = tp_swiglu_backward(x, w13, w2, dy)
    assert torch.equal(xr.grad, g["x"]) and torch.equal(w13r.grad, g["w13"]) and torch.equal(w2r.grad, g["w2"])


def test_backward_full_size_subsets():
    # Llama-3-8B FFN shape over W=8 shards: 64 rows of dx and 16 ffn columns of every weight gradient
    S, d, ffn, W = 8192, 4096, 14336, 8
    F = ffn // W
    from expert_gemm_layers_gb300 import tp_swiglu_backward
    x, w13, w2 = synth.tp_swiglu_inputs(S, d, ffn, W, seed=7, device=DEV)
    dy = synth.tp_swiglu_inputs(S, d, ffn, W, seed=8, device=DEV)[0]
    g = tp_swiglu_backward(x, w13, w2, dy)
    torch.cuda.synchronize()
    xb, w13b, w2b, dyb = synth.bits(x), synth.bits(w13), synth.bits(w2), synth.bits(dy)
    rng = np.random.default_rng(8)
    rows = rng.choice(S, size=64, replace=False)
    ref = O.tp_swiglu_backward_rows(xb, w13b, w2b, dyb, W, rows)
    assert_close(g["x"].reshape(-1, d)[torch.from_numpy(rows).to(DEV)], ref, TOL_BF16, "dx (64 rows)")
    cols = np.sort(np.concatenate([rng.choice(ffn, size=14, replace=False), [0, ffn - 1]]))
    ref = O.tp_swiglu_backward_weight_cols(xb, w13b, w2b, dyb, W, cols)
    c = torch.from_numpy(cols).to(DEV)
    s_idx, c_idx = torch.from_numpy(cols // F).to(DEV), torch.from_numpy(cols % F).to(DEV)
    assert_close(g["w2"][:, c], ref["dw2"], TOL_BF16, "dw2 (16 columns)")
    assert_close(g["w13"][s_idx, c_idx], ref["dw1"], TOL_BF16, "dw1 (16 rows)")
    assert_close(g["w13"][s_idx, F + c_idx], ref["dw3"], TOL_BF16, "dw3 (16 rows)")
