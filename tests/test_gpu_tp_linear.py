"""Attention-projection parity: libdg's linear (column-parallel QKV, row-parallel wo)
against the fp64 oracle's explicit per-shard all-gather linear / linear reduce-scatter."""
import numpy as np
import pytest
import torch

import oracle as O
from expert_gemm_layers_gb300 import synth, tp_linear, tp_linear_backward, tp_linear_layer
from _compare import TOL_BF16, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _bf16(shape, scale, g):
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _ranks_gathered(t, W):
    """[W, bsz, S/W, f] in memory order -> [W, rows, f/W]: rank s's feature block of the
    rows in gathered order (rank, seq_local, batch)."""
    Wn, b_, sl, f = t.shape
    rows = t.permute(0, 2, 1, 3).reshape(Wn * sl * b_, f)
    return torch.stack([rows[:, s * (f // W):(s + 1) * (f // W)] for s in range(W)])


def _from_ranks(y, W, bsz):
    """Inverse of _ranks_gathered for a float64 numpy [W, rows, f/W]."""
    rows = np.concatenate(list(y), axis=1)
    sl = rows.shape[0] // (W * bsz)
    return rows.reshape(W, sl, bsz, -1).transpose(0, 2, 1, 3)


SHAPES = [  # (S, in, out, W, bsz, bias)
    (256, 128, 384, 2, 1, True),
    (8 * 20, 136, 8 * 24, 8, 1, False),    # ragged rows, K % 64 != 0, N % 256 != 0
    (512, 256, 192, 4, 2, True),           # bsz 2: rows in (rank, batch, seq_local) memory order
    (8, 8, 16, 2, 1, True),                # below one tile in every dimension
]


@pytest.mark.parametrize("S,din,dout,W,bsz,has_bias", SHAPES)
def test_column_parallel_forward_backward(S, din, dout, W, bsz, has_bias):
    g = torch.Generator().manual_seed(S + din + dout)
    x = _bf16((W, bsz, S // W, din), 1.0, g)
    w = _bf16((dout, din), din ** -0.5, g)
    b = _bf16((dout,), 0.5, g) if has_bias else None
    dy = _bf16((W, bsz, S // W, dout), 1.0, g)
    y = tp_linear(x.to(DEV), w.to(DEV), None if b is None else b.to(DEV))
    gr = tp_linear_backward(x.to(DEV), w.to(DEV), dy.to(DEV), need_db=has_bias)
    torch.cuda.synchronize()
    ref = O.allgather_linear(synth.bits(x), synth.bits(w), None if b is None else synth.bits(b), W=W)
    assert_close(y, _from_ranks(ref, W, bsz), TOL_BF16, "column-parallel forward")
    rg = O.allgather_linear_backward(synth.bits(x), synth.bits(w), synth.bits(_ranks_gathered(dy, W).contiguous()),
                                     W=W)
    assert_close(gr["x"], rg["dx"], TOL_BF16, "dx")
    assert_close(gr["weight"], rg["d_weight"], TOL_BF16, "d_weight")
    if has_bias:
        assert_close(gr["bias"], rg["d_bias"], TOL_BF16, "d_bias")


@pytest.mark.parametrize("S,din,dout,W,bsz,has_bias", SHAPES)
def test_row_parallel_forward_backward(S, din, dout, W, bsz, has_bias):
    g = torch.Generator().manual_seed(S + din + dout + 1)
    a = _bf16((W, bsz, S // W, din), 1.0, g)
    w = _bf16((dout, din), din ** -0.5, g)
    b = _bf16((dout,), 0.5, g) if has_bias else None
    dy = _bf16((W, bsz, S // W, dout), 1.0, g)
    y = tp_linear(a.to(DEV), w.to(DEV), None if b is None else b.to(DEV))
    gr = tp_linear_backward(a.to(DEV), w.to(DEV), dy.to(DEV), need_db=has_bias)
    torch.cuda.synchronize()
    a_ranks = synth.bits(_ranks_gathered(a, W).contiguous())
    ref = O.linear_reduce_scatter(a_ranks, synth.bits(w), None if b is None else synth.bits(b), W=W, bsz=bsz)
    assert_close(y, ref, TOL_BF16, "row-parallel forward")
    rg = O.linear_reduce_scatter_backward(a_ranks, synth.bits(w), synth.bits(dy), W=W)
    assert_close(gr["x"], _from_ranks(rg["da"], W, bsz), TOL_BF16, "da")
    assert_close(gr["weight"], rg["d_weight"], TOL_BF16, "d_weight")
    if has_bias:
        assert_close(gr["bias"], rg["d_bias"], TOL_BF16, "d_bias")


def test_autograd_matches_direct_calls():
    g = torch.Generator(device=DEV).manual_seed(3)
    x = torch.randn((2, 1, 64, 128), generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn((256, 128), generator=g, device=DEV) / 12).to(torch.bfloat16)
    b = torch.randn((256,), generator=g, device=DEV).to(torch.bfloat16)
    dy = torch.randn((2, 1, 64, 256), generator=g, device=DEV).to(torch.bfloat16)
    xr, wr, br = (t.clone().requires_grad_(True) for t in (x, w, b))
    y = tp_linear_layer(xr, wr, br)
    assert torch.equal(y.detach(), tp_linear(x, w, b))
    y.backward(dy)
    gd = tp_linear_backward(x, w, dy, need_db=True)
    assert torch.equal(xr.grad, gd["x"]) and torch.equal(wr.grad, gd["weight"]) and torch.equal(br.grad, gd["bias"])


@pytest.mark.parametrize("proj", ["qkv", "wo"])
def test_llama3_8b_attention_shapes_subsets(proj):
    # Llama-3-8B attention over W=8 shards, S=8192 tokens: fused QKV [4096 + 2*1024, 4096]
    # (32 query and 8 key/value heads of 128), wo [4096, 4096]; no bias, as in the model
    S, W, d = 8192, 8, 4096
    dout = 6144 if proj == "qkv" else 4096
    g = torch.Generator(device=DEV).manual_seed(7 if proj == "qkv" else 8)
    x = torch.randn((W, 1, S // W, d), generator=g, device=DEV).to(torch.bfloat16)
    w = ((torch.rand((dout, d), generator=g, device=DEV) - 0.5) * (2 / d ** 0.5)).to(torch.bfloat16)
    dy = torch.randn((W, 1, S // W, dout), generator=g, device=DEV).to(torch.bfloat16)
    y = tp_linear(x, w)
    gr = tp_linear_backward(x, w, dy)
    torch.cuda.synchronize()
    rng = np.random.default_rng(9)
    rows = rng.choice(S, size=64, replace=False)
    xb, wb, dyb = synth.bits(x).reshape(S, d), synth.bits(w), synth.bits(dy).reshape(S, dout)
    r = torch.from_numpy(rows).to(DEV)
    # The layer is row-local, so y and dx of a row need only that row: the oracle
    # at W = 1 on the sampled rows (shard blocks are column blocks, pinned above).
    x_rows = xb[rows].reshape(1, 1, 64, d)
    assert_close(y.reshape(S, dout)[r], O.allgather_linear(x_rows, wb, None, W=1)[0], TOL_BF16,
                 f"{proj} y (64 rows)")
    ref = O.allgather_linear_backward(x_rows, wb, dyb[rows].reshape(1, 64, dout), W=1)
    assert_close(gr["x"].reshape(S, d)[r], ref["dx"].reshape(64, d), TOL_BF16, f"{proj} dx (64 rows)")
    # d_weight of 16 output features needs those features' dY over all rows
    feats = np.sort(np.concatenate([rng.choice(dout, size=14, replace=False), [0, dout - 1]]))
    ref = O.allgather_linear_backward(xb.reshape(1, 1, S, d), wb[feats], dyb[:, feats].reshape(1, S, 16), W=1)
    assert_close(gr["weight"][torch.from_numpy(feats).to(DEV)], ref["d_weight"], TOL_BF16,
                 f"{proj} d_weight (16 features)")
