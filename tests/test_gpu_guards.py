"""Guard regions around every buffer the library writes.

Each output, the forward's saved buffer, the packed e4m3 weights and every
workspace are placed between two regions filled with a sentinel byte; after
the call both regions must still hold the sentinel, bit for bit.  A write
past the end or before the start of a buffer -- a TMA box or a plain store at
a ragged edge that was not clipped -- shows up here even where the values
inside the buffer are right.  Shapes are ragged on purpose (rows, columns and
K off the tile grid) and include the FP8 GEMM's 224-column tiles, whose last
32 columns are written with plain stores."""
import ctypes

import pytest
import torch

import expert_gemm_layers_gb300 as dg
from expert_gemm_layers_gb300 import _lib, synth
from test_gpu_a2a_ffn import SMALL_SHAPES

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
PAD = 4096          # guard bytes on each side of a buffer
SENTINEL = 0xA7


class Guarded:
    """Allocates buffers inside sentinel-filled guard regions and checks the guards."""

    def __init__(self):
        self.bufs = []

    def raw(self, nbytes: int) -> torch.Tensor:
        """nbytes of uint8 between two guard regions."""
        body = (nbytes + 255) // 256 * 256
        buf = torch.full((PAD + body + PAD,), SENTINEL, dtype=torch.uint8, device=DEV)
        self.bufs.append((buf, nbytes))
        return buf[PAD:PAD + nbytes]

    def workspace(self, nbytes: int) -> torch.Tensor:
        """A guarded workspace whose error block (the first 256 bytes) is zero."""
        ws = self.raw(max(nbytes, 256))
        ws[:256].zero_()
        return ws

    def tensor(self, shape, dtype) -> torch.Tensor:
        n = 1
        for s in shape:
            n *= s
        itemsize = torch.empty((), dtype=dtype).element_size()
        return self.raw(n * itemsize).view(dtype).view(*shape)

    def like(self, t: torch.Tensor) -> torch.Tensor:
        return self.tensor(tuple(t.shape), t.dtype)

    def check(self, what: str):
        torch.cuda.synchronize()
        for i, (buf, nbytes) in enumerate(self.bufs):
            body = (nbytes + 255) // 256 * 256
            before = buf[:PAD]
            after = buf[PAD + nbytes:]
            assert bool((before == SENTINEL).all()), f"{what}: buffer {i} written before its start"
            assert bool((after == SENTINEL).all()), f"{what}: buffer {i} written past its end ({nbytes} bytes)"
            assert after.numel() == body - nbytes + PAD


@pytest.mark.parametrize("M,N,K,beta", [
    (200, 136, 48, 1.0),     # one ragged tile in each direction
    (257, 232, 64, 0.0),     # a second row tile of one row; no C
    (4000, 4000, 64, 1.0),   # ragged edges of a many-tile grid
    (4096, 4096, 128, 1.0),  # the benchmark grid: 224-column tiles, plain stores at the right edge
])
def test_gemm_fp8_writes_only_d(M, N, K, beta):
    A, B, C = synth.fp8_gemm_inputs(M, N, K, seed=M + N + K, device=DEV)
    g = Guarded()
    D = g.tensor((M, N), torch.bfloat16)
    dg.gemm_fp8(A, B, C if beta != 0.0 else None, 0.5, beta, out=D, ws=g.workspace(256))
    g.check(f"gemm_fp8 {M}x{N}x{K}")
    assert torch.isfinite(D.float()).all()


@pytest.mark.parametrize("P,B,T,D,k", SMALL_SHAPES)
def test_a2a_ffn_forward_backward_write_only_their_buffers(P, B, T, D, k):
    t = synth.ffn_inputs(P, B, T, D, k, seed=P + B + T + D + k, device=DEV)
    params = {n: t[n] for n in dg.FFN_PARAM_NAMES}
    x = t["inputs"]
    dY = synth.ffn_grad_output(P, B, T, D, seed=7, device=DEV)
    lib = _lib.load()
    sh = _lib.FFNShape(P, B, T, D, k, 1e-5)
    g = Guarded()
    out = g.like(x)
    saved = g.raw(lib.dg_a2a_ffn_saved_bytes(ctypes.byref(sh)))
    dg.a2a_ffn_forward(x, params, saved=saved, out=out, ws=g.workspace(256))
    ws = g.workspace(lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), 0))
    grads = {"inputs": g.like(x)}
    grads.update({n: g.like(params[n]) for n in dg.FFN_PARAM_NAMES})
    dg.a2a_ffn_backward(x, params, saved, dY, workspace=ws, grads=grads)
    g.check(f"a2a_ffn {P, B, T, D, k}")


@pytest.mark.parametrize("P,B,T,D,k", [(2, 4, 16, 128, 2), (2, 3, 4, 144, 3), (4, 40, 16, 64, 2)])
def test_a2a_ffn_fp8_forward_writes_only_its_buffers(P, B, T, D, k):
    t = synth.ffn_inputs(P, B, T, D, k, seed=P * B + T + D + k, device=DEV)
    params = {n: t[n] for n in dg.FFN_PARAM_NAMES}
    x = t["inputs"]
    lib = _lib.load()
    sh = _lib.FFNShape(P, B, T, D, k, 1e-5)
    g = Guarded()
    packed = g.raw(lib.dg_a2a_ffn_fp8_weights_bytes(ctypes.byref(sh)))
    dg.a2a_ffn_fp8_pack_weights(params, P, B, T, D, packed=packed)
    ws = g.workspace(lib.dg_a2a_ffn_fp8_workspace_bytes(ctypes.byref(sh)))
    out = g.like(x)
    dg.a2a_ffn_forward_fp8(x, params, packed, workspace=ws, out=out)
    g.check(f"a2a_ffn_fp8 {P, B, T, D, k}")


@pytest.mark.parametrize("P,B,T,D", [(2, 4, 16, 128), (8, 3, 64, 24), (4, 1, 16, 8)])
def test_dispatch_combine_write_only_their_outputs(P, B, T, D):
    x = synth.ffn_grad_output(P, B, T, D, seed=3, device=DEV)
    lib = _lib.load()
    g = Guarded()
    L = T // P
    xl = g.tensor((P, P * B, L, D), torch.bfloat16)
    back = g.like(x)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.dg_a2a_dispatch(P, B, T, D, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(xl.data_ptr()), stream) == 0
    assert lib.dg_a2a_combine(P, B, T, D, ctypes.c_void_p(xl.data_ptr()), ctypes.c_void_p(back.data_ptr()), stream) == 0
    g.check(f"dispatch/combine {P, B, T, D}")
    assert torch.equal(back, x)


@pytest.mark.parametrize("S,d,ffn,W,bsz", [(256, 128, 512, 2, 1), (8 * 40, 136, 8 * 72, 8, 1), (512, 256, 1024, 4, 2)])
def test_tp_swiglu_forward_backward_write_only_their_buffers(S, d, ffn, W, bsz):
    xs, w13, w2 = synth.tp_swiglu_inputs(S, d, ffn, W, bsz=bsz, seed=S + d, device=DEV)
    dy = synth.tp_swiglu_inputs(S, d, ffn, W, bsz=bsz, seed=S + d + 1, device=DEV)[0]
    lib = _lib.load()
    g = Guarded()
    ws = g.workspace(lib.dg_tp_swiglu_workspace_bytes(S, d, ffn, W, bsz))
    y = g.like(xs)
    dg.tp_swiglu(xs, w13, w2, workspace=ws, out=y)
    bws = g.workspace(lib.dg_tp_swiglu_bwd_workspace_bytes(S, d, ffn, W, bsz))
    grads = dict(x=g.like(xs), w13=g.like(w13), w2=g.like(w2))
    dg.tp_swiglu_backward(xs, w13, w2, dy, workspace=bws, grads=grads)
    g.check(f"tp_swiglu {S, d, ffn, W, bsz}")


@pytest.mark.parametrize("rows,fin,fout", [(256, 128, 384), (160, 136, 192), (8, 8, 16)])
def test_tp_linear_forward_backward_write_only_their_outputs(rows, fin, fout):
    gen = torch.Generator(device=DEV)
    gen.manual_seed(rows + fin + fout)
    x = torch.randn(rows, fin, device=DEV, generator=gen).to(torch.bfloat16)
    w = (torch.rand(fout, fin, device=DEV, generator=gen) - 0.5).to(torch.bfloat16)
    b = (torch.rand(fout, device=DEV, generator=gen) - 0.5).to(torch.bfloat16)
    dy = torch.randn(rows, fout, device=DEV, generator=gen).to(torch.bfloat16)
    lib = _lib.load()
    g = Guarded()
    y = g.tensor((rows, fout), torch.bfloat16)
    dg.tp_linear(x, w, b, out=y)
    dx, dw, db = g.like(x), g.like(w), g.like(b)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    ws = g.workspace(256)
    st = lib.dg_tp_linear_bwd(rows, fin, fout, p(x), p(w), p(dy), p(dx), p(dw), p(db), p(ws), 256,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.dg_last_error()
    g.check(f"tp_linear {rows, fin, fout}")


@pytest.mark.parametrize("P,B,T,D,k", [(2, 4, 16, 128, 2), (2, 3, 4, 136, 3), (4, 40, 16, 64, 2)])
@pytest.mark.parametrize("flags", [0, dg.DG_FFN_COMP_ONLY, dg.DG_FFN_SEPARATE_GATE,
                                   dg.DG_FFN_COMP_ONLY | dg.DG_FFN_SEPARATE_GATE])
def test_a2a_ffn_inference_and_comp_only_write_only_their_buffers(P, B, T, D, k, flags):
    t = synth.ffn_inputs(P, B, T, D, k, seed=P + B + T + D + k + 1, device=DEV)
    params = {n: t[n] for n in dg.FFN_PARAM_NAMES}
    x = t["inputs"]
    lib = _lib.load()
    sh = _lib.FFNShape(P, B, T, D, k, 1e-5)
    g = Guarded()
    out = g.like(x)
    ws = g.workspace(lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 1, flags))
    dg.a2a_ffn_forward(x, params, out=out, inference=True, flags=flags, ws=ws)
    g.check(f"a2a_ffn inference {P, B, T, D, k} flags={flags}")
    if flags & dg.DG_FFN_COMP_ONLY:
        saved = g.raw(lib.dg_a2a_ffn_saved_bytes(ctypes.byref(sh)))
        fws = g.workspace(lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 0, flags))
        dg.a2a_ffn_forward(x, params, saved=saved, out=g.like(x), flags=flags, ws=fws)
        dY = synth.ffn_grad_output(P, B, T, D, seed=8, device=DEV)
        bws = g.workspace(lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), flags))
        grads = {"inputs": g.like(x)}
        grads.update({n: g.like(params[n]) for n in dg.FFN_PARAM_NAMES})
        dg.a2a_ffn_backward(x, params, saved, dY, workspace=bws, grads=grads, flags=flags)
        g.check(f"a2a_ffn comp_only backward {P, B, T, D, k}")
