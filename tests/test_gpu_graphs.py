"""The library's calls inside CUDA graphs: a captured step replays with new data
and gives bit-identical results to the same calls made eagerly (every path is
deterministic), so a caller can capture whole layers.  The first (eager) call of
each entry point does the per-device set-up (function attributes, occupancy),
which must happen before capture."""
import pytest
import torch

import expert_gemm_layers_gb300 as dg
from expert_gemm_layers_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _step(t):
    out = {}
    out["D"] = dg.gemm_fp8(t["A"], t["B"], t["C"], 0.5, 1.0, out=t["D"], ws=t["err"])
    y, saved = dg.a2a_ffn_forward(t["x"], t["params"], saved=t["saved"], out=t["out"], ws=t["err"])
    g = dg.a2a_ffn_backward(t["x"], t["params"], t["saved"], t["dY"], workspace=t["ws"], grads=t["grads"])
    dg.tp_swiglu(t["xs"], t["w13"], t["w2"], workspace=t["tp_ws"], out=t["y"])
    dg.tp_swiglu_backward(t["xs"], t["w13"], t["w2"], t["tp_dy"], workspace=t["tp_bws"], grads=t["tp_grads"])
    dg.tp_linear(t["xs"], t["wq"], t["bq"], out=t["q"])
    return out


def _tensors():
    import ctypes
    P, B, T, D, k = 2, 4, 16, 128, 2
    f = synth.ffn_inputs(P, B, T, D, k, seed=5, device=DEV, norm_affine="random")
    params = {n: f[n] for n in dg.FFN_PARAM_NAMES}
    lib = dg._lib.load()
    sh = dg.ffn_shape(P, B, T, D, k)
    A, Bm, C = synth.fp8_gemm_inputs(256, 512, 256, seed=6, device=DEV)
    xs, w13, w2 = synth.tp_swiglu_inputs(256, 128, 512, 4, seed=7, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(8)
    t = dict(A=A, B=Bm, C=C, D=torch.empty(256, 512, dtype=torch.bfloat16, device=DEV),
             x=f["inputs"], params=params, dY=synth.ffn_grad_output(P, B, T, D, seed=9, device=DEV),
             out=torch.empty_like(f["inputs"]),
             saved=torch.empty(lib.dg_a2a_ffn_saved_bytes(ctypes.byref(sh)), dtype=torch.uint8, device=DEV),
             ws=dg.alloc_workspace(lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), 0), DEV),
             grads={**{n: torch.empty_like(v) for n, v in params.items()}, "inputs": torch.empty_like(f["inputs"])},
             xs=xs, w13=w13, w2=w2, y=torch.empty_like(xs),
             tp_ws=dg.alloc_workspace(lib.dg_tp_swiglu_workspace_bytes(256, 128, 512, 4, 1), DEV),
             tp_dy=torch.randn(xs.shape, generator=g, device=DEV).to(torch.bfloat16),
             tp_bws=dg.alloc_workspace(lib.dg_tp_swiglu_bwd_workspace_bytes(256, 128, 512, 4, 1), DEV),
             err=dg.alloc_workspace(256, DEV),
             tp_grads=dict(x=torch.empty_like(xs), w13=torch.empty_like(w13), w2=torch.empty_like(w2)),
             wq=(torch.randn((384, 128), generator=g, device=DEV) / 12).to(torch.bfloat16),
             bq=torch.randn((384,), generator=g, device=DEV).to(torch.bfloat16))
    t["q"] = torch.empty((*xs.shape[:-1], 384), dtype=torch.bfloat16, device=DEV)
    return t


def _results(t):
    r = {"D": t["D"], "out": t["out"], "y": t["y"], "q": t["q"]}
    r.update({"g_" + n: v for n, v in t["grads"].items()})
    r.update({"tp_" + n: v for n, v in t["tp_grads"].items()})
    return {n: v.clone() for n, v in r.items()}


def test_captured_step_replays_bit_identical():
    t = _tensors()
    _step(t)                                   # eager warm-up: per-device set-up before capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            _step(t)
    torch.cuda.current_stream().wait_stream(side)
    # new data into the captured input tensors, then replay and compare with eager calls
    g = torch.Generator(device=DEV).manual_seed(21)
    for name in ("x", "dY", "xs", "tp_dy"):
        t[name].copy_(torch.randn(t[name].shape, generator=g, device=DEV).to(torch.bfloat16))
    t["C"].copy_(torch.randn(t["C"].shape, generator=g, device=DEV).to(torch.bfloat16))
    graph.replay()
    torch.cuda.synchronize()
    replayed = _results(t)
    _step(t)
    torch.cuda.synchronize()
    eager = _results(t)
    for name in eager:
        assert torch.equal(replayed[name], eager[name]), name
    for ws in (t["err"], t["ws"], t["tp_ws"], t["tp_bws"]):
        st, code = dg.device_status(workspace=ws)
        assert st == 0, hex(code)
