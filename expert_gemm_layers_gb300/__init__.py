"""dg: the local compute of expert- and tensor-parallel linear layers on one GB300.

Three operations, each a C-ABI entry point of libdg (include/dg.h) backed by
hand-written sm_103a kernels (tcgen05 UMMA with TMEM accumulators fed by
TMA/mbarrier pipelines):

* gemm_fp8      D = alpha * (A @ B^T) + beta * C, e4m3 inputs, bf16 output
* a2a_ffn       the all-to-all expert-parallel FFN layer (forward, backward,
                autograd), P logical ranks in one GPU's memory; a forward with
                both GEMMs on e4m3 operands (a2a_ffn_forward_fp8)
* tp_swiglu     the SwiGLU column/row-parallel pair over W shards (forward,
                backward, autograd)
* tp_linear     the attention projections (column-parallel QKV, row-parallel
                wo) over W shards (forward, backward, autograd)

The library is loaded lazily on first use and fails loudly if it is missing.
"""
from .ops import (A2AFFN, DG_FFN_COMP_ONLY, DG_FFN_FUSED_GATE, DG_FFN_SEPARATE_GATE, FFN_PARAM_NAMES, TPSwiGLU,
                  a2a_combine,
                  a2a_dispatch, a2a_ffn, a2a_ffn_backward, a2a_ffn_forward, a2a_ffn_forward_fp8,
                  a2a_ffn_fp8_pack_weights, alloc_workspace, debug_wait_timeout, device_status, error_block,
                  ffn_shape, gemm_fp8, tp_swiglu, tp_linear, tp_linear_backward, tp_linear_layer, TPLinear,
                  tp_swiglu_backward, tp_swiglu_layer, trace_begin, trace_end)

__all__ = [
    "A2AFFN", "DG_FFN_COMP_ONLY", "DG_FFN_FUSED_GATE", "DG_FFN_SEPARATE_GATE", "FFN_PARAM_NAMES", "a2a_combine",
    "a2a_dispatch",
    "a2a_ffn", "a2a_ffn_backward", "a2a_ffn_forward", "a2a_ffn_forward_fp8", "a2a_ffn_fp8_pack_weights",
    "alloc_workspace", "debug_wait_timeout", "device_status", "error_block", "ffn_shape", "gemm_fp8", "tp_swiglu",
    "tp_swiglu_backward", "TPSwiGLU", "tp_swiglu_layer", "tp_linear", "tp_linear_backward", "TPLinear",
    "tp_linear_layer", "trace_begin", "trace_end",
]
