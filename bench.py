#!/usr/bin/env python
"""Benchmark of the dg hot path: one JSON line on rank 0.

A step is one pass of the whole path over one batch of seeded synthetic input:
  1. FP8 GEMM D = 0.5*(A @ B^T) + C, M = N = K = 4096 (e4m3 in, bf16 out)
  2. A2A FFN layer forward + backward, P=8 ranks, B=512, T=64, D=1280, k=6
  3. TP SwiGLU pair, 8 shards, S=8192, d=4096, ffn=14336
The metric is TFLOP/s over GEMM FLOPs (2*M*N*K per problem; the backward
counts its own GEMMs).  Every input is far larger than L2 per step (the FFN
weights alone are 3.8 GB), so L2 holds nothing from one use of an operand
to its next.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dg|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas: the path needs no exchange between GPUs); value sums the ranks'
work over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FP8 = dict(M=4096, N=4096, K=4096, alpha=0.5, beta=1.0, seed=1)
FFN = dict(P=8, B=512, T=64, D=1280, k=6, seed=42, dy_seed=43)
TP = dict(S=8192, d=4096, ffn=14336, W=8, seed=7)
ATTN = dict(qkv_out=4096 + 2 * 1024)  # fused QKV rows of Llama-3-8B: 32 query + 2 x 8 key/value heads of 128

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
# GB300 nominal dense tensor rates (TFLOP/s; the vendor's figures without 2:4
# sparsity), the second denominator of each part.
NOMINAL_TFLOPS = {"bf16": 2250.0, "fp8": 4500.0}
FALLBACK_PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)

# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of each kernel of the FFN layer at T=8 token positions (an
# eighth of the benchmark's problems; traffic grows in proportion, so it is
# scaled by 8), with the sha256 of the kernel's sources (for a GEMM also the
# launch code, which picks its tile order) at capture time; a kernel whose
# sources changed since reports null.  The capture's summary is committed with
# the other ncu summaries of this repository.
TRAFFIC = {
    "ffn_gemm1": {"bytes_per_launch": 8 * 1.386602e+09, "sources": ["expert_gemm_layers_gb300/csrc/dg_gemm.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh", "expert_gemm_layers_gb300/csrc/dg_gemm_bf16_km_lnstats.cu", "expert_gemm_layers_gb300/csrc/dg_api.cu"], "sha256": "07b159e4bbb09f23988902b0bf077ef8b80bf25753960ae9df865d51fe835018"},
    "ffn_ln_stats": {"bytes_per_launch": 8 * 3.147341e+07, "sources": ["expert_gemm_layers_gb300/csrc/dg_rowops.cu", "expert_gemm_layers_gb300/csrc/dg_gate.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh"], "sha256": "34454a0547e4ce1103037b8d8921ba87fd8ba11de4a1f897e625b5b5d8c168bf"},
    "ffn_gemm2_gated": {"bytes_per_launch": 8 * 1.573366e+09, "sources": ["expert_gemm_layers_gb300/csrc/dg_gemm_gated.cu", "expert_gemm_layers_gb300/csrc/dg_gate.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh", "expert_gemm_layers_gb300/csrc/dg_api.cu"], "sha256": "c3cf68bbbb7cd6b7f06a5b36ba41ec9dbbced9bfb478687bf7ed3481c1a5d275"},
    "ffn_gemm2_rest": {"bytes_per_launch": 8 * 7.040044e+08, "sources": ["expert_gemm_layers_gb300/csrc/dg_gemm.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh", "expert_gemm_layers_gb300/csrc/dg_gemm_bf16_km_bias.cu", "expert_gemm_layers_gb300/csrc/dg_api.cu"], "sha256": "dde9856cb24d1e3024b1048dc8e39beee94f6dec81c34cbc31c4fff404065c8a"},
    "ffn_bwd_dhl": {"bytes_per_launch": 8 * 6.894607e+08, "sources": ["expert_gemm_layers_gb300/csrc/dg_gemm.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh", "expert_gemm_layers_gb300/csrc/dg_gemm_bf16_kk_store.cu", "expert_gemm_layers_gb300/csrc/dg_api.cu"], "sha256": "efe94c9ca71d215ebdd5e913e5138fef6ff3499d726d470b4b62b71e9d1aa699"},
    "ffn_bwd_dwout": {"bytes_per_launch": 8 * 7.436754e+08, "sources": ["expert_gemm_layers_gb300/csrc/dg_gemm.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh", "expert_gemm_layers_gb300/csrc/dg_gemm_bf16_mm_store.cu", "expert_gemm_layers_gb300/csrc/dg_api.cu"], "sha256": "b1b66f1d79739eea6a711feb91d7f7b1457367056fea15b1edada529e34530cc"},
    "ffn_bwd_dbout": {"bytes_per_launch": 8 * 8.392038e+07, "sources": ["expert_gemm_layers_gb300/csrc/dg_rowops.cu", "expert_gemm_layers_gb300/csrc/dg_gate.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh"], "sha256": "34454a0547e4ce1103037b8d8921ba87fd8ba11de4a1f897e625b5b5d8c168bf"},
    "ffn_bwd_ln_rowsum": {"bytes_per_launch": 8 * 1.512565e+09, "sources": ["expert_gemm_layers_gb300/csrc/dg_rowops.cu", "expert_gemm_layers_gb300/csrc/dg_gate.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh"], "sha256": "34454a0547e4ce1103037b8d8921ba87fd8ba11de4a1f897e625b5b5d8c168bf"},
    "ffn_bwd_ln_apply": {"bytes_per_launch": 8 * 2.527671e+09, "sources": ["expert_gemm_layers_gb300/csrc/dg_rowops.cu", "expert_gemm_layers_gb300/csrc/dg_gate.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh"], "sha256": "34454a0547e4ce1103037b8d8921ba87fd8ba11de4a1f897e625b5b5d8c168bf"},
    "ffn_bwd_grad_reduce": {"bytes_per_launch": 8 * 4.725248e+07, "sources": ["expert_gemm_layers_gb300/csrc/dg_rowops.cu", "expert_gemm_layers_gb300/csrc/dg_gate.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh"], "sha256": "34454a0547e4ce1103037b8d8921ba87fd8ba11de4a1f897e625b5b5d8c168bf"},
    "ffn_bwd_dx": {"bytes_per_launch": 8 * 1.848908e+09, "sources": ["expert_gemm_layers_gb300/csrc/dg_gemm.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh", "expert_gemm_layers_gb300/csrc/dg_gemm_bf16_kk_store.cu", "expert_gemm_layers_gb300/csrc/dg_api.cu"], "sha256": "efe94c9ca71d215ebdd5e913e5138fef6ff3499d726d470b4b62b71e9d1aa699"},
    "ffn_bwd_dw1": {"bytes_per_launch": 8 * 1.415758e+09, "sources": ["expert_gemm_layers_gb300/csrc/dg_gemm.cuh", "expert_gemm_layers_gb300/csrc/dg_ptx.cuh", "expert_gemm_layers_gb300/csrc/dg_gemm_bf16_mm_store.cu", "expert_gemm_layers_gb300/csrc/dg_api.cu"], "sha256": "b1b66f1d79739eea6a711feb91d7f7b1457367056fea15b1edada529e34530cc"},
}


def traffic_for(kernel: str):
    import hashlib
    t = TRAFFIC.get(kernel)
    if not t:
        return None
    h = hashlib.sha256()
    for f in t["sources"]:
        try:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        except OSError:
            return None
    return t["bytes_per_launch"] if h.hexdigest() == t["sha256"] else None


def gemm_flops():
    f = {}
    f["fp8_gemm"] = 2.0 * FP8["M"] * FP8["N"] * FP8["K"]
    P, B, T, D, k = FFN["P"], FFN["B"], FFN["T"], FFN["D"], FFN["k"]
    H, M = D * k, P * B
    fwd = T * (2.0 * M * D * 2 * H + 2.0 * M * H * D)
    f["ffn_fwd"] = fwd
    f["ffn_bwd"] = 2.0 * fwd      # dHl, dwout, dX, dw1
    S, d, ffn = TP["S"], TP["d"], TP["ffn"]
    f["tp_swiglu"] = 2.0 * S * d * 2 * ffn + 2.0 * S * ffn * d
    return f


def load_peaks():
    try:
        with open(MEASURED_PEAKS) as fh:
            p = json.load(fh)
        out = dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                   bf16_tflops_sustained=float(p["bf16_tflops_sustained"]), source="measured")
        mhz = (p.get("clocks_under_load") or {}).get("sm_mhz_median")
        if mhz:
            out["sustained_sm_mhz"] = float(mhz)  # median SM clock of the sustained measurement
        return out
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- workload

class Workload:
    """Device buffers of one step, inputs drawn once from the seeded generators."""

    def __init__(self, dev):
        import torch

        import expert_gemm_layers_gb300 as dg
        from expert_gemm_layers_gb300 import synth
        self.dg, self.torch, self.dev = dg, torch, dev
        bf = torch.bfloat16
        self.A, self.B, self.C = synth.fp8_gemm_inputs(FP8["M"], FP8["N"], FP8["K"], seed=FP8["seed"], device=dev)
        self.D = torch.empty((FP8["M"], FP8["N"]), dtype=bf, device=dev)
        P, B, T, D, k = FFN["P"], FFN["B"], FFN["T"], FFN["D"], FFN["k"]
        t = synth.ffn_inputs(P, B, T, D, k, seed=FFN["seed"], device=dev)
        self.x = t["inputs"]
        self.params = {n: t[n] for n in dg.FFN_PARAM_NAMES}
        self.dY = synth.ffn_grad_output(P, B, T, D, seed=FFN["dy_seed"], device=dev)
        self.out = torch.empty_like(self.x)
        sh = dg.ffn_shape(P, B, T, D, k)
        lib = dg._lib.load()
        import ctypes
        self.saved = torch.empty(lib.dg_a2a_ffn_saved_bytes(ctypes.byref(sh)), dtype=torch.uint8, device=dev)
        self.ws = dg.alloc_workspace(lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), 0), dev)
        self.grads = {n: torch.empty_like(v) for n, v in self.params.items()}
        self.grads["inputs"] = torch.empty_like(self.x)
        self.xs, self.w13, self.w2 = synth.tp_swiglu_inputs(TP["S"], TP["d"], TP["ffn"], TP["W"], seed=TP["seed"],
                                                            device=dev)
        self.y = torch.empty_like(self.xs)
        self.tp_ws = dg.alloc_workspace(lib.dg_tp_swiglu_workspace_bytes(TP["S"], TP["d"], TP["ffn"], TP["W"], 1),
                                        dev)
        # the TP SwiGLU backward, timed on its own after the step
        self.tp_dy = synth.tp_swiglu_inputs(TP["S"], TP["d"], TP["ffn"], TP["W"], seed=TP["seed"] + 1,
                                            device=dev)[0]
        self.tp_bws = dg.alloc_workspace(
            lib.dg_tp_swiglu_bwd_workspace_bytes(TP["S"], TP["d"], TP["ffn"], TP["W"], 1), dev)
        self.tp_grads = dict(x=torch.empty_like(self.xs), w13=torch.empty_like(self.w13), w2=torch.empty_like(self.w2))
        # attention projections at the same Llama-3-8B shape (32 query / 8 key-value heads of 128), no bias
        S, W, d = TP["S"], TP["W"], TP["d"]
        gen = torch.Generator(device=dev).manual_seed(TP["seed"] + 2)
        self.attn_x = torch.randn((W, 1, S // W, d), generator=gen, device=dev).to(bf)
        self.wqkv = ((torch.rand((ATTN["qkv_out"], d), generator=gen, device=dev) - 0.5) * (2 / d ** 0.5)).to(bf)
        self.attn_a = torch.randn((W, 1, S // W, d), generator=gen, device=dev).to(bf)
        self.wo = ((torch.rand((d, d), generator=gen, device=dev) - 0.5) * (2 / d ** 0.5)).to(bf)
        self.qkv = torch.empty((W, 1, S // W, ATTN["qkv_out"]), dtype=bf, device=dev)
        self.attn_y = torch.empty((W, 1, S // W, d), dtype=bf, device=dev)
        self.dqkv = torch.randn_like(self.qkv, dtype=torch.float32).to(bf)
        self.dattn_y = torch.randn_like(self.attn_y, dtype=torch.float32).to(bf)

    def status(self):
        """Reads and clears the error word of every workspace the step uses: (status, raw code)."""
        for ws in (None, self.ws, self.tp_ws, self.tp_bws):
            st, code = self.dg.device_status(self.dev, workspace=ws)
            if st != 0:
                return st, code
        return 0, 0

    def step(self, marks=None):
        dg = self.dg
        dg.gemm_fp8(self.A, self.B, self.C, FP8["alpha"], FP8["beta"], out=self.D)
        if marks is not None:
            marks[0].record()
        dg.a2a_ffn_forward(self.x, self.params, saved=self.saved, out=self.out)
        if marks is not None:
            marks[1].record()
        dg.a2a_ffn_backward(self.x, self.params, self.saved, self.dY, workspace=self.ws, grads=self.grads)
        if marks is not None:
            marks[2].record()
        dg.tp_swiglu(self.xs, self.w13, self.w2, workspace=self.tp_ws, out=self.y)

    def parts(self):
        """The step as (name, inputs read, outputs written, call) in launch order; the
        names are those of the streamed tensors."""
        dg = self.dg
        return [
            ("fp8_gemm", ("A", "B", "C"), ("D",),
             lambda: dg.gemm_fp8(self.A, self.B, self.C, FP8["alpha"], FP8["beta"], out=self.D)),
            ("ffn_fwd", ("x",), ("out",),
             lambda: dg.a2a_ffn_forward(self.x, self.params, saved=self.saved, out=self.out)),
            ("ffn_bwd", ("x", "dY"), ("d_inputs",),
             lambda: dg.a2a_ffn_backward(self.x, self.params, self.saved, self.dY, workspace=self.ws,
                                         grads=self.grads)),
            ("tp_swiglu", ("xs",), ("y",),
             lambda: dg.tp_swiglu(self.xs, self.w13, self.w2, workspace=self.tp_ws, out=self.y)),
        ]

    def attn_proj(self):
        dg = self.dg
        dg.tp_linear(self.attn_x, self.wqkv, out=self.qkv)
        dg.tp_linear(self.attn_a, self.wo, out=self.attn_y)
        dg.tp_linear_backward(self.attn_a, self.wo, self.dattn_y)
        dg.tp_linear_backward(self.attn_x, self.wqkv, self.dqkv)

    def tp_backward(self):
        self.dg.tp_swiglu_backward(self.xs, self.w13, self.w2, self.tp_dy, workspace=self.tp_bws,
                                   grads=self.tp_grads)


# ---------------------------------------------------------------- oracle sample

class OracleSample:
    """A bounded sample of the same workload run by the CPU oracle (fp64 numpy).

    Per step: rows 0-255 of the FP8 GEMM; 256 FFN output rows, 64 from each of
    4 seeded token positions; 64 rows of d_inputs, 32 from each of 2 seeded
    token positions; 32 seeded rows of the TP SwiGLU output.  Its FLOPs are the
    GEMM FLOPs of exactly those rows.  The oracle decodes the weights of every
    problem it touches once per call, so the rows are grouped into few
    problems to keep that decode a small part of the sample; decode_seconds()
    times those decodes alone.
    """

    def __init__(self, host):
        import oracle as O
        self.O = O
        self.h = host
        rng = np.random.default_rng(0)
        P, B, T, D, k = FFN["P"], FFN["B"], FFN["T"], FFN["D"], FFN["k"]
        M = P * B
        self.sh = O.FFNShape(P, B, T, D, k)
        self.fp8_rows = np.arange(256)
        self.ffn_t = rng.choice(T, size=4, replace=False)
        self.ffn_rows = np.concatenate([rng.choice(M, size=64, replace=False) * T + t for t in self.ffn_t])
        self.dx_t = rng.choice(T, size=2, replace=False)
        self.dx_rows = np.concatenate([rng.choice(M, size=32, replace=False) * T + t for t in self.dx_t])
        self.tp_rows = rng.choice(TP["S"], size=32, replace=False)
        H = D * k
        row_fwd = 2.0 * D * 2 * H + 2.0 * H * D
        self.flops = (2.0 * len(self.fp8_rows) * FP8["N"] * FP8["K"] + len(self.ffn_rows) * row_fwd
                      + len(self.dx_rows) * (row_fwd + 2.0 * H * D + 2.0 * 2 * H * D)
                      + len(self.tp_rows) * (2.0 * TP["d"] * 2 * TP["ffn"] + 2.0 * TP["ffn"] * TP["d"]))
        self.desc = ("per step: FP8 GEMM rows 0-255 of 4096; 256 FFN output rows (64 from each of 4 seeded token "
                     "positions); 64 d_inputs rows (32 from each of 2 seeded token positions); 32 seeded TP SwiGLU "
                     "rows (GEMM FLOPs of those rows only)")

    def step(self):
        O, h = self.O, self.h
        O.gemm_fp8(h["A"], h["B"], h["C"], FP8["alpha"], FP8["beta"], rows=self.fp8_rows)
        O.ffn_forward_rows(self.sh, h["inputs"], h, self.ffn_rows)
        O.ffn_backward_dx_rows(self.sh, h["inputs"], h, h["dY"], self.dx_rows)
        O.tp_swiglu_rows(h["xs"], h["w13"], h["w2"], TP["W"], self.tp_rows)

    def decode_seconds(self):
        """Time of the exact decodes of the operands one step touches (part of step())."""
        O, h = self.O, self.h
        sh = self.sh
        P, L, D, H = sh.P, sh.L, sh.D, sh.H
        t0 = time.perf_counter()
        O.e4m3_to_f64(h["B"])
        O.e4m3_to_f64(np.asarray(h["A"]).reshape(FP8["M"], FP8["K"])[self.fp8_rows])
        for t in list(self.ffn_t) + list(self.dx_t):
            r, l = divmod(int(t), L)
            O.bf16_to_f64(np.asarray(h["w1"]).reshape(P, L, D, 2 * H)[r, l])
            O.bf16_to_f64(np.asarray(h["wout"]).reshape(P, L, H, D)[r, l])
        O.bf16_to_f64(h["w13"])
        O.bf16_to_f64(h["w2"])
        return time.perf_counter() - t0


def host_bits(w):
    from expert_gemm_layers_gb300 import synth
    h = dict(A=synth.bits(w.A), B=synth.bits(w.B), C=synth.bits(w.C), inputs=synth.bits(w.x), dY=synth.bits(w.dY),
             xs=synth.bits(w.xs), w13=synth.bits(w.w13), w2=synth.bits(w.w2))
    for n, v in w.params.items():
        h[n] = synth.bits(v)
    return h


def time_oracle(sample, steps, warmup=0):
    for _ in range(warmup):
        sample.step()
    t0 = time.perf_counter()
    for _ in range(steps):
        sample.step()
    return (time.perf_counter() - t0) / steps


def oracle_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- arms

def run_reference(args, rank, world):
    """The oracle as the reference arm: rank 0 only, host cores only."""
    if rank != 0:
        return
    import torch
    from expert_gemm_layers_gb300 import synth

    class HostWorkload:
        pass

    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    w = HostWorkload()
    w.A, w.B, w.C = synth.fp8_gemm_inputs(FP8["M"], FP8["N"], FP8["K"], seed=FP8["seed"], device=dev)
    t = synth.ffn_inputs(FFN["P"], FFN["B"], FFN["T"], FFN["D"], FFN["k"], seed=FFN["seed"], device=dev)
    w.x = t["inputs"]
    w.params = {n: t[n] for n in ("w1", "b1", "wout", "bout", "nx_w", "nx_b", "ng_w", "ng_b")}
    w.dY = synth.ffn_grad_output(FFN["P"], FFN["B"], FFN["T"], FFN["D"], seed=FFN["dy_seed"], device=dev)
    w.xs, w.w13, w.w2 = synth.tp_swiglu_inputs(TP["S"], TP["d"], TP["ffn"], TP["W"], seed=TP["seed"], device=dev)
    h = host_bits(w)
    del w, t
    sample = OracleSample(h)
    sec = time_oracle(sample, args.steps, args.warmup)
    value = sample.flops / sec / 1e12
    cores = oracle_threads()
    line = {
        "impl": "reference", "metric": "hot-path GEMM TFLOP/s (FP8 GEMM + A2A FFN fwd+bwd + TP SwiGLU)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": workload_config(),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample.desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config():
    return {"workload": "fp8_gemm_4096^3 + a2a_ffn_fwd_bwd(P=8,B=512,T=64,D=1280,k=6) + "
                        "tp_swiglu(S=8192,d=4096,ffn=14336,W=8)",
            "fp8_gemm": "M=N=K=4096, alpha=0.5, beta=1, seed 1",
            "a2a_ffn": "P=8, B=512, T=64, D=1280, k=6, H=7680, L=8, seed 42 (+rank), dY seed 43",
            "tp_swiglu": "S=8192, d=4096, ffn=14336, W=8, bsz=1, seed 7",
            "l2": "inputs larger than L2 (5.2 GB of operands per step; no L2 flush)"}


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (all ranks get it); the identity on one rank."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_tflops(world: int, step_flops: float, ms: float) -> float:
    """Whole-job throughput: every rank's step of work over the slowest rank's step time."""
    return world * step_flops / (ms * 1e-3) / 1e12


def run_dg(args, rank, world):
    import torch
    import torch.distributed as dist

    import expert_gemm_layers_gb300 as dg
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = Workload(dev)
    flops = gemm_flops()
    step_flops = sum(flops.values())
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        w.step()
    torch.cuda.synchronize(dev)
    st, code = w.status()
    if st != 0:
        raise RuntimeError(f"device error word after warm-up: {code:#x}")

    def barrier():
        if world > 1:
            dist.barrier()

    # Per-kernel table from two fully traced steps before the timed region:
    # every launch bracketed by events (which costs each kernel its
    # programmatic-launch overlap with its neighbours, so not while timing).
    dg.trace_begin()
    for _ in range(2):
        w.step()
    torch.cuda.synchronize(dev)
    table = dg.trace_end()
    top_name = max(table, key=lambda e: e["total_ms"])["name"]
    launches_per_step = sum(e["launches"] for e in table) / 2

    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    dg.trace_begin(only=top_name)  # the dominant kernel's launches, timed inside the timed region
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        w.step(marks[i])
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    trace = dg.trace_end()
    clk = clocks.stop()
    barrier()
    ms = max_over_ranks(t_start.elapsed_time(t_end) / args.steps, world, dev)
    st, code = w.status()
    if st != 0:
        raise RuntimeError(f"device error word after the timed steps: {code:#x}")

    step_ms = [starts[i].elapsed_time(ends[i]) for i in range(args.steps)]
    part_ms = {"fp8_gemm": [], "ffn_fwd": [], "ffn_bwd": [], "tp_swiglu": []}
    for i in range(args.steps):
        m = marks[i]
        part_ms["fp8_gemm"].append(starts[i].elapsed_time(m[0]))
        part_ms["ffn_fwd"].append(m[0].elapsed_time(m[1]))
        part_ms["ffn_bwd"].append(m[1].elapsed_time(m[2]))
        part_ms["tp_swiglu"].append(m[2].elapsed_time(ends[i]))

    peaks = load_peaks()
    run_mhz = (clk or {}).get("sm_mhz")
    parts = {}
    for name, vals in part_ms.items():
        pm = statistics.mean(vals)
        tf = flops[name] / (pm * 1e-3) / 1e12
        peak = (2.0 * peaks["bf16_tflops"]) if name == "fp8_gemm" else peaks["bf16_tflops"]
        nominal = NOMINAL_TFLOPS["fp8" if name == "fp8_gemm" else "bf16"]
        parts[name] = {"ms": round(pm, 4), "ms_min": round(min(vals), 4), "ms_max": round(max(vals), 4),
                       "tflops": round(tf, 2), "peak_tflops": peak, "frac_of_peak": round(tf / peak, 4),
                       "frac_of_nominal": round(tf / nominal, 4)}
        if run_mhz and peaks.get("sustained_sm_mhz"):
            # the measured sustained rate per MHz of its own clock, at the clock the step ran at
            at_clock = peaks["bf16_tflops_sustained"] * (2.0 if name == "fp8_gemm" else 1.0) * run_mhz / \
                peaks["sustained_sm_mhz"]
            parts[name]["frac_of_sustained_at_run_clock"] = round(tf / at_clock, 4)
    parts["fp8_gemm"]["peak_note"] = "2 x measured bf16 burst (nominal fp8:bf16 ratio 2)"

    # roofline of the dominant kernel (largest share of device time in the traced steps)
    top = trace[0]
    per_launch_ms = top["total_ms"] / top["launches"]
    if top["flops"] > 0:
        achieved = top["flops"] / top["launches"] / (per_launch_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops_sustained"] * (2.0 if top["name"].startswith("gemm_fp8") else 1.0)
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4)}
    else:
        achieved = top["bytes"] / top["launches"] / (per_launch_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4)}
    roof["kernel"] = top["name"]
    roof["peak_source"] = peaks["source"] + (" sustained bf16" if top["flops"] > 0 else " HBM copy")
    roof["traffic"] = traffic_for(top["name"])
    if roof["traffic"] is not None:
        roof["traffic_source"] = "ncu dram__bytes_read+write of the kernel at T=8 token positions, scaled x8"
    roof["launches_timed"] = top["launches"]
    total_ms = sum(e["total_ms"] for e in table)
    kernel_table = {e["name"]: {"launches_per_step": e["launches"] // 2,
                                "ms_per_launch": round(e["total_ms"] / e["launches"], 4),
                                "share": round(e["total_ms"] / total_ms, 4)} for e in table}
    launches = int(launches_per_step * args.steps)

    # end to end: inputs from pinned host memory in, results back to pinned
    # host memory; right after the device-timed steps, in the same state of the GPU
    # (with its own clock record: it runs after the device-timed steps, and at
    # the power cap the SM clock can differ between the two)
    e2e_clocks = ClockSampler(local)
    e2e_clocks.start()
    e2e = run_e2e(w, args, dev, step_flops, world)
    e2e["clocks"] = e2e_clocks.stop()

    # outside the step: the FP8 GEMM alone (L2 flushed before each launch),
    # the TP SwiGLU backward (recompute [a|b], dh, gate backward, dw2, dX,
    # dw13), the attention projections, the e4m3 FFN forward, the FFN forward
    # variants and the tiny workload's latency
    extra = {}
    if not args.step_only:
        extra = run_fp8_alone(w, args, dev, peaks)
        extra.update(run_tp_backward(w, args, dev, peaks))
        extra.update(run_attn_proj(w, args, dev, peaks))
        extra.update(run_ffn_fp8(w, args, dev, peaks))
        extra.update(run_ffn_forward_variants(w, args, dev, peaks))
        extra.update(run_tiny_latency(args, dev))

    value = job_tflops(world, step_flops, ms)
    line = {
        "metric": "hot-path GEMM TFLOP/s (FP8 GEMM + A2A FFN fwd+bwd + TP SwiGLU)",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "ms_per_step_min": round(min(step_ms), 4), "ms_per_step_max": round(max(step_ms), 4),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16+e4m3 (fp32 accumulate)", "data": "synthetic",
        "config": workload_config(),
        "parts": dict(parts, **({"ffn_tiny_latency": extra["ffn_tiny_latency"]} if "ffn_tiny_latency" in extra else {})),
        "roofline": roof, "kernels": kernel_table,
        "gpu_launches": launches, "e2e": e2e, "clocks": clk, "outside_step": extra,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = OracleSample(host_bits(w))
        sec = time_oracle(sample, 1)
        dec = sample.decode_seconds()
        line["cpu_baseline"] = {"value": round(sample.flops / sec / 1e12, 6), "unit": "TFLOP/s",
                                "cores": oracle_threads(), "kind": "oracle", "sample": sample.desc,
                                "seconds": round(sec, 2), "decode_seconds": round(dec, 2),
                                "arith_tflops": round(sample.flops / max(sec - dec, 1e-9) / 1e12, 6)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_fp8_alone(w, args, dev, peaks):
    """The 4096^3 FP8 GEMM timed launch by launch, L2 flushed before each (its
    100 MB of operands would otherwise stay in the 129 MB L2)."""
    import torch
    dg = w.dg
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    iters = 30
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    dg.trace_begin()  # only to learn which tile variant the launch picks
    for _ in range(3):
        dg.gemm_fp8(w.A, w.B, w.C, FP8["alpha"], FP8["beta"], out=w.D)
    torch.cuda.synchronize(dev)
    trace = dg.trace_end()
    for e0, e1 in ev:
        flush.zero_()
        flush_sum = flush.sum()  # read back: the L2 holds clean lines of the flush buffer
        e0.record(stream)
        dg.gemm_fp8(w.A, w.B, w.C, FP8["alpha"], FP8["beta"], out=w.D)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    del flush_sum
    st, code = w.status()
    if st != 0:
        raise RuntimeError(f"device error word after the FP8 GEMM: {code:#x}")
    ms = sorted(e0.elapsed_time(e1) for e0, e1 in ev)
    med = ms[len(ms) // 2]
    flops = 2.0 * FP8["M"] * FP8["N"] * FP8["K"]
    peak = 2.0 * peaks["bf16_tflops"]
    tf = flops / (med * 1e-3) / 1e12
    return {"fp8_gemm_alone": {
        "ms_median": round(med, 4), "ms_min": round(ms[0], 4), "tflops": round(tf, 2), "peak_tflops": peak,
        "frac_of_peak": round(tf / peak, 4), "iters": iters,
        "l2": "flushed before each launch (256 MB written, then read back)",
        "peak_note": "2 x measured bf16 burst (nominal fp8:bf16 ratio 2)",
        "kernel": [e["name"] for e in trace]}}


def run_tp_backward(w, args, dev, peaks):
    """The TP SwiGLU backward at the forward's shape, timed alone (not part of the step)."""
    import torch
    dg = w.dg
    for _ in range(max(args.warmup, 2)):
        w.tp_backward()
    iters = 5
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize(dev)
    dg.trace_begin()
    ev[0].record(stream)
    for _ in range(iters):
        w.tp_backward()
    ev[1].record(stream)
    torch.cuda.synchronize(dev)
    trace = dg.trace_end()
    st, code = w.status()
    if st != 0:
        raise RuntimeError(f"device error word after the TP backward: {code:#x}")
    ms = ev[0].elapsed_time(ev[1]) / iters
    R, d, ffn = TP["S"], TP["d"], TP["ffn"]
    flops = 16.0 * R * d * ffn  # [a|b] 4, dh 2, dw2 2, dX 4, dw13 4 (x R*d*ffn)
    tf = flops / (ms * 1e-3) / 1e12
    return {"tp_swiglu_bwd": {
        "ms": round(ms, 4), "tflops": round(tf, 2), "peak_tflops": peaks["bf16_tflops"],
        "frac_of_peak": round(tf / peaks["bf16_tflops"], 4), "iters": iters,
        "kernels": {e["name"]: {"launches": e["launches"], "ms_per_launch": round(e["total_ms"] / e["launches"], 4)}
                    for e in trace}}}


def run_ffn_fp8(w, args, dev, peaks):
    """The FFN forward with both GEMMs on e4m3 operands at the step's shape
    (outside the step; weights packed once, before timing)."""
    import torch
    dg = w.dg
    P, B, T, D = FFN["P"], FFN["B"], FFN["T"], FFN["D"]
    packed = dg.a2a_ffn_fp8_pack_weights(w.params, P, B, T, D)
    out = torch.empty_like(w.out)
    lib = dg._lib.load()
    import ctypes
    ws = dg.alloc_workspace(lib.dg_a2a_ffn_fp8_workspace_bytes(ctypes.byref(dg.ffn_shape(P, B, T, D, FFN["k"]))),
                            dev)
    run = lambda: dg.a2a_ffn_forward_fp8(w.x, w.params, packed, workspace=ws, out=out)
    for _ in range(max(args.warmup, 2)):
        run()
    iters = 5
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize(dev)
    dg.trace_begin()
    ev[0].record(stream)
    for _ in range(iters):
        run()
    ev[1].record(stream)
    torch.cuda.synchronize(dev)
    trace = dg.trace_end()
    st, code = dg.device_status(dev, workspace=ws)
    if st != 0:
        raise RuntimeError(f"device error word after the FP8 FFN forward: {code:#x}")
    ms = ev[0].elapsed_time(ev[1]) / iters
    flops = gemm_flops()["ffn_fwd"]
    tf = flops / (ms * 1e-3) / 1e12
    peak = 2.0 * peaks["bf16_tflops"]
    return {"ffn_fwd_fp8": {
        "ms": round(ms, 4), "tflops": round(tf, 2), "peak_tflops": peak, "frac_of_peak": round(tf / peak, 4),
        "peak_note": "2 x measured bf16 burst (nominal fp8:bf16 ratio 2)", "iters": iters,
        "kernels": {e["name"]: {"launches": e["launches"], "ms_per_launch": round(e["total_ms"] / e["launches"], 4)}
                    for e in trace}}}


def _timed(run, iters, dev):
    """Mean device time (ms) of `iters` back-to-back calls, and the kernel table of those calls."""
    import torch
    from expert_gemm_layers_gb300 import trace_begin, trace_end
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize(dev)
    ev[0].record(stream)
    for _ in range(iters):
        run()
    ev[1].record(stream)
    torch.cuda.synchronize(dev)
    ms = ev[0].elapsed_time(ev[1]) / iters
    trace_begin()
    run()
    torch.cuda.synchronize(dev)
    table = trace_end()
    return ms, {e["name"]: round(e["total_ms"] / e["launches"], 4) for e in table}


def run_ffn_forward_variants(w, args, dev, peaks):
    """The FFN forward at the step's shape in four forms, timed alone (outside
    the step, same box and run): training with the normalise-and-gate computed
    by the second GEMM's producer warps (the default, as in the step) and with
    the separate pass through HBM; inference (nothing saved) in both forms."""
    import ctypes
    dg = w.dg
    lib = dg._lib.load()
    sh = dg.ffn_shape(FFN["P"], FFN["B"], FFN["T"], FFN["D"], FFN["k"])
    ws_inf = dg.alloc_workspace(lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 1, 0), dev)
    ws_inf_sep = dg.alloc_workspace(
        lib.dg_a2a_ffn_fwd_workspace_bytes(ctypes.byref(sh), 1, dg.DG_FFN_SEPARATE_GATE), dev)
    variants = {
        "fused_gate": lambda: dg.a2a_ffn_forward(w.x, w.params, saved=w.saved, out=w.out),
        "separate_gate": lambda: dg.a2a_ffn_forward(w.x, w.params, saved=w.saved, out=w.out,
                                                    flags=dg.DG_FFN_SEPARATE_GATE),
        "inference_fused_gate": lambda: dg.a2a_ffn_forward(w.x, w.params, out=w.out, inference=True, ws=ws_inf),
        "inference_separate_gate": lambda: dg.a2a_ffn_forward(w.x, w.params, out=w.out, inference=True,
                                                              ws=ws_inf_sep, flags=dg.DG_FFN_SEPARATE_GATE),
    }
    flops = gemm_flops()["ffn_fwd"]
    res = {}
    for _ in range(2):                                    # two rounds, alternating the variants
        for name, run in variants.items():
            run()
            ms, kernels = _timed(run, 5, dev)
            tf = flops / (ms * 1e-3) / 1e12
            prev = res.get(name)
            if prev is None or ms < prev["ms"]:
                res[name] = {"ms": round(ms, 4), "tflops": round(tf, 2), "peak_tflops": peaks["bf16_tflops"],
                             "frac_of_peak": round(tf / peaks["bf16_tflops"], 4), "kernels_ms": kernels}
    for wsx in (ws_inf, ws_inf_sep):
        st, code = dg.device_status(dev, workspace=wsx)
        if st != 0:
            raise RuntimeError(f"device error word after the FFN forward variants: {code:#x}")
    st, code = w.status()
    if st != 0:
        raise RuntimeError(f"device error word after the FFN forward variants: {code:#x}")
    del ws_inf, ws_inf_sep
    return {"ffn_fwd_variants": dict(res, note="best of two rounds of 5 back-to-back calls each")}


def run_tiny_latency(args, dev):
    """Latency of the tiny A2A FFN workload (P=2, B=4, T=16, D=128, k=2, seed 42):
    device time of each forward and each forward + backward call, in microseconds."""
    import torch

    import expert_gemm_layers_gb300 as dg
    from expert_gemm_layers_gb300 import synth
    t = synth.ffn_inputs(2, 4, 16, 128, 2, seed=42, device=dev)
    params = {n: t[n] for n in dg.FFN_PARAM_NAMES}
    x = t["inputs"]
    dY = synth.ffn_grad_output(2, 4, 16, 128, seed=43, device=dev)
    import ctypes
    lib = dg._lib.load()
    sh = dg.ffn_shape(2, 4, 16, 128, 2)
    saved = torch.empty(lib.dg_a2a_ffn_saved_bytes(ctypes.byref(sh)), dtype=torch.uint8, device=dev)
    ws = dg.alloc_workspace(lib.dg_a2a_ffn_bwd_workspace_bytes(ctypes.byref(sh), 0), dev)
    out = torch.empty_like(x)
    grads = {n: torch.empty_like(v) for n, v in params.items()}
    grads["inputs"] = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    iters = 100
    res = {}
    for name, with_bwd in (("forward", False), ("forward_backward", True)):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for i in range(iters + 10):
            if i >= 10:
                ev[i - 10][0].record(stream)
            dg.a2a_ffn_forward(x, params, saved=saved, out=out)
            if with_bwd:
                dg.a2a_ffn_backward(x, params, saved, dY, workspace=ws, grads=grads)
            if i >= 10:
                ev[i - 10][1].record(stream)
        torch.cuda.synchronize(dev)
        us = [1e3 * a.elapsed_time(b) for a, b in ev]
        res[name] = {"us_mean": round(statistics.mean(us), 2), "us_min": round(min(us), 2),
                     "us_max": round(max(us), 2), "iters": iters}
    for wsx in (None, ws):
        st, code = dg.device_status(dev, workspace=wsx)
        if st != 0:
            raise RuntimeError(f"device error word after the tiny workload: {code:#x}")
    return {"ffn_tiny_latency": dict(res, workload="A2A FFN P=2, B=4, T=16, D=128, k=2 (H=256), seed 42",
                                     timing="CUDA events around each call, back to back, 10 untimed first")}


def run_attn_proj(w, args, dev, peaks):
    """Attention projections at the Llama-3-8B shape over W=8 shards (outside the step):
    fused QKV and wo forward, then both backward (dx and d_weight)."""
    import torch
    dg = w.dg
    for _ in range(max(args.warmup, 2)):
        w.attn_proj()
    iters = 5
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize(dev)
    dg.trace_begin()
    ev[0].record(stream)
    for _ in range(iters):
        w.attn_proj()
    ev[1].record(stream)
    torch.cuda.synchronize(dev)
    trace = dg.trace_end()
    st, code = w.status()
    if st != 0:
        raise RuntimeError(f"device error word after the attention projections: {code:#x}")
    ms = ev[0].elapsed_time(ev[1]) / iters
    S, d = TP["S"], TP["d"]
    flops = 3 * 2.0 * S * d * (ATTN["qkv_out"] + d)  # forward, dx and d_weight of both projections
    tf = flops / (ms * 1e-3) / 1e12
    return {"attn_proj_fwd_bwd": {
        "ms": round(ms, 4), "tflops": round(tf, 2), "peak_tflops": peaks["bf16_tflops"],
        "frac_of_peak": round(tf / peaks["bf16_tflops"], 4), "iters": iters,
        "shape": f"S={S}, d={d}, QKV out {ATTN['qkv_out']}, wo {d}x{d}, W={TP['W']}, no bias",
        "kernels": {e["name"]: {"launches": e["launches"], "ms_per_launch": round(e["total_ms"] / e["launches"], 4)}
                    for e in trace}}}


# Per-step data of the end-to-end run: the step's activations come from the
# host and its outputs go back; weights and weight gradients stay resident.
E2E_INPUTS = ("A", "B", "C", "x", "dY", "xs")
E2E_OUTPUTS = ("D", "out", "d_inputs", "y")


def _io_get(w, name):
    return w.grads["inputs"] if name == "d_inputs" else getattr(w, name)


def _io_set(w, name, t):
    if name == "d_inputs":
        w.grads["inputs"] = t
    else:
        setattr(w, name, t)


def run_e2e(w, args, dev, step_flops, world):
    """The step through the public API with its data streamed in and out.

    Each step copies its activations host -> device (pinned) and its outputs
    device -> host.  Two device buffer sets and two copy streams let the
    uploads of step i+1 and the downloads of step i-1 overlap the compute of
    step i.  The dependencies are per part of the step: a part waits only for
    its own inputs, an input of the next step is uploaded once the last part
    that reads it has run, and each output is downloaded as soon as its part
    has written it.  One untimed pass of two steps touches the pinned buffers
    and both device sets first; the timed region runs from the first upload to
    the last download."""
    import torch
    sets = [{n: _io_get(w, n) for n in E2E_INPUTS + E2E_OUTPUTS}]
    sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
    h_in = {n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype, pin_memory=True) for n in E2E_INPUTS}
    for n in E2E_INPUTS:
        h_in[n].copy_(sets[0][n])
    h_out = {n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype, pin_memory=True) for n in E2E_OUTPUTS}
    compute = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    parts = w.parts()
    last_reader = {n: max(j for j, (_, ins, _, _) in enumerate(parts) if n in ins) for n in E2E_INPUTS}
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_ready = [{n: ev() for n in E2E_INPUTS} for _ in range(2)]
    consumed = [{n: ev() for n in E2E_INPUTS} for _ in range(2)]
    out_free = [{n: ev() for n in E2E_OUTPUTS} for _ in range(2)]
    written = [{n: ev() for n in E2E_OUTPUTS} for _ in range(2)]

    def upload(k):
        s = k % 2
        for n in E2E_INPUTS:                              # in the order the parts read them
            if k >= 2:
                up.wait_event(consumed[s][n])             # step k-2 has read this buffer
            with torch.cuda.stream(up):
                sets[s][n].copy_(h_in[n], non_blocking=True)
            in_ready[s][n].record(up)

    def loop(steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(compute)
        up.wait_event(e0)
        down.wait_event(e0)
        upload(0)
        for i in range(steps):
            s = i % 2
            if i + 1 < steps:
                upload(i + 1)
            for n, t in sets[s].items():
                _io_set(w, n, t)
            for j, (_, ins, outs, fn) in enumerate(parts):
                for n in ins:
                    compute.wait_event(in_ready[s][n])
                if i >= 2:
                    for n in outs:
                        compute.wait_event(out_free[s][n])  # step i-2's output is on the host
                fn()
                for n in ins:
                    if last_reader[n] == j:
                        consumed[s][n].record(compute)
                for n in outs:
                    written[s][n].record(compute)
                    down.wait_event(written[s][n])
                    with torch.cuda.stream(down):
                        h_out[n].copy_(sets[s][n], non_blocking=True)
                    out_free[s][n].record(down)
        e1.record(down)
        torch.cuda.synchronize(dev)
        for n, t in sets[0].items():
            _io_set(w, n, t)
        return e0.elapsed_time(e1) / steps

    loop(2)                                               # untimed: first touch of the pinned buffers
    steps = max(1, min(args.steps, 20))                  # the device-timed step count, up to 20
    ms = max_over_ranks(loop(steps), world, dev)
    return {"value": round(job_tflops(world, step_flops, ms), 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "steps": steps, "warmup": 2,
            "h2d_bytes_per_step": int(sum(h_in[n].numel() * h_in[n].element_size() for n in E2E_INPUTS)),
            "d2h_bytes_per_step": int(sum(h_out[n].numel() * h_out[n].element_size() for n in E2E_OUTPUTS)),
            "copies": "per step: activations (FP8 A, B, C; FFN inputs and dY; TP x) uploaded from pinned host "
                      "memory, outputs (FP8 D, FFN output and d_inputs, TP y) downloaded; weights and weight "
                      "gradients resident on the device; two copy streams and two device buffer sets, with "
                      "per-part dependencies, overlap the copies with the neighbouring steps' compute"}


PROFILE_CASES = {
    "fp8": "FP8 GEMM 4096^3 (alpha 0.5, beta 1)",
    "ffn_fwd_small": "A2A FFN forward, P=8, B=512, T=8, D=1280, k=6 (the full shape with 8 token positions)",
    "ffn_fwd_small_separate": "the same forward with the normalise-and-gate as a separate pass through HBM",
    "ffn_small": "A2A FFN forward + backward, P=8, B=512, T=8, D=1280, k=6",
    "tp": "TP SwiGLU, S=8192, d=4096, ffn=14336, W=8",
    "ffn_fp8_small": "A2A FFN forward on e4m3 GEMMs, P=8, B=512, T=8, D=1280, k=6",
}


def run_profile_case(args):
    """Runs one part of the path `--steps` times on a case small enough for an ncu capture."""
    import torch

    import expert_gemm_layers_gb300 as dg
    from expert_gemm_layers_gb300 import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    case = args.profile_case
    if case == "fp8":
        A, B, C = synth.fp8_gemm_inputs(4096, 4096, 4096, seed=1, device=dev)
        D = torch.empty((4096, 4096), dtype=torch.bfloat16, device=dev)
        run = lambda: dg.gemm_fp8(A, B, C, 0.5, 1.0, out=D)
    elif case in ("ffn_fwd_small", "ffn_small", "ffn_fwd_small_separate"):
        t = synth.ffn_inputs(8, 512, 8, 1280, 6, seed=42, device=dev)
        params = {n: t[n] for n in dg.FFN_PARAM_NAMES}
        x = t["inputs"]
        dY = synth.ffn_grad_output(8, 512, 8, 1280, seed=43, device=dev)
        flags = dg.DG_FFN_SEPARATE_GATE if case == "ffn_fwd_small_separate" else 0

        def run():
            out, saved = dg.a2a_ffn_forward(x, params, flags=flags)
            if case == "ffn_small":
                dg.a2a_ffn_backward(x, params, saved, dY)
    elif case == "ffn_fp8_small":
        t = synth.ffn_inputs(8, 512, 8, 1280, 6, seed=42, device=dev)
        params = {n: t[n] for n in dg.FFN_PARAM_NAMES}
        x = t["inputs"]
        packed = dg.a2a_ffn_fp8_pack_weights(params, 8, 512, 8, 1280)
        run = lambda: dg.a2a_ffn_forward_fp8(x, params, packed)
    elif case == "tp":
        xs, w13, w2 = synth.tp_swiglu_inputs(8192, 4096, 14336, 8, seed=7, device=dev)
        run = lambda: dg.tp_swiglu(xs, w13, w2)
    else:
        raise SystemExit(f"unknown profile case {case}; one of {sorted(PROFILE_CASES)}")
    for _ in range(args.steps):
        run()
    torch.cuda.synchronize(dev)
    st, code = dg.device_status(dev)
    if st != 0:
        raise SystemExit(f"device error word set: {code:#x}")
    print(json.dumps({"profile_case": case, "what": PROFILE_CASES[case], "steps": args.steps}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("dg", "reference"), default="dg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--step-only", action="store_true",
                    help="skip the measurements outside the step (for a launch list of the step alone)")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default=None,
                    help="run one small part of the path (for ncu captures) instead of the benchmark")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_dg(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
