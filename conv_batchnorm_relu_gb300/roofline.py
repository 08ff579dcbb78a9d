"""Algorithmic roofline ledger of one CBR training step (forward + backward).

Minimum bytes per pass: every input read once and every output written once, activations
in the storage dtype, the ReLU mask at one bit per element.  This is the fused transaction
count of the Tech-Renaissance CBR page, section 9 (conv_output written once and read once;
no bn_output; dy*mask kept on chip).  FLOPs count 2*M*K_red*Cout per convolution; BN and
recompute arithmetic is not counted.

Design "store z once": the forward conv writes z, the apply pass reads it, and the backward
passes re-derive dz from (dy, z, mask) in both dgrad and wgrad.

Peaks: a step of this operator lasts well under a millisecond, so the tensor roofs use the
measured burst bf16 GEMM rate (a kernel timed in isolation); `sustained=True` gives the
seconds-long power-capped rate instead, for comparison.

`kernel_passes` gives the same minimum-traffic count per kernel of the implemented step, whose
backward either evaluates dz on chip in one kernel for both convolutions (the fused design) or
materialises it once (dz pass, then wgrad and dgrad reading it).
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


@dataclass
class Pass:
    name: str
    bytes: int
    flops: int

    def roof_us(self, peaks: dict, sustained: bool = False) -> tuple[float, str]:
        tf = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        t_mem = self.bytes / (peaks["hbm_gbs"] * 1e9) * 1e6
        t_tc = self.flops / (tf * 1e12) * 1e6
        return (t_tc, "tensor") if t_tc > t_mem else (t_mem, "hbm")


def load_peaks() -> tuple[dict, str]:
    """Measured peaks of the GB300s (driver-written), else the stated fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    return dict(FALLBACK), "fallback"


def ledger(spec, need_dx: bool = True) -> list[Pass]:
    e = 2  # fp16 / bf16
    x = spec.n * spec.h * spec.w * spec.c_in * e
    s = spec.n * spec.p * spec.q * spec.c_out * e        # one output-sized activation
    mask = spec.n * spec.p * spec.q * spec.c_out // 8
    w = spec.c_out * spec.r * spec.s * spec.c_in * e
    dw = spec.c_out * spec.r * spec.s * spec.c_in * 4
    cv = spec.conv_flops()
    passes = [
        Pass("conv_fprop_genstats", x + w + s, cv),
        Pass("bn_apply_relu", s + s + mask, 0),
        Pass("bn_bwd_reduce", s + s + mask, 0),
        Pass("conv_wgrad", x + s + s + mask + dw, cv),
    ]
    if need_dx:
        passes.append(Pass("conv_dgrad", s + s + mask + w + x, cv))
    return passes


def kernel_passes(spec, need_dx: bool = True, fused: bool = True, persist: bool = False) -> list[Pass]:
    """Minimum bytes and algorithmic FLOPs of each kernel of the implemented step (names as the
    benchmark reports them). persist: the forward is one persistent kernel (conv, statistics,
    finalize, apply) that writes z, y and the mask."""
    e = 2
    x = spec.n * spec.h * spec.w * spec.c_in * e
    s = spec.n * spec.p * spec.q * spec.c_out * e
    mask = spec.n * spec.p * spec.q * spec.c_out // 8
    w = spec.c_out * spec.r * spec.s * spec.c_in * e
    dw = spec.c_out * spec.r * spec.s * spec.c_in * 4
    cv = spec.conv_flops()
    if persist:
        passes = [Pass("conv_fprop_apply", x + w + s + s + mask, cv)]
    else:
        passes = [Pass("conv_fprop_genstats", x + w + s, cv), Pass("bn_apply_relu", s + s + mask, 0)]
    passes.append(Pass("bn_bwd_reduce", s + s + mask, 0))
    if fused:
        # dy, z, mask and x read once; dx and the fp32 dW written once
        passes.append(Pass("conv_bwd_fused", s + s + mask + x + dw + ((w + x) if need_dx else 0),
                           cv * (2 if need_dx else 1)))
    else:
        passes.append(Pass("bn_dz", s + s + mask + s, 0))
        passes.append(Pass("conv_wgrad", x + s + dw, cv))
        if need_dx:
            passes.append(Pass("conv_dgrad", s + w + x, cv))
    return passes


def infer_pass(spec) -> Pass:
    """Folded inference: x and W_fold in, y out (bias + ReLU in the conv epilogue)."""
    e = 2
    x = spec.n * spec.h * spec.w * spec.c_in * e
    y = spec.n * spec.p * spec.q * spec.c_out * e
    w = spec.c_out * spec.r * spec.s * spec.c_in * e
    return Pass("conv_infer", x + w + y + spec.c_out * 4, spec.conv_flops())


def step_roof_us(spec, peaks: dict, need_dx: bool = True, sustained: bool = False) -> float:
    return sum(p.roof_us(peaks, sustained)[0] for p in ledger(spec, need_dx))


def ridge(tflops: float, tbs: float) -> float:
    """FLOP per byte at which compute and memory time are equal."""
    return tflops / tbs
