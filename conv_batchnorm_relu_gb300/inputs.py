"""Seeded synthetic inputs for the CBR operator.

This module is the one piece that both the CUDA path's tests and the CPU oracle use.  It draws
random numbers and rounds them to the storage dtype; it contains none of the operator's
arithmetic.

Recipe (the same for every workload):
  * generator: ``torch.Generator('cpu').manual_seed(seed)``; draws in fp32 in the order
    x, W, gamma, beta, dy;
  * x ~ N(0, 1), or U(-2.5, 2.5) for the first-layer (image-like) workload;
  * W ~ Kaiming-normal, std = sqrt(2 / (Cin*R*S)), no conv bias;
  * gamma ~ U(0.5, 1.5), beta ~ N(0, 0.1^2), running_mean = 0, running_var = 1;
  * dy ~ N(0, 1) with the output's shape;
  * x, W and dy are rounded to fp16 / bf16 (round-to-nearest-even); gamma, beta and the
    running statistics stay fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class CBRSpec:
    """Shape of one CBR layer: x NHWC [n,h,w,c_in], W KRSC [c_out,r,s,c_in]."""

    name: str
    n: int
    h: int
    w: int
    c_in: int
    c_out: int
    r: int = 3
    s: int = 3
    stride: int = 1
    pad: int = 1
    dtype: str = "f16"          # "f16" or "bf16"
    x_dist: str = "normal"      # "normal" -> N(0,1); "uniform2.5" -> U(-2.5, 2.5)
    first_layer: bool = False   # backward skips dx
    infer: bool = False         # the workload also runs the folded inference path
    eps: float = 1e-5
    momentum: float = 0.1

    @property
    def p(self) -> int:
        return (self.h + 2 * self.pad - self.r) // self.stride + 1

    @property
    def q(self) -> int:
        return (self.w + 2 * self.pad - self.s) // self.stride + 1

    @property
    def m(self) -> int:
        """Rows reduced per BN channel: N*P*Q."""
        return self.n * self.p * self.q

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float16 if self.dtype == "f16" else torch.bfloat16

    def conv_flops(self) -> int:
        """2*M*K_red*Cout for one convolution (fprop, dgrad or wgrad)."""
        return 2 * self.m * self.r * self.s * self.c_in * self.c_out

    def with_(self, **kw) -> "CBRSpec":
        return replace(self, **kw)


# The five workloads.  Index i is seeded with 1234 + i (1-based).
CONFIGS: dict[int, CBRSpec] = {
    1: CBRSpec("tiny 2x8x8 8->16 3x3", n=2, h=8, w=8, c_in=8, c_out=16),
    2: CBRSpec("resnet-stage1 32x56x56 64->64 3x3", n=32, h=56, w=56, c_in=64, c_out=64),
    3: CBRSpec("large-batch 256x56x56 64->64 3x3", n=256, h=56, w=56, c_in=64, c_out=64),
    4: CBRSpec("first-layer 256x224x224 3->64 7x7 s2", n=256, h=224, w=224, c_in=3, c_out=64,
               r=7, s=7, stride=2, pad=3, x_dist="uniform2.5", first_layer=True),
    5: CBRSpec("vgg-hires 64x112x112 128->128 3x3 bf16", n=64, h=112, w=112, c_in=128,
               c_out=128, dtype="bf16", infer=True),
}


def seed_for(cfg_id: int) -> int:
    return 1234 + cfg_id


def make_inputs(spec: CBRSpec, seed: int, with_dy: bool = True) -> dict[str, torch.Tensor]:
    """Draw one set of CPU tensors for ``spec``: x, w (storage dtype), gamma, beta,
    running_mean, running_var (fp32) and dy (storage dtype)."""
    g = torch.Generator("cpu").manual_seed(seed)
    dt = spec.torch_dtype
    if spec.x_dist == "normal":
        x = torch.randn((spec.n, spec.h, spec.w, spec.c_in), generator=g, dtype=torch.float32)
    elif spec.x_dist == "uniform2.5":
        x = torch.rand((spec.n, spec.h, spec.w, spec.c_in), generator=g, dtype=torch.float32)
        x = x * 5.0 - 2.5
    else:
        raise ValueError(spec.x_dist)
    std = (2.0 / (spec.c_in * spec.r * spec.s)) ** 0.5
    w = torch.randn((spec.c_out, spec.r, spec.s, spec.c_in), generator=g, dtype=torch.float32) * std
    gamma = torch.rand((spec.c_out,), generator=g, dtype=torch.float32) + 0.5
    beta = torch.randn((spec.c_out,), generator=g, dtype=torch.float32) * 0.1
    out = dict(x=x.to(dt), w=w.to(dt), gamma=gamma, beta=beta,
               running_mean=torch.zeros(spec.c_out, dtype=torch.float32),
               running_var=torch.ones(spec.c_out, dtype=torch.float32))
    if with_dy:
        dy = torch.randn((spec.n, spec.p, spec.q, spec.c_out), generator=g, dtype=torch.float32)
        out["dy"] = dy.to(dt)
    return out
