"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and casts them; it holds none of the attention arithmetic.
Every tensor is drawn in fp32 on the CPU from a seeded ``torch.Generator`` (normal
distribution times a standard deviation), then rounded to bf16 (round to nearest even).  The
same bits go to the fp64 oracle (widened exactly) and, after a host-to-device copy, to the GPU.

The named workloads are the shapes "Self-attention, CUDA kernels and FlashAttention" talks
about (section 1: a 224x224 ViT image in 16x16 patches gives N=196 tokens, 12 heads, D=768;
section 3: high-resolution images and long text sequences), with Gaussian values standing
in for real images, text and trained weights, none of which the article uses or supplies.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    qk_std: float = 1.0     # standard deviation of Q and K entries
    v_std: float = 1.0      # standard deviation of V and dO entries
    backward: bool = True   # whether the workload includes the backward pass
    seed: int = 0
    model_dim: int = 0      # >0: Q, K, V come from X [B,N,model_dim] times per-head projections

    @property
    def bh(self) -> int:
        return self.B * self.H

    @property
    def scale(self) -> float:
        """1/sqrt(d_k) rounded to fp32: the scale both sides receive."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    def fwd_flops(self) -> float:
        return 4.0 * self.B * self.H * self.N * self.N * self.d

    def bwd_flops(self) -> float:
        return 10.0 * self.B * self.H * self.N * self.N * self.d


WORKLOADS = {
    w.name: w
    for w in (
        Workload("vit_b16_single", B=1, H=12, N=196, d=64, backward=False, seed=1001),
        Workload("vit_b16_batch", B=64, H=12, N=196, d=64, seed=1002),
        Workload("vit_l_highres", B=8, H=16, N=4096, d=64, seed=1003),
        Workload("long_text", B=2, H=16, N=16384, d=128, qk_std=2.0, seed=1004),
        Workload("vit_b_mhsa_block", B=32, H=12, N=576, d=64, seed=1005, model_dim=768),
    )
}


def _randn(gen: torch.Generator, shape, std: float) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def make_qkv(B: int, H: int, N: int, d: int, seed: int, qk_std: float = 1.0,
             v_std: float = 1.0, with_do: bool = True) -> dict:
    """Q, K, V (and dO) as contiguous [B,H,N,d] bf16 CPU tensors, drawn in that order."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    out = {
        "q": _randn(gen, (B, H, N, d), qk_std),
        "k": _randn(gen, (B, H, N, d), qk_std),
        "v": _randn(gen, (B, H, N, d), v_std),
    }
    if with_do:
        out["do"] = _randn(gen, (B, H, N, d), v_std)
    return out


def make_block_inputs(w: Workload) -> dict:
    """The full ViT-B block workload: X [B,N,D] ~ N(0,1); W_Q, W_K, W_V [D,D] ~ N(0,1/D), split
    column-wise into H heads of d_k = D/H; dO [B,H,N,d_k] ~ N(0,1).  Q = X W_Q (and likewise K, V)
    is formed on the CPU in fp32 from the bf16 values and rounded to bf16: it is the input
    preparation of this workload, not part of the attention path."""
    D = w.model_dim
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    x = _randn(gen, (w.B, w.N, D), 1.0)
    ws = [_randn(gen, (D, D), 1.0 / math.sqrt(D)) for _ in range(3)]
    dout = _randn(gen, (w.B, w.H, w.N, w.d), w.v_std)
    xf = x.float()

    def project(wm):
        y = xf @ wm.float()                                   # [B,N,D]
        y = y.view(w.B, w.N, w.H, w.d).permute(0, 2, 1, 3)    # head h = columns [h*d, (h+1)*d)
        return y.contiguous().to(torch.bfloat16)

    return {"q": project(ws[0]), "k": project(ws[1]), "v": project(ws[2]), "do": dout,
            "x": x, "w_q": ws[0], "w_k": ws[1], "w_v": ws[2]}


def make_workload_inputs(w: Workload) -> dict:
    if w.model_dim:
        return make_block_inputs(w)
    return make_qkv(w.B, w.H, w.N, w.d, w.seed, w.qk_std, w.v_std, with_do=True)
