"""Seeded synthetic workloads: shapes, seeds and input generators.

This module holds no arithmetic of the method itself.  It only draws the
inputs (q, k, v, the per-head decay values and the per-feature gates) that
both the CUDA path and the CPU oracle consume, so the two sides always see the
same numbers.

Recipe: a CPU ``torch.Generator`` seeded per workload draws fp32 N(0, 1)
samples in the order q, k, v; they are multiplied by the workload's scale and
rounded once to the workload's dtype.  The oracle widens exactly those rounded
values, the GPU reads them as they are.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    causal: bool
    B: int
    H: int
    N: int
    D: int
    Dv: int
    dtype: torch.dtype
    scale: float
    seed: int
    decayed: bool = False
    eps: float = 1e-6
    # decode workloads: number of single-token steps after the prefill of N
    steps: int = 0
    step_seed0: int = 0
    # gated workloads: fp32 gates a [B, H, N, D] uniform in [gate_lo, 1)
    gated: bool = False
    gate_lo: float = 0.9
    # Performer workloads: r random features from block-orthogonal
    # directions drawn with seed + 2
    favor_r: int = 0
    # backward workloads: one la_backward over the causal form, with an
    # upstream gradient dL/do ~ N(0, 1) drawn with seed + 3
    backward: bool = False

    @property
    def tokens(self) -> int:
        return self.B * self.N

    def gamma(self) -> Optional[torch.Tensor]:
        return retnet_gammas(self.H) if self.decayed else None


def retnet_gammas(H: int) -> torch.Tensor:
    """Per-head fixed decays gamma_h = 1 - 2^(-5 - h/4), h = 0..H-1, computed
    in fp64 and rounded once to fp32 (the value both sides use)."""
    h = torch.arange(H, dtype=torch.float64)
    return (1.0 - torch.pow(2.0, -5.0 - h / 4.0)).to(torch.float32)


WORKLOADS = {
    # causal, gamma = 1, fp32, B1 H1 N256 D=Dv=64, N(0,1), seed 0
    "causal_f32_n256": Workload("causal_f32_n256", True, 1, 1, 256, 64, 64,
                                torch.float32, 1.0, 0),
    # causal, gamma = 1, bf16, B4 H8 N4096 D=Dv=64, N(0,1)*0.5, seed 1
    "causal_bf16_n4096": Workload("causal_bf16_n4096", True, 4, 8, 4096, 64,
                                  64, torch.bfloat16, 0.5, 1),
    # causal with per-head RetNet decay, bf16, B2 H16 N16384 D=Dv=128, seed 2
    "causal_decay_bf16_n16384": Workload("causal_decay_bf16_n16384", True, 2,
                                         16, 16384, 128, 128, torch.bfloat16,
                                         0.5, 2, decayed=True),
    # the same at half the sequence length (same grid of CTAs, 268 MB of
    # inputs, above the L2 size): the case for multi-pass counter captures
    "causal_decay_bf16_n8192": Workload("causal_decay_bf16_n8192", True, 2,
                                        16, 8192, 128, 128, torch.bfloat16,
                                        0.5, 2, decayed=True),
    # non-causal, bf16, B8 H16 N65536 D=Dv=64, seed 3
    "noncausal_bf16_n65536": Workload("noncausal_bf16_n65536", False, 8, 16,
                                      65536, 64, 64, torch.bfloat16, 0.5, 3),
    # the same at an eighth of the sequence length (the same CTA grid per
    # pass, 537 MB of inputs and output, above the L2 size): the case for
    # multi-pass counter captures
    "noncausal_bf16_n8192": Workload("noncausal_bf16_n8192", False, 8, 16,
                                     8192, 64, 64, torch.bfloat16, 0.5, 3),
    # gated (one gate per key feature and token), bf16, B2 H16 N16384
    # D=Dv=128, gates U[0.9, 1) from seed 5 + 1
    "gla_bf16_n16384": Workload("gla_bf16_n16384", True, 2, 16, 16384, 128,
                                128, torch.bfloat16, 0.5, 5, gated=True),
    # Performer (FAVOR+) causal, bf16, B2 H16 N16384 D=Dv=128, r = 128
    # block-orthogonal features; q, k ~ N(0, 1) * D^(-1/4) (the usual
    # softmax temperature folded into the inputs)
    "favor_bf16_n16384": Workload("favor_bf16_n16384", True, 2, 16, 16384, 128,
                                  128, torch.bfloat16, 128 ** -0.25, 6, favor_r=128),
    # backward of the causal form, bf16, B4 H8 N4096 D=Dv=64 (the training
    # shape of the causal configurations), gamma = 1
    "backward_bf16_n4096": Workload("backward_bf16_n4096", True, 4, 8, 4096, 64, 64,
                                    torch.bfloat16, 0.5, 7, backward=True),
    # gated decode: the decode workload's shape, a fresh fp32 gate per step
    # and key feature, U[0.9, 1) (seed of step t: 1000 + t + 50000)
    "decode_gated_bf16_h32": Workload("decode_gated_bf16_h32", True, 256, 32, 512, 128,
                                      128, torch.bfloat16, 0.5, 4, steps=1024,
                                      step_seed0=1000, gated=True),
    # decode: 256 sequences x H32, D=Dv=128; prefill of 512 tokens (seed 4),
    # then 1024 single-token steps with fresh inputs from seed 1000 + t
    "decode_bf16_h32": Workload("decode_bf16_h32", True, 256, 32, 512, 128,
                                128, torch.bfloat16, 0.5, 4, steps=1024,
                                step_seed0=1000),
}


def make_qkv(B, H, N, D, Dv, dtype=torch.bfloat16, seed=0, scale=1.0,
             device="cpu"):
    """q, k: [B, H, N, D]; v: [B, H, N, Dv], drawn on the CPU in the order
    q, k, v from one generator seeded with ``seed``, scaled, then rounded to
    ``dtype`` and moved to ``device``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = []
    for shape in ((B, H, N, D), (B, H, N, D), (B, H, N, Dv)):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        out.append(x.to(dtype).to(device))
    return tuple(out)


def workload_inputs(w: Workload, device="cpu"):
    """The q, k, v of workload ``w`` (for decode workloads: the prefill)."""
    return make_qkv(w.B, w.H, w.N, w.D, w.Dv, w.dtype, w.seed, w.scale, device)


def decode_step_inputs(w: Workload, t: int, device="cpu"):
    """Fresh q, k: [B, H, D] and v: [B, H, Dv] for decode step t."""
    q, k, v = make_qkv(w.B, w.H, 1, w.D, w.Dv, w.dtype, w.step_seed0 + t,
                       w.scale, device)
    return q[:, :, 0], k[:, :, 0], v[:, :, 0]


def make_gates(B, H, N, D, seed=0, lo=0.9, hi=1.0, zero_frac=0.0, one_frac=0.0,
               device="cpu"):
    """Gates a: [B, H, N, D] fp32, uniform in [lo, hi) from a CPU generator
    seeded with ``seed``; then a ``zero_frac`` share of the entries (drawn
    from the same generator) is set to exactly 0 and a ``one_frac`` share to
    exactly 1."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    a = torch.rand((B, H, N, D), generator=g, dtype=torch.float32) * (hi - lo) + lo
    a.clamp_(0.0, 1.0)
    if zero_frac > 0:
        a[torch.rand(a.shape, generator=g) < zero_frac] = 0.0
    if one_frac > 0:
        a[torch.rand(a.shape, generator=g) < one_frac] = 1.0
    return a.to(device)


def workload_gates(w: Workload, device="cpu"):
    """The gates of a gated workload (seed + 1, uniform in [gate_lo, 1))."""
    return make_gates(w.B, w.H, w.N, w.D, w.seed + 1, w.gate_lo, 1.0, device=device)


def favor_matrix(r, D, seed=0, orthogonal=True, dtype=torch.float32, device="cpu"):
    """Random directions W [r, D] for the Performer feature map, drawn on the
    CPU in fp64 and rounded once to ``dtype``.

    orthogonal=False: every entry N(0, 1).  orthogonal=True (positive
    orthogonal random features): each block of D rows is the transpose of the
    Q factor of a D x D Gaussian matrix (signs fixed by R's diagonal, so the
    block is Haar-distributed), and every row is rescaled by the norm of a
    fresh D-dimensional Gaussian vector, so each row is still marginally
    N(0, I) while the rows of a block are exactly orthogonal."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    if not orthogonal:
        W = torch.randn((r, D), generator=g, dtype=torch.float64)
    else:
        blocks = []
        for _ in range(-(-r // D)):
            G = torch.randn((D, D), generator=g, dtype=torch.float64)
            Q, R = torch.linalg.qr(G)
            Q = Q * torch.sign(torch.diagonal(R))
            blocks.append(Q.T)
        W = torch.cat(blocks)[:r]
        norms = torch.randn((r, D), generator=g, dtype=torch.float64).norm(dim=1)
        W = W * norms[:, None]
    return W.to(dtype).to(device)


def workload_favor_matrix(w: Workload, device="cpu"):
    """The block-orthogonal directions [r, D] of a Performer workload."""
    return favor_matrix(w.favor_r, w.D, w.seed + 2, True, w.dtype, device)


def workload_upstream(w: Workload, device="cpu"):
    """The upstream gradient dL/do [B, H, N, Dv] of a backward workload:
    N(0, 1) from seed + 3, rounded once to the workload dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed + 3))
    return torch.randn((w.B, w.H, w.N, w.Dv), generator=g).to(w.dtype).to(device)


def decode_step_gates(w: Workload, t: int, device="cpu"):
    """The gates a: [B, H, D] fp32 of gated decode step t."""
    return make_gates(w.B, w.H, 1, w.D, w.step_seed0 + t + 50000, w.gate_lo, 1.0,
                      device=device)[:, :, 0].contiguous()
