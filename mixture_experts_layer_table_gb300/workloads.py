"""Seeded synthetic workloads for one MoE layer.

This module only draws random numbers and fixes shapes. It holds none of the
layer's arithmetic (no router, no top-k, no GEMM), so the CUDA path and the CPU
oracle can both consume its tensors without sharing any of the method.

The shapes follow the pages on Mixture-of-Kittens: hidden 7168 and expert
intermediate 2048 come from "把 MoE 通信延迟从 103μs 压到 18μs：Cursor 开源 GPU
内核 MoK" (aientropygate.com), section 03 ② (Megakernel); top-8 of 256 routed
experts is the DeepSeek-V3 layout those pages target ("Mixture-of-Kittens (MoK)",
sd114.wiki, section on hardware and scope). The pages train on real data; no
dataset is named, so seeded Gaussians stand in for activations and weights.

Every tensor has its own generator seeded ``seed + i`` (i = 0..4 for x, W_r,
W13, W2, dY), is sampled in float32 and rounded to bfloat16 (round to nearest
even, torch's cast).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import torch

ROUTER_SOFTMAX = 0
ROUTER_SIGMOID = 1


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """Shape and routing mode of one MoE layer call.

    T tokens of width H are routed to k of E experts; each expert is a SwiGLU FFN
    with intermediate width I.  ``router`` selects softmax or sigmoid scores,
    ``renorm`` renormalises the k selected gates to sum to one.
    """

    name: str
    T: int
    H: int
    E: int
    I: int
    k: int
    router: int
    renorm: bool
    x_std: float
    w_std: float
    dy_std: float = 1.0
    skew: bool = False          # router bias giving Zipf-Mandelbrot expert loads
    mxfp8: bool = False

    @property
    def R(self) -> int:
        """Number of (token, expert) assignments, T*k."""
        return self.T * self.k

    def scaled(self, **kw) -> "MoEShape":
        return dataclasses.replace(self, **kw)


# The five workloads (names state what they are).
TINY = MoEShape("tiny_T256_H256_E8_I512_top2_softmax", T=256, H=256, E=8, I=512, k=2,
                router=ROUTER_SOFTMAX, renorm=False, x_std=0.02, w_std=0.02)
DSV3 = MoEShape("dsv3_T4096_H7168_E256_I2048_top8_sigmoid", T=4096, H=7168, E=256, I=2048, k=8,
                router=ROUTER_SIGMOID, renorm=True, x_std=1.0, w_std=0.006)
DSV3_SKEW = DSV3.scaled(name="dsv3_skew_zipf1.2_T4096_H7168_E256_I2048_top8", skew=True)
DSV3_MXFP8 = DSV3.scaled(name="dsv3_mxfp8_T4096_H7168_E256_I2048_top8", mxfp8=True)
RING = DSV3.scaled(name="dsv3_ring_T16384_H7168_E256_I2048_top8", T=16384)
RING_BYTES = 512 * 2**20
RING_MINIBATCHES = (512, 1024, 2368, 2560, 4096)

WORKLOADS = {w.name: w for w in (TINY, DSV3, DSV3_SKEW, DSV3_MXFP8, RING)}

# Skewed routing: the target load of expert e is Zipf-Mandelbrot
# p_e ~ (e + 1 + q)^-s with s = 1.2 and q = 9.55, which puts the hottest expert at
# 10x the mean (a pure Zipf(1.2) over 256 experts would need 65x, more than top-8
# of distinct experts allows).  The bias added to the selection score is
# b_e = ALPHA * ln(E * p_e); ALPHA = 0.07 was fixed once offline so that the
# hottest expert sees about 10x the mean load on sigmoid scores of this spread.
ZIPF_S = 1.2
ZIPF_Q = 9.55
SKEW_ALPHA = 0.07


def skew_bias(E: int) -> torch.Tensor:
    """Router selection bias (float32 [E]) for the Zipf-Mandelbrot skewed workload."""
    e = torch.arange(E, dtype=torch.float64)
    p = (e + 1.0 + ZIPF_Q) ** (-ZIPF_S)
    p = p / p.sum()
    return (SKEW_ALPHA * torch.log(E * p)).to(torch.float32)


def _normal(shape: Tuple[int, ...], std: float, seed: int, device: str) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=g)
    return t.to(torch.bfloat16)


def make_inputs(shape: MoEShape, seed: int = 0, device: str = "cpu",
                with_dy: bool = True) -> Dict[str, Optional[torch.Tensor]]:
    """Seeded bf16 inputs of one layer call.

    Returns x [T][H], w_router [E][H], w13 [E][2I][H] (rows 0..I-1 gate, I..2I-1 up),
    w2 [E][H][I], dy [T][H] (or None) and router_bias (float32 [E] or None).
    Tensors drawn on ``device``; the CPU and CUDA generators give different values,
    so the two sides of a comparison must share the same tensors.
    """
    T, H, E, I = shape.T, shape.H, shape.E, shape.I
    out: Dict[str, Optional[torch.Tensor]] = {
        "x": _normal((T, H), shape.x_std, seed + 0, device),
        "w_router": _normal((E, H), shape.w_std, seed + 1, device),
        "w13": _normal((E, 2 * I, H), shape.w_std, seed + 2, device),
        "w2": _normal((E, H, I), shape.w_std, seed + 3, device),
        "dy": _normal((T, H), shape.dy_std, seed + 4, device) if with_dy else None,
        "router_bias": skew_bias(E).to(device) if shape.skew else None,
    }
    return out


def algorithmic_flops(shape: MoEShape, passes: str = "fwd") -> float:
    """Dense-equivalent FLOPs of the layer: router GEMM plus the three expert GEMMs.

    forward 2*T*H*E + 6*R*H*I; backward twice that (dgrad and wgrad of each
    GEMM); ``passes`` is "fwd", "bwd" or "fwd+bwd".
    """
    fwd = 2.0 * shape.T * shape.H * shape.E + 6.0 * shape.R * shape.H * shape.I
    return {"fwd": fwd, "bwd": 2.0 * fwd, "fwd+bwd": 3.0 * fwd}[passes]
