"""Seeded synthetic inputs shared by the tests, the bench and the CPU oracle.

This module only draws numbers: it holds none of the pruning, packing or GEMM
arithmetic, so both the CUDA path and the oracle can take their inputs from it
without sharing any of the method's code.

Every tensor is drawn from its own torch.Generator seeded with
(seed, tensor id); tensor ids: X=1, W_up=2, W_down=3, b_up=4, b_down=5, dY=6.
Weights and activations follow the workload table below (normal with the stated
sigma, rounded to bf16 by torch's round-to-nearest-even conversion).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

TENSOR_IDS = {"X": 1, "W_up": 2, "W_down": 3, "b_up": 4, "b_down": 5, "dY": 6}


def _generator(seed: int, tensor_id: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    # splitmix-style mixing keeps the streams of different tensors apart
    z = (seed * 0x9E3779B97F4A7C15 + tensor_id * 0xBF58476D1CE4E5B9) & ((1 << 63) - 1)
    g.manual_seed(z)
    return g


def normal_bf16(shape, sigma: float, seed: int, tensor_id: int, device="cpu") -> torch.Tensor:
    """N(0, sigma^2) samples rounded to bf16."""
    g = _generator(seed, tensor_id, device)
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    if sigma != 1.0:
        t.mul_(sigma)
    return t.to(torch.bfloat16)


def normal_f32(shape, sigma: float, seed: int, tensor_id: int, device="cpu") -> torch.Tensor:
    g = _generator(seed, tensor_id, device)
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device) * sigma


def small_int_bf16(shape, lo: int, hi: int, seed: int, tensor_id: int, device="cpu") -> torch.Tensor:
    """Integers uniform in [lo, hi] as bf16: many exact magnitude ties (tie-stress inputs)."""
    g = _generator(seed, tensor_id, device)
    return torch.randint(lo, hi + 1, tuple(shape), generator=g, device=device).to(torch.bfloat16)


@dataclass(frozen=True)
class FFNWorkload:
    """One synthetic FFN layer: X [M, d], W_up [ffn, d], W_down [d, ffn], dY [M, d]."""
    name: str
    M: int
    d: int
    ffn: int
    w_sigma: float
    x_sigma: float = 1.0
    dy_sigma: float = 1.0
    reprune: bool = True      # prune from the dense weights inside every step
    act24: bool = False       # 2:4-prune ReLU(up) along ffn and feed it as the sparse operand

    @property
    def dense_equiv_flop(self) -> int:
        """Six GEMMs of 2*M*d*ffn each: up/down forward, two dX, two dW."""
        return 12 * self.M * self.d * self.ffn


# The workloads of the sparse FFN training benchmark.
WORKLOADS = {
    "tiny": FFNWorkload("tiny_single_linear_N256_K512_M128", 128, 512, 256, 1.0),
    "gpt2": FFNWorkload("gpt2_small_ffn_d768_ffn3072_M4096", 4096, 768, 3072, 0.02),
    "1p3b": FFNWorkload("ffn_1p3b_d2048_ffn8192_M8192_reprune", 8192, 2048, 8192, 0.02),
    "7b_act24": FFNWorkload("ffn_7b_d4096_ffn16384_M16384_act24", 16384, 4096, 16384, 0.02, act24=True),
    "70b_m2048": FFNWorkload("ffn_70b_d8192_ffn28672_M2048", 2048, 8192, 28672, 0.01),
    "70b_m8192": FFNWorkload("ffn_70b_d8192_ffn28672_M8192", 8192, 8192, 28672, 0.01),
    "70b_m16384": FFNWorkload("ffn_70b_d8192_ffn28672_M16384", 16384, 8192, 28672, 0.01),
    # the 70B tail shapes (M = 1000 tokens, K = 8200, so K % 128 != 0) as one FFN layer
    "70b_tail": FFNWorkload("ffn_70b_tail_d8200_ffn28672_M1000", 1000, 8200, 28672, 0.01),
}


def ffn_inputs(w: FFNWorkload, seed: int = 0, device="cpu", bias: bool = False) -> dict:
    """X, W_up, W_down, dY (bf16) and b_up, b_down (fp32) for one workload."""
    out = {
        "X": normal_bf16((w.M, w.d), w.x_sigma, seed, TENSOR_IDS["X"], device),
        "W_up": normal_bf16((w.ffn, w.d), w.w_sigma, seed, TENSOR_IDS["W_up"], device),
        "W_down": normal_bf16((w.d, w.ffn), w.w_sigma, seed, TENSOR_IDS["W_down"], device),
        "dY": normal_bf16((w.M, w.d), w.dy_sigma, seed, TENSOR_IDS["dY"], device),
    }
    if bias:
        out["b_up"] = normal_f32((w.ffn,), 0.1, seed, TENSOR_IDS["b_up"], device)
        out["b_down"] = normal_f32((w.d,), 0.1, seed, TENSOR_IDS["b_down"], device)
    else:
        out["b_up"] = torch.zeros(w.ffn, dtype=torch.float32, device=device)
        out["b_down"] = torch.zeros(w.d, dtype=torch.float32, device=device)
    return out
