"""Seeded synthetic inputs for the group-affine projection.

This module only draws random tensors; it holds none of the method's
arithmetic (no dequantization, no projection).  Tests, the bench and the
oracle checks all take their inputs from here so that both sides of a parity
check read the very same tensors.

Recipe (the value distributions the workloads use):
  * codes  q ~ uniform over [0, 2^bits - 1], one uint8 per code, shape [N, K]
  * scales s = bf16(|N(0, 0.02)| / 8), shape [N, K/g]
  * biases b = bf16(-2^(bits-1) * s + N(0, 1e-3)), computed from the already
    rounded s, shape [N, K/g]
  * activations x = bf16(N(0, 1)), shape [M, K]
Draw order from one generator: q, s, the bias noise, then x.
"""
from __future__ import annotations

import torch


def generator(seed: int, device: str | torch.device = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def affine_table(bits: int, group: int, N: int, K: int, gen: torch.Generator,
                 device: str | torch.device = "cpu"):
    """Return (codes uint8 [N,K], scales bf16 [N,K/g], biases bf16 [N,K/g])."""
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    G = K // group
    codes = torch.randint(0, 1 << bits, (N, K), generator=gen, device=device, dtype=torch.uint8)
    s = (torch.randn(N, G, generator=gen, device=device, dtype=torch.float32) * 0.02).abs() / 8
    scales = s.to(torch.bfloat16)
    noise = torch.randn(N, G, generator=gen, device=device, dtype=torch.float32) * 1e-3
    biases = (-(2.0 ** (bits - 1)) * scales.float() + noise).to(torch.bfloat16)
    return codes, scales, biases


def activations(M: int, K: int, gen: torch.Generator, device: str | torch.device = "cpu"):
    """bf16 [M, K] rows drawn from N(0, 1)."""
    return torch.randn(M, K, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def problem(bits: int, group: int, M: int, N: int, K: int, seed: int,
            device: str | torch.device = "cpu"):
    """One projection's inputs from one seed: (x, codes, scales, biases)."""
    g = generator(seed, device)
    codes, scales, biases = affine_table(bits, group, N, K, g, device)
    x = activations(M, K, g, device)
    return x, codes, scales, biases


def bits_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def from_bits_u16(a) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 CPU tensor."""
    import numpy as np
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)


# The workloads: shapes and seeds of the five standard cases.
DECODER_LAYER_SHAPES = {          # (N, K) of each projection of one decoder layer
    "qkv": (12288, 5376),
    "o": (5376, 8192),
    "gate_up": (43008, 5376),
    "down": (5376, 21504),
}
HEAD_SHAPE = (262144, 5376)
N_LAYERS = 60

TINY = dict(M=1, K=256, N=512, bits=4, group=64, seed=0)
GATE_UP_DECODE = dict(M=1, K=3840, N=30720, bits=4, group=64, seed=1)
DECODE_STEP_SEED = 2
PROMPT_CHUNK = dict(M=128, bits=4, group=64, seed=3)
SWEEP_SHAPE = dict(K=3840, N=15360, seed=4)
EMBED_SEED = 5
SWEEP_CASES = [(2, 4, 64), (4, 4, 64), (8, 4, 64), (16, 4, 64),
               (16, 8, 32), (16, 3, 64), (16, 2, 128)]   # (M, bits, group)


def step_seed(seed: int, layer: int, proj_index: int) -> int:
    """Seed of one projection of a multi-layer workload."""
    return seed + 1000 * layer + proj_index
