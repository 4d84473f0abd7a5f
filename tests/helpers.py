"""Shared test helpers: inputs from the seeded generators, the output tolerance,
and conversions between torch bf16 tensors and numpy bit patterns."""
from __future__ import annotations

import numpy as np
import torch

from group_affine_bit_gb300 import synth


def u16(t: torch.Tensor) -> np.ndarray:
    return synth.bits_u16(t)


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def tolerance_report(y_gpu_bits: np.ndarray, y_ref: np.ndarray):
    """The output bound |y - y_ref| <= 2^-7 |y_ref| + 1e-3 * rms(y_ref row).
    Returns (ok, worst ratio of error to bound, count out of bound)."""
    y = bf16_to_f64(y_gpu_bits)
    rms = np.sqrt(np.mean(y_ref ** 2, axis=1, keepdims=True))
    bound = 2.0 ** -7 * np.abs(y_ref) + 1e-3 * rms
    err = np.abs(y - y_ref)
    ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1), np.where(err > 0, np.inf, 0))
    bad = int(np.count_nonzero(err > bound))
    return bad == 0, float(np.max(ratio)) if ratio.size else 0.0, bad


def assert_within_tolerance(y_gpu: torch.Tensor, y_ref: np.ndarray, what=""):
    ok, worst, bad = tolerance_report(u16(y_gpu), y_ref)
    assert ok, f"{what}: {bad} outputs outside 2^-7|y|+1e-3 rms (worst {worst:.3f} of the bound)"
    return worst


# ----------------------------------------------------------------------------- decode split, replayed on the host
DECODE_CTAS_PER_SM = 2   # decode CTAs one SM holds (110 KB of shared memory each)


def decode_tile_split(N: int, K: int, sms: int, ctas_per_sm: int = DECODE_CTAS_PER_SM):
    """How the decode launch cuts one projection: its (128-row tile, 128-deep
    block) units, numbered tile-major, are cut into PC contiguous runs, run
    c = [c*U//PC, (c+1)*U//PC), PC = min(resident CTAs, units) -- or, when
    there are fewer tiles than resident CTAs, tiles x S if S = floor(resident
    / tiles) > 1 fills 90 % of them (every tile cut into S runs), else the
    number of tiles if that fills 75 % (one whole tile per run).  Returns (whole, split): tiles that one run covers entirely
    (stored straight from registers) and tiles that two or more runs share
    (fp32 partials merged in run order)."""
    tiles = -(-N // 128)
    KB = -(-K // 128)
    U = tiles * KB
    resident = sms * ctas_per_sm
    PC = min(resident, U)
    if tiles < resident:
        S = min(resident // tiles, KB)
        if S > 1 and tiles * S * 100 >= resident * 90:
            PC = tiles * S
        elif tiles * 100 >= resident * 75:
            PC = tiles

    def run_of(u):
        return ((u + 1) * PC - 1) // U

    whole = sum(1 for t in range(tiles) if run_of(t * KB) == run_of(t * KB + KB - 1))
    return whole, tiles - whole
