"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the mathematics or the pages fix:

* bf16 rounding against torch's CPU float->bfloat16 conversion (a library
  routine) and against the edge cases listed on the "cuda gemma4: images on
  the 12B" page (the bf16(-2^-135) commit), stored under tests/golden/;
* the single-rounding dequantization bf16(s*q + b) against exact rational
  arithmetic (``fractions.Fraction``) with a round-to-nearest-even written
  here from the IEEE definition, on random and adversarial scales and biases;
* the projection against an exact rational brute force on tiny shapes,
  against torch's float64 matmul of the oracle's weights, against one-hot
  activation rows, against the constant-code closed form, and against the
  group-sum identity within its stated bound.

tests/test_oracle.py runs them on the real oracle; tests/test_oracle_plants.py
runs them on copies of the oracle with a planted mistake and requires each
copy to fail at least one of them.
"""
from __future__ import annotations

import math
import os
import random
import struct
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

BF16_MAX = Fraction(255) * Fraction(2) ** 120          # (2 - 2^-7) * 2^127
MIN_ULP = Fraction(1, 2 ** 133)                      # smallest bf16 subnormal


# ----------------------------------------------------------------------------
# Independent exact helpers (Fraction arithmetic, IEEE definition)
# ----------------------------------------------------------------------------
def bf16_value(h: int):
    """Exact value of a bf16 pattern as Fraction, or float('inf')/nan."""
    f = struct.unpack("<f", struct.pack("<I", (h & 0xFFFF) << 16))[0]
    if math.isinf(f) or math.isnan(f):
        return f
    return Fraction(f)


def rne_bf16_bits(v: Fraction, negative_zero: bool = False) -> int:
    """Round an exact rational to bf16 (nearest, ties to even); return bits."""
    if v == 0:
        return 0x8000 if negative_zero else 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    # make 2^(e-1) <= a < 2^e
    while Fraction(2) ** e <= a:
        e += 1
    while Fraction(2) ** (e - 1) > a:
        e -= 1
    ulp = max(Fraction(2) ** (e - 8), MIN_ULP)
    n = a / ulp
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * ulp
    if r > BF16_MAX:
        return sign | 0x7F80
    if r == 0:
        return sign
    bits = struct.unpack("<I", struct.pack("<f", float(r)))[0]
    assert Fraction(struct.unpack("<f", struct.pack("<I", bits))[0]) == r
    return sign | (bits >> 16)


def exact_dequant_bits(q: int, s: int, b: int) -> int:
    """bf16(s*q + b) rounded once from the exact rational value."""
    sv, bv = bf16_value(s), bf16_value(b)
    v = sv * q + bv
    if v == 0:
        # IEEE: an exact zero sum is -0 only when both addends are -0.
        p_neg_zero = bool(s & 0x8000) and (sv == 0 or q == 0)
        return 0x8000 if (p_neg_zero and b == 0x8000) else 0x0000
    return rne_bf16_bits(v)


def bits_from_torch_bf16(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def random_bf16(rng: random.Random, lo_exp: int, hi_exp: int, sign=None) -> int:
    """A normal bf16 with an unbiased exponent in [lo_exp, hi_exp]."""
    assert -126 <= lo_exp <= hi_exp <= 127
    e = rng.randint(lo_exp, hi_exp) + 127
    m = rng.randint(0, 127)
    sg = (rng.randint(0, 1) if sign is None else sign) << 15
    return sg | (e << 7) | m


# ----------------------------------------------------------------------------
# bf16 rounding
# ----------------------------------------------------------------------------
def _sweep_patterns() -> np.ndarray:
    """Every fp32 exponent and bf16 pattern, with the low halves that decide a
    rounding: exact, just above/below a tie, the tie itself, and random."""
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xBFFF, 0xFFFF],
                    dtype=np.uint32)
    rng = np.random.default_rng(12345)
    lows = np.concatenate([lows, rng.integers(0, 65536, 24, dtype=np.uint32)])
    pats = (hi[:, None] | lows[None, :]).reshape(-1)
    extra = rng.integers(0, 2 ** 32, 1 << 22, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([pats, extra])


def pin_bf16_against_torch(orc):
    pats = _sweep_patterns()
    ours = orc.bf16_from_f32_bits(pats)
    f = torch.from_numpy(pats.view(np.float32).copy())
    ref = bits_from_torch_bf16(f.to(torch.bfloat16))
    nan = np.isnan(pats.view(np.float32))
    ours_nan = (ours & 0x7F80) == 0x7F80
    ours_nan &= (ours & 0x007F) != 0
    assert np.array_equal(ours_nan, nan), "NaN class differs from torch"
    bad = np.nonzero((ours != ref) & ~nan)[0]
    assert bad.size == 0, (
        f"{bad.size} fp32 patterns round differently from torch, e.g. "
        f"{pats[bad[0]]:#010x}: oracle {ours[bad[0]]:#06x} torch {ref[bad[0]]:#06x}")


def load_golden_bf16():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_edges.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            num, den_exp, want = line.split()
            rows.append((int(num), int(den_exp), int(want, 16)))
    return rows


def pin_bf16_golden(orc):
    for num, e, want in load_golden_bf16():
        got = orc.bf16_from_double(math.ldexp(float(num), e))
        assert got == want, f"bf16({num}*2^{e}) = {got:#06x}, expected {want:#06x}"
        if num != 0:  # the stored value also agrees with the rational rounding here
            assert rne_bf16_bits(Fraction(num) * Fraction(2) ** e) == want, (num, e)


# ----------------------------------------------------------------------------
# Dequantization: bf16(s*q + b), one rounding
# ----------------------------------------------------------------------------
def _adversarial_sb(rng: random.Random, bits: int):
    """(s, b) pairs that stress the single rounding."""
    qmax = (1 << bits) - 1
    out = []
    for _ in range(40):          # the workloads' ranges
        s = random_bf16(rng, -12, -6, sign=0)
        b = random_bf16(rng, -9, -3)
        out.append((s, b))
    for _ in range(40):          # wide exponent gaps: tiny s with a large b and back
        out.append((random_bf16(rng, -120, -60, sign=0), random_bf16(rng, -5, 5)))
        out.append((random_bf16(rng, 0, 10, sign=0), random_bf16(rng, -126, -100)))
    for _ in range(30):          # subnormal scales and biases
        out.append((rng.randint(1, 127), rng.randint(0, 0xFFFF) & 0x807F))
    out.append((0x0000, 0x3F80))  # s = 0: W = b exactly
    out.append((0x0000, 0xBF80))
    out.append((0x3F80, 0x0000))  # s = 1, b = 0: W = q
    # Midpoint constructions: s*q lands on a bf16 midpoint when b = 0 for some q,
    # and b = +-2^-k nudges it to just either side or leaves a true tie.
    for _ in range(60):
        e = rng.randint(-20, 5)
        s = random_bf16(rng, e, e, sign=0) | 0x7F   # all-ones mantissa: s*q has 16 bits
        tiny = rng.choice([0, 1, -1])
        if tiny == 0:
            b = 0
        else:
            sv = bf16_value(s)
            mag = sv * Fraction(1, 2 ** 40)
            b = rne_bf16_bits(mag if tiny > 0 else -mag)
        out.append((s, b))
    # Biases that cancel most of s*q (catastrophic cancellation keeps it exact).
    for _ in range(40):
        s = random_bf16(rng, -10, -6, sign=0)
        q = rng.randint(1, qmax)
        b = rne_bf16_bits(-bf16_value(s) * q * Fraction(rng.randint(250, 262), 256))
        out.append((s, b))
    # Overflow: s*q + b beyond bf16's largest finite value.
    out.append((0x7F7F, 0x7F7F))
    out.append((0x7F00, 0x7F7F))
    out.append((0xFF7F, 0xFF00))
    return out


def pin_dequant_exact(orc, bits_list=(2, 3, 4, 5, 6, 8), seed=7):
    rng = random.Random(seed)
    for bits in bits_list:
        qmax = (1 << bits) - 1
        for s, b in _adversarial_sb(rng, bits):
            for q in range(qmax + 1):
                want = exact_dequant_bits(q, s, b)
                got = orc.dequant_one(q, s, b)
                assert got == want, (
                    f"bits={bits} q={q} s={s:#06x} b={b:#06x}: oracle {got:#06x}, "
                    f"exact {want:#06x}")


def pin_dequant_array_matches_scalar(orc, seed=11):
    """oracle_dequant indexes groups along K within a row, scale/bias [N, K/g]."""
    rng = np.random.default_rng(seed)
    for bits, group in [(4, 64), (3, 32), (8, 128), (2, 64)]:
        N, K = 5, 3 * group
        G = K // group
        codes = rng.integers(0, 1 << bits, (N, K), dtype=np.uint8)
        s = rng.integers(0x3A00, 0x3D00, (N, G), dtype=np.uint16)
        b = rng.integers(0xBC00, 0xBE00, (N, G), dtype=np.uint16)
        W = orc.dequant(bits, group, codes, s, b)
        for n in range(N):
            for k in range(K):
                j = k // group
                assert W[n, k] == exact_dequant_bits(int(codes[n, k]), int(s[n, j]), int(b[n, j]))


# ----------------------------------------------------------------------------
# Projection
# ----------------------------------------------------------------------------
def _small_problem(rng, bits, group, M, N, K):
    G = K // group
    codes = rng.integers(0, 1 << bits, (N, K), dtype=np.uint8)
    s = (np.abs(rng.normal(0, 0.02, (N, G))) / 8).astype(np.float32)
    s_b = bits_from_torch_bf16(torch.from_numpy(s).to(torch.bfloat16))
    sv = torch.from_numpy(s_b.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    bb = (-(2.0 ** (bits - 1)) * sv + rng.normal(0, 1e-3, (N, G))).astype(np.float32)
    b_b = bits_from_torch_bf16(torch.from_numpy(bb).to(torch.bfloat16))
    x = rng.normal(0, 1, (M, K)).astype(np.float32)
    x_b = bits_from_torch_bf16(torch.from_numpy(x).to(torch.bfloat16))
    return x_b, codes, s_b, b_b


def pin_qmm_bruteforce(orc, seed=3):
    rng = np.random.default_rng(seed)
    for bits, group, M, N, K in [(4, 64, 2, 6, 128), (3, 32, 2, 4, 96), (8, 32, 1, 3, 64),
                                 (2, 128, 2, 5, 128), (5, 64, 1, 4, 64), (6, 32, 2, 3, 64)]:
        x, codes, s, b = _small_problem(rng, bits, group, M, N, K)
        y = orc.qmm(bits, group, x, codes, s, b)
        G = K // group
        for m in range(M):
            for n in range(N):
                terms = []
                for k in range(K):
                    j = k // group
                    w = bf16_value(exact_dequant_bits(int(codes[n, k]), int(s[n, j]), int(b[n, j])))
                    terms.append(w * bf16_value(int(x[m, k])))
                exact = sum(terms, Fraction(0))
                scale = sum((abs(t) for t in terms), Fraction(0))
                err = abs(Fraction(float(y[m, n])) - exact)
                assert err <= scale * Fraction(1, 2 ** 44), (bits, group, m, n, float(err), float(scale))


def pin_qmm_vs_float64_matmul(orc, seed=5):
    rng = np.random.default_rng(seed)
    for bits, group, M, N, K in [(4, 64, 4, 64, 512), (8, 32, 3, 32, 256), (3, 64, 2, 48, 384)]:
        x, codes, s, b = _small_problem(rng, bits, group, M, N, K)
        W = orc.dequant(bits, group, codes, s, b)
        Wd = torch.from_numpy(W.view(np.int16).copy()).view(torch.bfloat16).double()
        xd = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double()
        ref = (xd @ Wd.T).numpy()
        mag = (xd.abs() @ Wd.abs().T).numpy()
        y = orc.qmm(bits, group, x, codes, s, b)
        assert np.all(np.abs(y - ref) <= 1e-12 * mag + 1e-300), np.max(np.abs(y - ref) / mag)
        y4 = orc.qmm(bits, group, x, codes, s, b, nthreads=4)
        assert np.array_equal(y, y4), "threaded oracle differs from single-threaded"


def pin_one_hot_rows(orc, seed=9):
    """x = 2^j * e_k reproduces 2^j * W[:, k] exactly."""
    rng = np.random.default_rng(seed)
    for bits, group, N, K in [(4, 64, 16, 256), (2, 128, 8, 256), (8, 32, 8, 64)]:
        _, codes, s, b = _small_problem(rng, bits, group, 1, N, K)
        W = orc.dequant(bits, group, codes, s, b)
        ks = list(range(0, K, max(1, K // 16))) + [K - 1]
        for k in ks:
            for j in (0, 3, -2):
                x = np.zeros((1, K), dtype=np.uint16)
                x[0, k] = rne_bf16_bits(Fraction(2) ** j)
                y = orc.qmm(bits, group, x, codes, s, b)
                for n in range(N):
                    want = bf16_value(int(W[n, k])) * Fraction(2) ** j
                    assert Fraction(float(y[0, n])) == want, (bits, k, j, n)


def pin_constant_code_groups(orc, seed=13):
    """Constant codes c per group: y = sum_g bf16(s_g*c_g + b_g) * sum_{k in g} x_k."""
    rng = np.random.default_rng(seed)
    for bits, group in [(4, 64), (3, 32), (8, 128)]:
        N, K, M = 4, 4 * group, 2
        G = K // group
        x, _, s, b = _small_problem(rng, bits, group, M, N, K)
        c = rng.integers(0, 1 << bits, (N, G), dtype=np.uint8)
        codes = np.repeat(c, group, axis=1)
        y = orc.qmm(bits, group, x, codes, s, b)
        for m in range(M):
            for n in range(N):
                acc = Fraction(0)
                mag = Fraction(0)
                for j in range(G):
                    w = bf16_value(exact_dequant_bits(int(c[n, j]), int(s[n, j]), int(b[n, j])))
                    sx = sum((bf16_value(int(v)) for v in x[m, j * group:(j + 1) * group]),
                             Fraction(0))
                    acc += w * sx
                    mag += abs(w) * sum((abs(bf16_value(int(v))) for v in
                                         x[m, j * group:(j + 1) * group]), Fraction(0))
                assert abs(Fraction(float(y[m, n])) - acc) <= mag * Fraction(1, 2 ** 44)


def pin_group_sum_identity(orc, seed=17):
    """|y - sum_g(s_g*sum q x + b_g*sum x)| <= 2^-8 * sum |s q + b| |x|:
    each bf16 weight is within a relative 2^-8 of the exact s*q + b."""
    rng = np.random.default_rng(seed)
    for bits, group, M, N, K in [(4, 64, 2, 32, 512), (8, 32, 1, 16, 256), (2, 128, 2, 16, 256)]:
        x, codes, s, b = _small_problem(rng, bits, group, M, N, K)
        y = orc.qmm(bits, group, x, codes, s, b)
        y_gs, mag = orc.qmm_groupsum(bits, group, x, codes, s, b)
        dev = np.abs(y - y_gs)
        assert np.all(dev <= 2.0 ** -8 * mag * (1 + 1e-9)), float(np.max(dev / mag))
        # The two forms do differ (the bf16 rounding is real), by far less than the bound.
        assert np.max(dev / mag) > 0


def pin_qmm_groupsum_bruteforce(orc, seed=23):
    """The exact-codes form against exact rational arithmetic on tiny shapes:
    y_gs = sum_g (s_g * sum_{k in g} q_k x_k + b_g * sum_{k in g} x_k), with the
    codes exact (no bf16 rounding of the weights); and mag = sum |s q + b| |x|."""
    rng = np.random.default_rng(seed)
    for bits, group, M, N, K in [(4, 64, 2, 3, 128), (3, 32, 1, 2, 96), (8, 128, 1, 2, 256), (6, 32, 2, 2, 64)]:
        x, codes, s, b = _small_problem(rng, bits, group, M, N, K)
        y_gs, mag = orc.qmm_groupsum(bits, group, x, codes, s, b)
        G = K // group
        for m in range(M):
            for n in range(N):
                exact = Fraction(0)
                amag = Fraction(0)
                for j in range(G):
                    sv, bv = bf16_value(int(s[n, j])), bf16_value(int(b[n, j]))
                    xs = [bf16_value(int(v)) for v in x[m, j * group:(j + 1) * group]]
                    qs = [int(q) for q in codes[n, j * group:(j + 1) * group]]
                    exact += sv * sum((q * xv for q, xv in zip(qs, xs)), Fraction(0)) + bv * sum(xs, Fraction(0))
                    amag += sum((abs(sv * q + bv) * abs(xv) for q, xv in zip(qs, xs)), Fraction(0))
                assert abs(Fraction(float(y_gs[m, n])) - exact) <= amag * Fraction(1, 2 ** 44), (bits, group, m, n)
                assert abs(Fraction(float(mag[m, n])) - amag) <= amag * Fraction(1, 2 ** 44), (bits, group, m, n)


def _embed_exact_bits(orc_w_bits: int, scale_bits: int) -> int:
    """bf16(w * scale) from the exact product (w, scale finite bf16 patterns)."""
    w, sc = bf16_value(orc_w_bits), bf16_value(scale_bits)
    if isinstance(w, float) or isinstance(sc, float):
        raise ValueError("finite values only")
    prod = w * sc
    neg_zero = prod == 0 and ((orc_w_bits >> 15) ^ (scale_bits >> 15)) == 1
    return rne_bf16_bits(prod, negative_zero=neg_zero)


def pin_embed_rows_exact(orc, seed=19):
    """Scaled embedding rows against exact arithmetic: each output is the exact
    product of the exactly rounded weight and the scale, rounded once; the
    weight is the exact bf16(s*q + b) (two roundings in all, no fewer)."""
    rng = np.random.default_rng(seed)
    hidden = rne_bf16_bits(Fraction(math.sqrt(5376)))          # bf16(sqrt(hidden)), Gemma's embedding scale
    for bits, group, N, K in [(4, 64, 9, 128), (3, 32, 5, 96), (8, 128, 4, 256), (2, 32, 6, 64)]:
        _, codes, s, b = _small_problem(rng, bits, group, 1, N, K)
        ids = rng.integers(0, N, 7).astype(np.int32)
        ids[0] = N - 1
        for scale in (hidden, 0x3F80, 0x4180, 0xC0A0, 0x3DCD):   # sqrt(5376), 1, 16, -5, ~0.1
            out = orc.embed_rows(bits, group, codes, s, b, ids, scale)
            for t, n in enumerate(ids):
                for k in range(0, K, max(1, K // 24)):
                    wb = exact_dequant_bits(int(codes[n, k]), int(s[n, k // group]), int(b[n, k // group]))
                    assert int(out[t, k]) == _embed_exact_bits(wb, scale), (bits, t, k, hex(scale))


def pin_embed_rows_special_cases(orc, seed=23):
    """No scale gives the dequantized rows; scale 1 gives them too; a power-of-two
    scale multiplies exactly (no overflow or underflow at these magnitudes)."""
    rng = np.random.default_rng(seed)
    for bits, group, N, K in [(4, 64, 8, 256), (6, 32, 4, 128)]:
        _, codes, s, b = _small_problem(rng, bits, group, 1, N, K)
        W = orc.dequant(bits, group, codes, s, b)
        ids = np.arange(N, dtype=np.int32)[::-1].copy()
        assert np.array_equal(orc.embed_rows(bits, group, codes, s, b, ids, None), W[ids])
        assert np.array_equal(orc.embed_rows(bits, group, codes, s, b, ids, 0x3F80), W[ids])
        out = orc.embed_rows(bits, group, codes, s, b, ids, 0x4100)   # 8.0
        for t, n in enumerate(ids):
            for k in range(K):
                assert bf16_value(int(out[t, k])) == 8 * bf16_value(int(W[n, k]))


def pin_qmm_groupsum_given_bruteforce(orc, seed=29):
    """The exact-codes form with supplied group sums of x, against exact
    rational arithmetic: sum_g (s_g * sum q x + b_g * xs_g), the codes exact and
    the sums taken as given (here: fp32 values that are not the exact sums, so
    that a form that recomputes them from x fails)."""
    rng = np.random.default_rng(seed)
    for bits, group, M, N, K in [(4, 64, 2, 3, 128), (3, 32, 1, 2, 96), (8, 128, 2, 2, 256), (5, 32, 1, 3, 64)]:
        x, codes, s, b = _small_problem(rng, bits, group, M, N, K)
        G = K // group
        xs = rng.normal(0, 8, (M, G)).astype(np.float32)
        y = orc.qmm_groupsum_given(bits, group, x, xs, codes, s, b)
        for m in range(M):
            for n in range(N):
                exact = Fraction(0)
                amag = Fraction(0)
                for j in range(G):
                    sv, bv = bf16_value(int(s[n, j])), bf16_value(int(b[n, j]))
                    xv = [bf16_value(int(v)) for v in x[m, j * group:(j + 1) * group]]
                    qs = [int(q) for q in codes[n, j * group:(j + 1) * group]]
                    term_q = sv * sum((q * v for q, v in zip(qs, xv)), Fraction(0))
                    term_b = bv * Fraction(float(xs[m, j]))
                    exact += term_q + term_b
                    amag += abs(term_q) + abs(term_b)
                assert abs(Fraction(float(y[m, n])) - exact) <= amag * Fraction(1, 2 ** 44), (bits, group, m, n)
    # with the exact sums of x supplied, the form equals the exact-codes form within double rounding
    x, codes, s, b = _small_problem(rng, 4, 64, 2, 8, 256)
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    xs = xv.reshape(2, 4, 64).sum(axis=2).astype(np.float32)   # the sums of x rounded to fp32
    y = orc.qmm_groupsum_given(4, 64, x, xs, codes, s, b)
    y_gs, mag = orc.qmm_groupsum(4, 64, x, codes, s, b)
    bound = np.abs(xs.astype(np.float64) - xv.reshape(2, 4, 64).sum(axis=2))
    bsum = np.abs(torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).double().numpy())
    assert np.all(np.abs(y - y_gs) <= (bound @ bsum.T) + 1e-12 * mag + 1e-300)


# -- GeGLU (mlx_lm's gelu_approx(gate) * up as bf16 operations) ------------------
def _bf16_tensor(bits_u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits_u16, dtype=np.uint16).view(np.int16).copy()).view(torch.bfloat16)


def _geglu_inputs(rng, n):
    """bf16 gate/up patterns over many magnitudes, both signs, with zeros,
    subnormals and the values where tanh saturates."""
    mags = np.concatenate([rng.normal(0, 1, n // 2), rng.normal(0, 4, n // 4),
                           np.exp2(rng.uniform(-140, 20, n - n // 2 - n // 4)) * rng.choice([-1, 1], n - n // 2 - n // 4)])
    gate = bits_from_torch_bf16(torch.from_numpy(mags.astype(np.float32)).to(torch.bfloat16))
    up = bits_from_torch_bf16(torch.from_numpy(rng.normal(0, 2, n).astype(np.float32)).to(torch.bfloat16))
    gate[:4] = [0x0000, 0x8000, 0x0001, 0x8001]
    return gate, up


def pin_geglu_against_torch_bf16_ops(orc, seed=31):
    """Each step of the chain against torch's own bf16 arithmetic (a library:
    every op on bf16 tensors rounds its fp32 result to bf16; fp32 holds the
    exact product of two bf16 values and the exact cube of one): torch's
    result must be one of the oracle's two (they differ only where tanh's
    rounding is ambiguous)."""
    rng = np.random.default_rng(seed)
    gate, up = _geglu_inputs(rng, 200000)
    lo, hi = orc.geglu(gate, up)
    g, u = _bf16_tensor(gate), _bf16_tensor(up)
    gf = g.float()
    c3 = (gf * gf * gf).to(torch.bfloat16)
    c1 = torch.tensor(0.044715, dtype=torch.bfloat16)
    c2 = torch.tensor(math.sqrt(2 / math.pi), dtype=torch.bfloat16)
    z = g + c1 * c3
    t = torch.tanh(c2 * z)
    h = (torch.tensor(0.5, dtype=torch.bfloat16) * g) * (1 + t) * u
    hb = bits_from_torch_bf16(h)
    ok = (hb == lo) | (hb == hi)
    nan = np.isnan(h.float().numpy())
    ok |= nan & np.isnan(_bf16_tensor(lo).float().numpy())
    assert np.all(ok), f"{int(np.sum(~ok))} outputs differ from torch's bf16 operations, e.g. gate {gate[~ok][0]:#06x}"
    amb = np.mean(lo != hi)
    assert amb < 0.01, f"tanh's rounding is ambiguous on {amb:.3%} of outputs"


def pin_geglu_closed_forms(orc, seed=37):
    """Special cases with closed forms: gate = +-0 gives a zero; gate >= 16
    saturates tanh to 1 in bf16, so h = bf16(gate * up) exactly; gate <= -16
    gives 1 + tanh = 0 and h = +-0; |gate| <= 2^-12 leaves 1 + tanh = 1, so
    h = bf16(bf16(gate / 2) * up)."""
    rng = np.random.default_rng(seed)
    n = 4000
    up = bits_from_torch_bf16(torch.from_numpy(rng.normal(0, 3, n).astype(np.float32)).to(torch.bfloat16))
    big = np.array([random_bf16(random.Random(i), 4, 40, sign=0) for i in range(n)], dtype=np.uint16)
    lo, hi = orc.geglu(big, up)
    for i in range(n):
        want = rne_bf16_bits(bf16_value(int(big[i])) * bf16_value(int(up[i])),
                             negative_zero=bool(up[i] & 0x8000))
        assert lo[i] == want and hi[i] == want, (hex(big[i]), hex(up[i]), hex(lo[i]), hex(want))
    neg = big | 0x8000
    lo, hi = orc.geglu(neg, up)
    assert np.all((lo & 0x7FFF) == 0) and np.all((hi & 0x7FFF) == 0)
    tiny = np.array([random_bf16(random.Random(7 * i), -120, -12) for i in range(n)], dtype=np.uint16)
    lo, hi = orc.geglu(tiny, up)
    for i in range(n):
        half = rne_bf16_bits(bf16_value(int(tiny[i])) / 2, negative_zero=bool(tiny[i] & 0x8000))
        want = rne_bf16_bits(bf16_value(half) * bf16_value(int(up[i])),
                             negative_zero=bool((half ^ up[i]) & 0x8000))
        assert lo[i] == want and hi[i] == want, (hex(tiny[i]), hex(up[i]), hex(lo[i]), hex(want))
    zeros = np.array([0x0000, 0x8000] * 4, dtype=np.uint16)
    lo, _ = orc.geglu(zeros, up[:8])
    assert np.all((lo & 0x7FFF) == 0)


def pin_geglu_near_textbook_gelu(orc, seed=41):
    """Against the GELU tanh approximation evaluated in float64 (the textbook
    formula, no roundings): on |gate| <= 6 the bf16 chain stays within
    2^-6 * (1 + |gate|) of gelu(gate) (up = 1), which a wrong constant, a
    missing term or swapped operands does not."""
    rng = np.random.default_rng(seed)
    gv = rng.uniform(-6, 6, 50000).astype(np.float32)
    gate = bits_from_torch_bf16(torch.from_numpy(gv).to(torch.bfloat16))
    one = np.full(gate.shape, 0x3F80, dtype=np.uint16)
    lo, hi = orc.geglu(gate, one)
    x = _bf16_tensor(gate).double().numpy()
    ref = 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))
    for h in (lo, hi):
        got = _bf16_tensor(h).double().numpy()
        assert np.all(np.abs(got - ref) <= 2.0 ** -6 * (1 + np.abs(x))), float(np.max(np.abs(got - ref)))
    # and gate/up enter in their roles: h(g, u) != h(u, g) in general
    up = bits_from_torch_bf16(torch.from_numpy(rng.uniform(-6, 6, 50000).astype(np.float32)).to(torch.bfloat16))
    a, _ = orc.geglu(gate, up)
    b, _ = orc.geglu(up, gate)
    assert np.mean(a != b) > 0.5


ALL_PINS = [
    pin_bf16_golden,
    pin_bf16_against_torch,
    pin_dequant_exact,
    pin_dequant_array_matches_scalar,
    pin_qmm_bruteforce,
    pin_qmm_vs_float64_matmul,
    pin_one_hot_rows,
    pin_constant_code_groups,
    pin_group_sum_identity,
    pin_qmm_groupsum_bruteforce,
    pin_embed_rows_exact,
    pin_embed_rows_special_cases,
    pin_qmm_groupsum_given_bruteforce,
    pin_geglu_against_torch_bf16_ops,
    pin_geglu_closed_forms,
    pin_geglu_near_textbook_gelu,
]
