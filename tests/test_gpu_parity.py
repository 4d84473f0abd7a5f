"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Unpacking and dequantization must be bit-exact; projection outputs must lie
within |y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref row).  Inputs come from
the seeded generators (group_affine_bit_gb300.synth) on the CPU and are copied
to the GPU, so both sides read the same values.
"""
import random

import numpy as np
import pytest
import torch

import oracle_pins as P
from group_affine_bit_gb300 import api, build, synth
from helpers import assert_within_tolerance, bf16_to_f64, u16

pytestmark = pytest.mark.gpu

ALL_WIDTHS = [(b, g) for b in (2, 3, 4, 5, 6, 8) for g in (32, 64, 128)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return api.lib()


def cuda(*ts):
    return [t.cuda() for t in ts]


def packed_problem(bits, group, M, N, K, seed):
    x, codes, s, b = synth.problem(bits, group, M, N, K, seed)
    xd, cd, sd, bd = cuda(x, codes, s, b)
    w = api.pack(cd, sd, bd, bits, group)
    return (x, codes, s, b), w, xd


def oracle_y(orc, bits, group, x, codes, s, b, nthreads=8):
    return orc.qmm(bits, group, u16(x), codes.numpy(), u16(s), u16(b), nthreads=nthreads)


# --------------------------------------------------------------- dequant
@pytest.mark.parametrize("bits,group", ALL_WIDTHS)
def test_dequant_bit_exact(orc, bits, group):
    N, K = 37, 3 * 128 + group * (1 if group < 128 else 0) + (group if group == 32 else 0)
    K -= K % group
    _, codes, s, b = synth.problem(bits, group, 1, N, K, seed=100 + bits * 7 + group)
    w = api.pack(*cuda(codes, s, b), bits, group)
    got = u16(api.dequant(w))
    want = orc.dequant(bits, group, codes.numpy(), u16(s), u16(b))
    mism = np.argwhere(got != want)
    assert mism.size == 0, f"{len(mism)} weights differ, first at {mism[0]}"


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_dequant_adversarial_scales_bit_exact(orc, bits):
    """Tiny and subnormal scales, wide exponent gaps, exact bf16 midpoints and
    overflow: the device's single-rounding fma against the exact rounding."""
    rng = random.Random(1234 + bits)
    pairs = P._adversarial_sb(rng, bits)
    group = 32
    qmax = (1 << bits) - 1
    N = len(pairs)
    K = 128
    codes = np.zeros((N, K), dtype=np.uint8)
    for n in range(N):
        codes[n] = np.arange(K) % (qmax + 1)
    s = np.array([[p[0]] * (K // group) for p in pairs], dtype=np.uint16)
    b = np.array([[p[1]] * (K // group) for p in pairs], dtype=np.uint16)
    st = synth.from_bits_u16(s)
    bt = synth.from_bits_u16(b)
    w = api.pack(*cuda(torch.from_numpy(codes), st, bt), bits, group)
    got = u16(api.dequant(w))
    want = orc.dequant(bits, group, codes, s, b)
    nan_g = (got & 0x7F80) == 0x7F80
    nan_g &= (got & 0x7F) != 0
    nan_w = (want & 0x7F80) == 0x7F80
    nan_w &= (want & 0x7F) != 0
    assert np.array_equal(nan_g, nan_w)
    diff = np.argwhere((got != want) & ~nan_w)
    if diff.size:
        n, k = diff[0]
        raise AssertionError(
            f"{len(diff)} weights differ; first n={n} k={k} q={codes[n, k]} s={s[n, 0]:#06x} "
            f"b={b[n, 0]:#06x}: gpu {got[n, k]:#06x} oracle {want[n, k]:#06x}")


# --------------------------------------------------------------- run
def test_tiny_config(orc):
    c = synth.TINY
    (x, codes, s, b), w, xd = packed_problem(c["bits"], c["group"], c["M"], c["N"], c["K"], c["seed"])
    y = api.run(w, xd)
    assert_within_tolerance(y, oracle_y(orc, c["bits"], c["group"], x, codes, s, b), "tiny")


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 13, 16])
@pytest.mark.parametrize("N,K", [(37, 384), (80, 640), (512, 1024)])
def test_run_small_shapes(orc, M, N, K):
    (x, codes, s, b), w, xd = packed_problem(4, 64, M, N, K, seed=M * 1000 + N + K)
    y = api.run(w, xd)
    assert_within_tolerance(y, oracle_y(orc, 4, 64, x, codes, s, b), f"M={M} N={N} K={K}")


@pytest.mark.parametrize("bits,group", ALL_WIDTHS)
@pytest.mark.parametrize("M", [1, 16])
def test_run_all_widths(orc, bits, group, M):
    N, K = 45, 512 + (group if group < 128 else 0)
    (x, codes, s, b), w, xd = packed_problem(bits, group, M, N, K, seed=bits * 100 + group + M)
    y = api.run(w, xd)
    assert_within_tolerance(y, oracle_y(orc, bits, group, x, codes, s, b), f"{bits}b g{group} M{M}")


@pytest.mark.parametrize("N,K", [(320, 8192), (96, 21504), (48, 5376)])
@pytest.mark.parametrize("M", [1, 16])
def test_run_split_depth(orc, N, K, M):
    """Few row tiles over a long depth: the depth is split across CTAs and the
    partials merged in slice order."""
    (x, codes, s, b), w, xd = packed_problem(4, 64, M, N, K, seed=N + K + M)
    y = api.run(w, xd)
    assert_within_tolerance(y, oracle_y(orc, 4, 64, x, codes, s, b), f"split N={N} K={K}")
    y2 = api.run(w, xd)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "split-depth result not deterministic"


@pytest.mark.parametrize("M", [1, 7, 16])
@pytest.mark.parametrize("bits,group", [(4, 64), (2, 128), (3, 64), (5, 32), (6, 64), (8, 32)])
def test_one_hot_rows_reproduce_weight_columns(orc, bits, group, M):
    """x rows = 2^j e_k give y[m, :] = 2^j W[:, k] exactly (one nonzero
    product): the decode kernel's matrix-fragment dequantization, bit for bit,
    for every width of codes.  W is the oracle's."""
    N, K = 200, 768
    _, codes, s, b = synth.problem(bits, group, 1, N, K, seed=77 + bits + group)
    w = api.pack(*cuda(codes, s, b), bits, group)
    W = synth.from_bits_u16(orc.dequant(bits, group, codes.numpy(), u16(s), u16(b))).float().cuda()
    ks = torch.randint(0, K, (M,), generator=torch.Generator().manual_seed(M))
    js = torch.tensor([0, 3, -2, 1, 0, -1, 2, 0] * 2)[:M]
    x = torch.zeros(M, K)
    for m in range(M):
        x[m, ks[m]] = 2.0 ** float(js[m])
    y = api.run(w, x.to(torch.bfloat16).cuda())
    want = (W[:, ks.cuda()].T * (2.0 ** js.float().cuda())[:, None]).to(torch.bfloat16)
    assert torch.equal(y.view(torch.int16), want.view(torch.int16))


def test_deterministic_repeat():
    (_, _, _, _), w, xd = packed_problem(4, 64, 1, 30720, 3840, seed=1)
    y1 = api.run(w, xd)
    y2 = api.run(w, xd)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("M", [1, 4, 16])
def test_stacked_equals_separate_and_oracle(orc, M):
    """A stacked call (the q/k/v shapes of a layer at a short depth, one
    launch) gives each projection the bits of its own call, and each output
    lies within the tolerance of the oracle's projection."""
    bits, group, K = 4, 64, 1024
    g = synth.generator(55)
    ws, singles, tables = [], [], []
    xc = synth.activations(M, K, g)
    x = xc.cuda()
    for N in (384, 100, 1024):
        codes, s, b = synth.affine_table(bits, group, N, K, g)
        w = api.pack(*cuda(codes, s, b), bits, group)
        ws.append(w)
        tables.append((codes, s, b))
        singles.append(api.run(w, x))
    ys = api.run_stacked(ws, x)
    for i, (a, c, (codes, s, b)) in enumerate(zip(ys, singles, tables)):
        assert torch.equal(a.view(torch.int16), c.view(torch.int16))
        assert_within_tolerance(a, oracle_y(orc, bits, group, xc, codes, s, b), f"stacked {i} M={M}")


def test_stacked_gate_up_halves_against_oracle(orc):
    """The gate/up decode configuration as two stacked halves of 15360 rows
    (one launch over both), each against the oracle."""
    c = synth.GATE_UP_DECODE
    bits, group, K = c["bits"], c["group"], c["K"]
    g = synth.generator(c["seed"] + 500)
    xc = synth.activations(1, K, g)
    tables = [synth.affine_table(bits, group, c["N"] // 2, K, g) for _ in range(2)]
    ws = [api.pack(*cuda(*t), bits, group) for t in tables]
    ys = api.run_stacked(ws, xc.cuda())
    for i, (y, (codes, s, b)) in enumerate(zip(ys, tables)):
        assert_within_tolerance(y, oracle_y(orc, bits, group, xc, codes, s, b, nthreads=16), f"gate/up half {i}")


@pytest.mark.parametrize("M", [4, 20])
def test_non_finite_activations_propagate(orc, M):
    """Infinite and NaN activations propagate as IEEE arithmetic does: an
    output is NaN exactly where the oracle's float64 sum is NaN and infinite
    with the oracle's sign; rows with finite activations stay within the
    tolerance.  (M = 4 runs the decode kernel, M = 20 the prompt kernel.)"""
    bits, group, N, K = 4, 64, 300, 640
    x, codes, s, b = synth.problem(bits, group, M, N, K, seed=4242 + M)
    xf = x.float()
    xf[1, 7] = float("inf")                  # a positive infinity
    xf[2, 130] = float("nan")                # a NaN
    xf[3, 5], xf[3, 600] = float("-inf"), float("inf")   # both signs: inf - inf where the weights agree in sign
    x = xf.to(torch.bfloat16)
    w = api.pack(*cuda(codes, s, b), bits, group)
    y = api.run(w, x.cuda()).float().cpu().numpy().astype(np.float64)
    y_ref = oracle_y(orc, bits, group, x, codes, s, b)
    bad_rows = [1, 2, 3]
    for m in bad_rows:
        assert np.array_equal(np.isnan(y[m]), np.isnan(y_ref[m])), f"row {m}: NaN pattern differs"
        inf = np.isinf(y_ref[m])
        assert np.array_equal(np.isinf(y[m]), inf), f"row {m}: infinity pattern differs"
        assert np.array_equal(np.sign(y[m][inf]), np.sign(y_ref[m][inf])), f"row {m}: infinity signs differ"
        assert not np.any(np.isfinite(y_ref[m])), "every output of a row with a non-finite input is non-finite"
    assert np.isnan(y_ref[3]).any() and np.isinf(y_ref[3]).any()
    ok_rows = [m for m in range(M) if m not in bad_rows]
    got = api.run(w, x.cuda())
    from helpers import tolerance_report
    ok, worst, nbad = tolerance_report(u16(got)[ok_rows], y_ref[ok_rows])
    assert ok, f"finite rows: {nbad} outputs out of tolerance (worst {worst:.3f})"


def test_empty_and_degenerate_shapes():
    bits, group = 4, 64
    # M = 0: nothing to compute
    _, codes, s, b = synth.problem(bits, group, 1, 32, 128, seed=5)
    w = api.pack(*cuda(codes, s, b), bits, group)
    y = api.run(w, torch.zeros(0, 128, dtype=torch.bfloat16, device="cuda"))
    assert y.shape == (0, 32)
    # K = 0: every output is the empty sum, +0
    w0 = api.pack(torch.zeros(16, 0, dtype=torch.uint8, device="cuda"),
                  torch.zeros(16, 0, dtype=torch.bfloat16, device="cuda"),
                  torch.zeros(16, 0, dtype=torch.bfloat16, device="cuda"), bits, group)
    y0 = torch.full((3, 16), 7.0, dtype=torch.bfloat16, device="cuda")
    api.run(w0, torch.zeros(3, 0, dtype=torch.bfloat16, device="cuda"), y=y0)
    assert torch.equal(y0.view(torch.int16), torch.zeros_like(y0.view(torch.int16)))
    # N = 0: nothing written
    wn = api.pack(torch.zeros(0, 128, dtype=torch.uint8, device="cuda"),
                  torch.zeros(0, 2, dtype=torch.bfloat16, device="cuda"),
                  torch.zeros(0, 2, dtype=torch.bfloat16, device="cuda"), bits, group)
    assert api.run(wn, torch.zeros(2, 128, dtype=torch.bfloat16, device="cuda")).shape == (2, 0)


def test_workspace_left_zeroed():
    (_, _, _, _), w, xd = packed_problem(4, 64, 1, 96, 21504, seed=9)
    ws = api.Workspace()
    api.run(w, xd, workspace=ws)
    torch.cuda.synchronize()
    need = api.workspace_bytes(w, 1)
    assert need > 0
    assert int(ws.buf[:api.WORKSPACE_ZEROED].count_nonzero()) == 0
    assert api.workspace_status(ws.buf) == 0


# --------------------------------------------------------------- standard workloads
def test_gate_up_decode_config(orc):
    c = synth.GATE_UP_DECODE
    (x, codes, s, b), w, xd = packed_problem(c["bits"], c["group"], c["M"], c["N"], c["K"], c["seed"])
    y = api.run(w, xd)
    assert_within_tolerance(y, oracle_y(orc, c["bits"], c["group"], x, codes, s, b, nthreads=16), "gate/up M=1")


@pytest.mark.parametrize("M,bits,group", synth.SWEEP_CASES)
def test_lane_width_sweep_config(orc, M, bits, group):
    c = synth.SWEEP_SHAPE
    (x, codes, s, b), w, xd = packed_problem(bits, group, M, c["N"], c["K"], c["seed"])
    y = api.run(w, xd)
    assert_within_tolerance(y, oracle_y(orc, bits, group, x, codes, s, b, nthreads=16),
                            f"sweep M={M} {bits}b g{group}")


def test_workspace_reused_across_shapes():
    """One workspace serving plans of different sizes in turn: every call must
    leave the status word and the merge counters zero, whatever the previous
    plan left in its partial-sum slots."""
    ws = api.Workspace()
    shapes = [(1, 512, 8192), (1, 96, 21504), (16, 40, 3840), (1, 3000, 1024), (3, 96, 21504)]
    probs = [packed_problem(4, 64, M, N, K, seed=M + N + K) for M, N, K in shapes]
    outs = []
    for _ in range(2):
        for (_, w, xd) in probs:
            outs.append(api.run(w, xd, workspace=ws))
            torch.cuda.synchronize()
            assert int(ws.buf[:api.WORKSPACE_ZEROED].count_nonzero()) == 0, "counters not left zeroed"
    n = len(probs)
    for a, b in zip(outs[:n], outs[n:]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M", [1, 40])
def test_stacked_with_an_empty_projection(M):
    """A stack that holds a projection with no rows between two others: the
    empty one is skipped (nothing to cut, nothing written) and the others
    give the bits of their separate calls, on both kernels."""
    bits, group, K = 4, 64, 512
    (_, c1, s1, b1), w1, xd = packed_problem(bits, group, M, 300, K, seed=61)
    _, c2, s2, b2 = synth.problem(bits, group, M, 500, K, seed=62)
    w2 = api.pack(*cuda(c2, s2, b2), bits, group)
    wn = api.pack(torch.zeros(0, K, dtype=torch.uint8, device="cuda"),
                  torch.zeros(0, K // group, dtype=torch.bfloat16, device="cuda"),
                  torch.zeros(0, K // group, dtype=torch.bfloat16, device="cuda"), bits, group)
    y1, yn, y2 = api.run_stacked([w1, wn, w2], xd)
    torch.cuda.synchronize()
    assert yn.shape == (M, 0)
    assert torch.equal(y1.view(torch.int16), api.run(w1, xd).view(torch.int16))
    assert torch.equal(y2.view(torch.int16), api.run(w2, xd).view(torch.int16))
