"""Parity of the exact-codes decode form (affqmm_run_exact) with the oracle's
exact-codes function (oracle_qmm_groupsum): y = sum_g s_g * sum q x + b_g * sum x
with the codes exact, within |y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref row)
-- every width and group, M = 1..16, ragged shapes, a long split depth, the
gate/up decode shape on sampled rows -- and deterministic."""
import numpy as np
import pytest
import torch

from group_affine_bit_gb300 import api, build, synth
from helpers import assert_within_tolerance, u16

pytestmark = pytest.mark.gpu

ALL_WIDTHS = [(b, g) for b in (2, 3, 4, 5, 6, 8) for g in (32, 64, 128)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return api.lib()


def _check(orc, bits, group, M, N, K, seed, rows=None):
    x, codes, s, b = synth.problem(bits, group, M, N, K, seed)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    y = api.run_exact(w, x.cuda(), workspace=api.Workspace())
    y2 = api.run_exact(w, x.cuda(), workspace=api.Workspace())
    torch.cuda.synchronize()
    what = f"exact {bits}b g{group} M={M} N={N} K={K}"
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), f"{what}: not deterministic"
    sel = np.arange(N) if rows is None else np.asarray(rows)
    y_ref, _ = orc.qmm_groupsum(bits, group, u16(x), codes.numpy()[sel], u16(s)[sel], u16(b)[sel])
    assert_within_tolerance(y[:, torch.as_tensor(sel, device="cuda")], y_ref, what)
    return y, w, x


@pytest.mark.parametrize("bits,group", ALL_WIDTHS)
def test_exact_all_widths(orc, bits, group):
    # a ragged depth for groups 32 and 64 (the last 128-deep block part full)
    _check(orc, bits, group, 3, 200, 512 + (group if group < 128 else 0), 41)


@pytest.mark.parametrize("M", [1, 2, 8, 9, 16])
def test_exact_decode_rows(orc, M):
    _check(orc, 4, 64, M, 384, 1024, 42)


def test_exact_long_split_depth(orc):
    # 2 row tiles x 168 depth blocks: every tile is cut across many CTAs
    _check(orc, 4, 64, 16, 200, 21504, 43)


def test_exact_gate_up_shape_sampled_rows(orc):
    c = synth.GATE_UP_DECODE
    rows = np.random.default_rng(44).choice(c["N"], 96, replace=False)
    _check(orc, c["bits"], c["group"], c["M"], c["N"], c["K"], c["seed"], rows=np.sort(rows))


def test_exact_and_rounded_forms_differ_but_agree_closely(orc):
    # the two forms differ only by the bf16 rounding of s*q + b
    y, w, x = _check(orc, 4, 64, 2, 256, 2048, 45)
    y_r = api.run(w, x.cuda(), workspace=api.Workspace())
    torch.cuda.synchronize()
    d = (y.float() - y_r.float()).abs()
    assert bool(d.max() > 0)
    assert float(d.max()) <= 0.05 * float(y_r.float().abs().max())


def test_exact_refuses_prompt_rows():
    w = api.pack(torch.zeros(64, 128, dtype=torch.uint8, device="cuda"),
                 torch.zeros(64, 2, dtype=torch.bfloat16, device="cuda"),
                 torch.zeros(64, 2, dtype=torch.bfloat16, device="cuda"), 4, 64)
    with pytest.raises(api.AffqmmError) as ei:
        api.run_exact(w, torch.zeros(17, 128, dtype=torch.bfloat16, device="cuda"))
    assert ei.value.name == "AFFQMM_E_M"
