"""The decode projection's fused forms against the oracle, through the C ABI.

* affqmm_run_exact_sums: the exact-codes form with the group sums of x written
  by the kernel that produced x; checked against oracle_qmm_groupsum_given on
  the very sums passed in (and on sums moved away from the true ones, which
  the kernel must use as given).
* affqmm_run_geglu: a gate/up stack whose rows are interleaved in 16-row
  blocks, with GeGLU (mlx_lm's gelu_approx(gate) * up as bf16 operations) as
  the projection's epilogue.  Its output must have the bits of the unfused
  projection followed by the oracle's GeGLU on that projection's own bf16
  outputs (fusing changes no bit), up to the one bf16 step an fp32 tanh
  within a few ulps may move (the oracle returns both candidates), for the
  rounded, exact-codes and producer-sums forms.
"""
import numpy as np
import pytest
import torch

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


def group_sums_fp32(x: torch.Tensor, group: int) -> torch.Tensor:
    """What a producer of x writes: each group's sum of the bf16 values, in
    float64 then rounded once to fp32."""
    M, K = x.shape
    return x.double().reshape(M, K // group, group).sum(dim=2).float().contiguous()


@pytest.mark.parametrize("bits,group", ALL_WIDTHS)
def test_exact_sums_all_widths(orc, bits, group):
    M, N, K = 3, 200, 512 + (group if group < 128 else 0)
    x, codes, s, b = synth.problem(bits, group, M, N, K, seed=600 + bits + group)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    xs = group_sums_fp32(x, group)
    y = api.run_exact_sums(w, x.cuda(), xs.cuda(), workspace=api.Workspace())
    y_ref = orc.qmm_groupsum_given(bits, group, u16(x), xs.numpy(), codes.numpy(), u16(s), u16(b))
    assert_within_tolerance(y, y_ref, f"exact sums {bits}b g{group}")


@pytest.mark.parametrize("M", [1, 8, 9, 16])
def test_exact_sums_are_used_as_given(orc, M):
    """Sums moved away from the true ones: the output follows the sums given
    (the oracle on the same sums), not the sums of x."""
    bits, group, N, K = 4, 64, 384, 21504 // 4
    x, codes, s, b = synth.problem(bits, group, M, N, K, seed=700 + M)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    xs = group_sums_fp32(x, group) + torch.linspace(-3, 3, K // group).float()
    y = api.run_exact_sums(w, x.cuda(), xs.contiguous().cuda(), workspace=api.Workspace())
    y2 = api.run_exact_sums(w, x.cuda(), xs.contiguous().cuda(), workspace=api.Workspace())
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    y_ref = orc.qmm_groupsum_given(bits, group, u16(x), xs.numpy(), codes.numpy(), u16(s), u16(b))
    assert_within_tolerance(y, y_ref, f"moved sums M={M}")
    y_true, _ = orc.qmm_groupsum(bits, group, u16(x), codes.numpy(), u16(s), u16(b))
    from helpers import tolerance_report
    ok, _, _ = tolerance_report(u16(y), y_true)
    assert not ok, "the kernel ignored the sums it was given"


def interleave(gate_t, up_t):
    """Rows of a gate/up stack interleaved in 16-row blocks: block 2j = gate
    rows 16j.., block 2j + 1 = up rows 16j.. (any [F, ...] tensors)."""
    F = gate_t.shape[0]
    rest = gate_t.shape[1:]
    return torch.stack([gate_t.reshape(F // 16, 16, *rest), up_t.reshape(F // 16, 16, *rest)], dim=1).reshape(2 * F, *rest)


def deinterleave_cols(y):
    """[M, 2F] outputs of an interleaved stack -> (gate [M, F], up [M, F])."""
    M, N = y.shape
    v = y.reshape(M, N // 32, 2, 16)
    return v[:, :, 0, :].reshape(M, N // 2), v[:, :, 1, :].reshape(M, N // 2)


def geglu_case(orc, bits, group, M, F, K, seed, form):
    g = synth.generator(seed)
    cg, sg, bg = synth.affine_table(bits, group, F, K, g)
    cu, su, bu = synth.affine_table(bits, group, F, K, g)
    x = synth.activations(M, K, g)
    codes, s, b = interleave(cg, cu), interleave(sg, su), interleave(bg, bu)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    xd = x.cuda()
    xs = group_sums_fp32(x, group).cuda()
    ws = api.Workspace()
    h = api.run_geglu(w, xd, form=form, xsums=xs, workspace=ws)
    if form == api.FORM_ROUNDED:
        y = api.run(w, xd, workspace=ws)
    elif form == api.FORM_EXACT:
        y = api.run_exact(w, xd, workspace=ws)
    else:
        y = api.run_exact_sums(w, xd, xs, workspace=ws)
    torch.cuda.synchronize()
    assert api.workspace_status(ws.buf) == 0
    gate, up = deinterleave_cols(y.cpu())
    lo, hi = orc.geglu(u16(gate), u16(up))
    hb = u16(h)
    ok = (hb == lo) | (hb == hi)
    what = f"geglu form {form} {bits}b g{group} M={M} F={F} K={K}"
    assert ok.all(), f"{what}: {int((~ok).sum())} outputs differ from the unfused projection + GeGLU"
    return w, x, codes, s, b, y, h


@pytest.mark.parametrize("form", [0, 1, 2])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_geglu_same_bits_as_apart(orc, form, M):
    geglu_case(orc, 4, 64, M, 1024, 1536, seed=800 + 10 * form + M, form=form)


@pytest.mark.parametrize("bits,group", [(2, 128), (3, 32), (5, 64), (6, 32), (8, 128)])
def test_geglu_other_widths(orc, bits, group):
    geglu_case(orc, bits, group, 3, 512, 640, seed=900 + bits + group, form=0)


@pytest.mark.parametrize("M", [1, 16])
def test_geglu_decode_step_gate_up_full(orc, M):
    """The decode step's gate/up stack (43008 x 5376: 21504 hidden units) at
    full size; the unfused projection it equals is also checked against the
    oracle on every output."""
    F, K = 21504, 5376
    w, x, codes, s, b, y, h = geglu_case(orc, 4, 64, M, F, K, seed=1000 + M, form=0)
    y_ref = orc.qmm(4, 64, u16(x), codes.numpy(), u16(s), u16(b), nthreads=16)
    assert_within_tolerance(y, y_ref, f"gate/up stack M={M}")


def test_geglu_refusals():
    w = api.pack(torch.zeros(48, 128, dtype=torch.uint8, device="cuda"),
                 torch.zeros(48, 2, dtype=torch.bfloat16, device="cuda"),
                 torch.zeros(48, 2, dtype=torch.bfloat16, device="cuda"), 4, 64)
    x = torch.zeros(1, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.AffqmmError) as ei:
        api.run_geglu(w, x)
    assert ei.value.name == "AFFQMM_E_SHAPE"     # 48 rows: not whole 32-row gate/up blocks
    w2 = api.pack(torch.zeros(64, 128, dtype=torch.uint8, device="cuda"),
                  torch.zeros(64, 2, dtype=torch.bfloat16, device="cuda"),
                  torch.zeros(64, 2, dtype=torch.bfloat16, device="cuda"), 4, 64)
    with pytest.raises(api.AffqmmError) as ei:
        api.run_geglu(w2, torch.zeros(17, 128, dtype=torch.bfloat16, device="cuda"))
    assert ei.value.name == "AFFQMM_E_M"
    with pytest.raises(api.AffqmmError) as ei:
        api.run_geglu(w2, x, form=7)
    assert ei.value.name == "AFFQMM_E_ARG"
