"""affqmm_run_noalloc, the entry point for callers that cannot allocate device
memory (a plug-in inside an engine that owns all of the GPU's memory, or a
loop that must not call cudaMalloc/cudaFree once running), against
affqmm_run, which works in a workspace the caller provides.

Both are called through the C ABI on the same inputs.  The no-alloc call is
made twice in a row on different projections -- the second finds the
scratch array as the first left it -- and each output must lie within the
output tolerance of the parity tests (and, as the two calls run the same
kernel on the same split of the work, match affqmm_run bit for bit).

This file is named to be collected last, so that a run stopping at its
first failure has run every other test before this one.
"""
import numpy as np
import pytest
import torch

from group_affine_bit_gb300 import api, build, synth
from helpers import assert_within_tolerance, bf16_to_f64, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return api.lib()


def _problem(bits, group, M, N, K, seed):
    x, codes, s, b = synth.problem(bits, group, M, N, K, seed)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    return w, x.cuda()


# (bits, group, M, N, K, seed): whole row tiles per CTA with M = 1; a long
# depth split across CTAs (partial sums and merge counters in the scratch)
# with M = 16 and a ragged last tile
CASES = [(4, 64, 1, 30720, 3840, 21), (4, 64, 16, 200, 21504, 22)]


def test_noalloc_matches_run_on_two_calls_in_a_row():
    probs = [_problem(*c) for c in CASES]
    # the existing entry point, each with its own workspace
    refs = [api.run(w, x, workspace=api.Workspace()) for w, x in probs]
    torch.cuda.synchronize()
    # the no-alloc entry point, twice in a row on one stream
    outs = [torch.empty_like(r) for r in refs]
    for (w, x), y in zip(probs, outs):
        api.run_noalloc(w, x, y)
    torch.cuda.synchronize()
    for c, y, r in zip(CASES, outs, refs):
        what = f"noalloc {c[0]}b g{c[1]} M={c[2]} N={c[3]} K={c[4]}"
        assert_within_tolerance(y, bf16_to_f64(u16(r)), what)
        assert torch.equal(y.view(torch.int16), r.view(torch.int16)), f"{what}: differs from affqmm_run"


def test_noalloc_against_the_oracle(orc):
    """The same two cases, each output against the CPU oracle's projection."""
    for bits, group, M, N, K, seed in CASES:
        x, codes, s, b = synth.problem(bits, group, M, N, K, seed)
        w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        api.run_noalloc(w, x.cuda(), y)
        torch.cuda.synchronize()
        y_ref = orc.qmm(bits, group, u16(x), codes.numpy(), u16(s), u16(b), nthreads=16)
        assert_within_tolerance(y, y_ref, f"noalloc {bits}b g{group} M={M} N={N} K={K} against the oracle")


def test_noalloc_refuses_beyond_its_scratch():
    w, x = _problem(4, 64, 17, 256, 256, 23)
    y = torch.empty(17, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.AffqmmError) as ei:
        api.run_noalloc(w, x, y)
    assert ei.value.name == "AFFQMM_E_SCRATCH"
