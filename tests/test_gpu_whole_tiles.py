"""The decode kernel's whole-tile store, against the CPU oracle on full rows.

A decode launch cuts a projection's (128-row tile, 128-deep block) units into
one contiguous run per resident CTA.  A tile that one run covers from its
first block to its last is stored as bf16 straight from the run's fp32
registers; a tile that several runs share goes through fp32 partials merged
in run order.  The first branch needs more units per run than blocks per
tile -- many rows over a short depth, or very many rows (the decode step's
gate/up stack, 43008 x 5376, and its tied head, 262144 x 5376).  Every case
here first checks, with the host's own replay of the split, that it really
takes that branch, then compares every output with the oracle (rounded
weights: oracle_qmm; exact codes: oracle_qmm_groupsum) within
|y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref row), the rms over the whole row.
"""
import os

import numpy as np
import pytest
import torch

from group_affine_bit_gb300 import api, build, synth
from helpers import assert_within_tolerance, decode_tile_split, u16

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, len(os.sched_getaffinity(0))))


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return api.lib()


def sms() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def _case(orc, bits, group, M, N, K, seed, exact=False, need_split=False):
    whole, split = decode_tile_split(N, K, sms())
    assert whole > 0, f"N={N} K={K}: no tile is covered by a single run"
    if need_split:
        assert split > 0, f"N={N} K={K}: no tile is shared by runs"
    x, codes, s, b = synth.problem(bits, group, M, N, K, seed)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    ws = api.Workspace()
    run = api.run_exact if exact else api.run
    y = run(w, x.cuda(), workspace=ws)
    y2 = run(w, x.cuda(), workspace=ws)
    torch.cuda.synchronize()
    what = f"{'exact ' if exact else ''}{bits}b g{group} M={M} N={N} K={K} ({whole} whole tiles, {split} shared)"
    assert api.workspace_status(ws.buf) == 0, what
    assert int(ws.buf[:api.WORKSPACE_ZEROED].count_nonzero()) == 0, f"{what}: counters not left zeroed"
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), f"{what}: not deterministic"
    del w
    if exact:
        y_ref, _ = orc.qmm_groupsum(bits, group, u16(x), codes.numpy(), u16(s), u16(b), nthreads=THREADS)
    else:
        y_ref = orc.qmm(bits, group, u16(x), codes.numpy(), u16(s), u16(b), nthreads=THREADS)
    assert_within_tolerance(y, y_ref, what)


# Short depths: every run holds whole tiles (77824 x 256), or whole tiles
# between shared ones (89600 x 640, 40000 x 384).
SMALL = [(77824, 256), (89600, 640), (40000, 384)]


@pytest.mark.parametrize("N,K", SMALL)
@pytest.mark.parametrize("M", [1, 6, 16])
def test_whole_tiles_short_depth(orc, N, K, M):
    _case(orc, 4, 64, M, N, K, seed=N + K + M)


@pytest.mark.parametrize("bits,group", [(8, 32), (3, 64), (2, 128), (5, 32), (6, 128)])
def test_whole_tiles_other_widths(orc, bits, group):
    _case(orc, bits, group, 16, 89600, 640, seed=bits * 10 + group, need_split=True)


@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("N,K", [(77824, 256), (89600, 640)])
def test_whole_tiles_exact_codes(orc, N, K, M):
    _case(orc, 4, 64, M, N, K, seed=N + K + M + 1, exact=True)


# The decode step's shapes at full size (a layer's gate/up stack and the tied
# head), every output row against the oracle.
GATE_UP = synth.DECODER_LAYER_SHAPES["gate_up"]
HEAD = synth.HEAD_SHAPE


@pytest.mark.parametrize("M", [1, 16])
def test_decode_step_gate_up_full(orc, M):
    N, K = GATE_UP
    _case(orc, 4, 64, M, N, K, seed=synth.step_seed(synth.DECODE_STEP_SEED, 0, 2) + M, need_split=True)


@pytest.mark.parametrize("M", [1, 16])
def test_decode_step_gate_up_full_exact(orc, M):
    N, K = GATE_UP
    _case(orc, 4, 64, M, N, K, seed=synth.step_seed(synth.DECODE_STEP_SEED, 0, 2) + 100 + M, exact=True,
          need_split=True)


@pytest.mark.parametrize("M", [1, 16])
def test_decode_step_head_full(orc, M):
    N, K = HEAD
    _case(orc, 4, 64, M, N, K, seed=synth.step_seed(synth.DECODE_STEP_SEED, synth.N_LAYERS, 0) + M,
          need_split=True)


def test_decode_step_head_full_exact(orc):
    N, K = HEAD
    _case(orc, 4, 64, 1, N, K, seed=synth.step_seed(synth.DECODE_STEP_SEED, synth.N_LAYERS, 0) + 100, exact=True,
          need_split=True)
