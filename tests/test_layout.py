"""The packed block layout (group_affine_bit_gb300/csrc/affqmm_format.cuh),
checked on the host from the header's own offset functions (compiled with
nvcc into a small dump program): every code and scale/bias byte of a block has
exactly one place, and both ways the kernels read the codes from shared
memory touch each bank once per access phase -- one thread per row reading a
16-byte chunk (prompt and embedding kernels, dequant hook), and the matrix-
fragment threads of the decode kernel reading their class's words of rows g
and g + 8."""
import os
import shutil
import subprocess
from collections import defaultdict

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "group_affine_bit_gb300", "csrc")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


@pytest.fixture(scope="module")
def layout(tmp_path_factory):
    if not (os.path.exists(NVCC) or shutil.which("nvcc")):
        pytest.skip("nvcc not found")
    exe = str(tmp_path_factory.mktemp("layout") / "layout_dump")
    nvcc = NVCC if os.path.exists(NVCC) else shutil.which("nvcc")
    subprocess.run([nvcc, "-std=c++17", "-I", CSRC, os.path.join(ROOT, "tests", "layout_dump.cu"), "-o", exe],
                   check=True, capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    words = defaultdict(dict)   # (bits, plane) -> {(row, word): offset}
    sbw = defaultdict(dict)     # (bits, group) -> {(row, j): offset}
    blk = {}
    for line in out.splitlines():
        f = line.split()
        if f[0] == "w":
            bits, plane, n, w, off = map(int, f[1:])
            words[(bits, plane)][(n, w)] = off
        else:
            bits, group, n, j, off, bb = map(int, f[1:])
            sbw[(bits, group)][(n, j)] = off
            blk[(bits, group)] = bb
    return words, sbw, blk


def plane_bits(bits):
    p0 = 2 if bits <= 3 else 4
    return p0, bits - p0


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_every_code_byte_has_one_place(layout, bits):
    words, _, _ = layout
    seen = []
    for plane, p in enumerate(plane_bits(bits)):
        for (n, w), off in words.get((bits, plane), {}).items():
            assert off % 4 == 0
            seen.extend(range(off, off + 4))
    assert sorted(seen) == list(range(2048 * bits))


@pytest.mark.parametrize("bits,group", [(b, g) for b in (2, 3, 4, 5, 6, 8) for g in (32, 64, 128)])
def test_scale_bias_words_follow_the_codes(layout, bits, group):
    _, sbw, blk = layout
    offs = sorted(o for o in sbw[(bits, group)].values())
    assert offs == list(range(2048 * bits, blk[(bits, group)], 4))


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_row_per_thread_chunk_reads_are_conflict_free(layout, bits):
    """8 consecutive rows (a quarter warp of 16-byte loads) reading the same
    chunk land on 8 distinct 16-byte bank groups."""
    words, _, _ = layout
    for plane, p in enumerate(plane_bits(bits)):
        if p == 0:
            continue
        m = words[(bits, plane)]
        for c in range(p):
            for r0 in range(0, 128, 8):
                starts = [m[(r0 + i, 4 * c)] for i in range(8)]
                assert all(s % 16 == 0 for s in starts)
                assert len({(s // 16) % 8 for s in starts}) == 8, (bits, plane, c, r0)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_fragment_class_reads_are_conflict_free(layout, bits):
    """Lane 4g + c of a decode warp reads the p words p*c .. p*c + p - 1 of
    row r0 + g (one 16-, 8- or 4-byte load).  Each access phase -- 8 lanes for
    16-byte loads, 16 for 8-byte, 32 for 4-byte -- covers distinct banks, and
    a lane's words are contiguous and aligned."""
    words, _, _ = layout
    for plane, p in enumerate(plane_bits(bits)):
        if p == 0:
            continue
        m = words[(bits, plane)]
        nbytes = 4 * p
        phase = 128 // nbytes  # lanes per shared-memory access phase
        for r0 in range(0, 128, 8):
            lanes = []
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                offs = [m[(r0 + g, p * c + v)] for v in range(p)]
                assert offs == list(range(offs[0], offs[0] + nbytes, 4)) and offs[0] % nbytes == 0
                lanes.append(offs[0])
            for ph in range(0, 32, phase):
                banks = set()
                for start in lanes[ph:ph + phase]:
                    for b in range(start // 4, start // 4 + nbytes // 4):
                        assert b % 32 not in banks, (bits, plane, r0, ph)
                        banks.add(b % 32)
