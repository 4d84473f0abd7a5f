"""Scaled embedding rows on the GPU (affqmm_embed_rows, and
affqmm_embed_rows_copy from the row-contiguous copy affqmm_pack_rows makes,
through the C ABI) against the CPU oracle: out[t, k] = bf16(bf16(s*q + b) *
scale), bit for bit, for every width and group, several scales (Gemma's
bf16(sqrt(hidden)), powers of two, negative, tiny), repeated and boundary
ids, and ids outside the table (zero rows and a status bit)."""
import math

import numpy as np
import pytest
import torch

from group_affine_bit_gb300 import api, build, synth
from helpers import u16

pytestmark = pytest.mark.gpu

ALL_WIDTHS = [(b, g) for b in (2, 3, 4, 5, 6, 8) for g in (32, 64, 128)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return api.lib()


def bf16_bits(v: float) -> int:
    return int(torch.tensor([v], dtype=torch.bfloat16).view(torch.int16).item()) & 0xFFFF


def table(bits, group, N, K, seed):
    g = synth.generator(seed)
    codes, s, b = synth.affine_table(bits, group, N, K, g)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    return w, codes, s, b


def ids_for(N, T, seed):
    g = torch.Generator().manual_seed(seed)
    ids = torch.randint(0, N, (T,), generator=g, dtype=torch.int32)
    ids[0], ids[-1] = 0, N - 1
    if T > 4:
        ids[1] = ids[2] = min(127, N - 1)   # a repeat, and the last row of the first tile
        ids[3] = min(128, N - 1)
    return ids


def gather(w, ids, scale, via, status=None):
    """The gather through one of the two entry points."""
    if via == "copy":
        return api.embed_rows_copy(w, api.pack_rows(w), ids, scale, status=status)
    return api.embed_rows(w, ids, scale, status=status)


@pytest.mark.parametrize("via", ["blocks", "copy"])
@pytest.mark.parametrize("bits,group", ALL_WIDTHS)
def test_embed_rows_bit_exact_all_widths(orc, bits, group, via):
    N, K, T = 300, 384 + (group if group < 128 else 0), 37
    K -= K % group
    w, codes, s, b = table(bits, group, N, K, seed=bits * 10 + group)
    ids = ids_for(N, T, seed=group)
    for scale in (None, math.sqrt(5376.0)):
        got = u16(gather(w, ids.cuda(), scale, via))
        want = orc.embed_rows(bits, group, codes.numpy(), u16(s), u16(b), ids.numpy(),
                              None if scale is None else bf16_bits(scale))
        diff = np.argwhere(got != want)
        assert diff.size == 0, f"{len(diff)} values differ, first at {diff[0]} (scale {scale})"


@pytest.mark.parametrize("scale", [1.0, 8.0, -5.0, 0.1, 3.0e-38, 1.0e30])
def test_embed_rows_scales(orc, scale):
    bits, group, N, K, T = 4, 64, 512, 1024, 64
    w, codes, s, b = table(bits, group, N, K, seed=91)
    ids = ids_for(N, T, seed=5)
    got = u16(api.embed_rows(w, ids.cuda(), scale))
    want = orc.embed_rows(bits, group, codes.numpy(), u16(s), u16(b), ids.numpy(), bf16_bits(scale))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("via", ["blocks", "copy"])
def test_embed_rows_head_shape_sampled(orc, via):
    """The tied head's table (262144 x 5376, 4-bit g64) gathered as a prompt's embedding."""
    bits, group, N, K, T = 4, 64, 262144, 5376, 256
    w, codes, s, b = table(bits, group, N, K, seed=7)
    ids = ids_for(N, T, seed=8)
    got = u16(gather(w, ids.cuda(), math.sqrt(5376.0), via))
    sel = np.unique(ids.numpy())
    sub = {int(n): i for i, n in enumerate(sel)}
    want_rows = orc.embed_rows(bits, group, codes.numpy()[sel], u16(s)[sel], u16(b)[sel],
                               np.arange(len(sel), dtype=np.int32), bf16_bits(math.sqrt(5376.0)))
    want = want_rows[[sub[int(n)] for n in ids.numpy()]]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("via", ["blocks", "copy"])
def test_embed_rows_bad_ids_and_empty(via):
    bits, group, N, K = 4, 64, 100, 256
    w, _, _, _ = table(bits, group, N, K, seed=3)
    ids = torch.tensor([5, -1, 100, 7], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gather(w, ids, 2.0, via, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 2
    assert int(out[1].view(torch.int16).abs().sum()) == 0 and int(out[2].view(torch.int16).abs().sum()) == 0
    ref = api.embed_rows(w, torch.tensor([5, 7], dtype=torch.int32, device="cuda"), 2.0)
    assert torch.equal(out[0].view(torch.int16), ref[0].view(torch.int16))
    assert torch.equal(out[3].view(torch.int16), ref[1].view(torch.int16))
    empty = api.embed_rows(w, torch.zeros(0, dtype=torch.int32, device="cuda"), 2.0)
    assert empty.shape == (0, K)


@pytest.mark.parametrize("bits,group,K", [(4, 64, 5376), (3, 32, 96), (8, 128, 640), (5, 32, 4000 - 4000 % 32)])
def test_row_copy_is_row_contiguous(bits, group, K):
    """Each row of the copy is one contiguous range that depends on that row
    alone: the copy of a table made of some rows of another, in another
    order, holds the same bytes for each row; its size is N x the stated
    stride; the stride's padding is zero."""
    N = 333
    g = synth.generator(40 + bits)
    codes, s, b = synth.affine_table(bits, group, N, K, g)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(bits))[:150]
    wa = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    wb = api.pack(codes[perm].contiguous().cuda(), s[perm].contiguous().cuda(), b[perm].contiguous().cuda(),
                  bits, group)
    kb = -(-K // 128)
    stride = -(-(kb * (16 * bits + 512 // group)) // 16) * 16
    assert api.rows_bytes(bits, group, N, K) == N * stride
    ra = api.pack_rows(wa).cpu().numpy()[:N * stride].reshape(N, stride)
    rb = api.pack_rows(wb).cpu().numpy()[:150 * stride].reshape(150, stride)
    assert np.array_equal(rb, ra[perm.numpy()])
    used = kb * (16 * bits + 512 // group)
    assert not ra[:, used:].any()
