"""The C ABI without a GPU: the library loads, exports every declared entry
point, and refuses bad arguments by name before touching a device."""
import ctypes
import os
import re

import pytest

from group_affine_bit_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "affqmm.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return api.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"AFFQMM_API\s+[\w\s\*]+?\b(affqmm_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for want in ["affqmm_pack", "affqmm_run", "affqmm_run_stacked", "affqmm_dequant",
                 "affqmm_packed_bytes", "affqmm_workspace_bytes", "affqmm_strerror",
                 "affqmm_embed_rows", "affqmm_rows_bytes", "affqmm_pack_rows", "affqmm_embed_rows_copy"]:
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in affqmm.h but not exported"


def test_strerror_names_every_status(L):
    seen = set()
    for code in range(13):
        s = api.strerror(code)
        assert s and s not in seen
        seen.add(s)
    assert "unknown" in api.strerror(999)


def test_version(L):
    assert L.affqmm_version() >= 100


@pytest.mark.parametrize("bits,group", [(b, g) for b in (2, 3, 4, 5, 6, 8) for g in (32, 64, 128)])
def test_packed_bytes_closed_form(bits, group):
    for N, K in [(512, 256), (30720, 3840), (17, 96 if group == 32 else 2 * group), (1, group), (0, 0)]:
        if K % group:
            continue
        tiles = -(-N // 128)          # 128-row tiles
        kb = -(-K // 128)             # 128-deep blocks
        want = tiles * kb * (128 * 128 * bits // 8 + 128 * 4 * (128 // group))
        assert api.packed_bytes(bits, group, N, K) == want


@pytest.mark.parametrize("bits,group", [(b, g) for b in (2, 3, 4, 5, 6, 8) for g in (32, 64, 128)])
def test_rows_bytes_closed_form(bits, group):
    """The row-contiguous copy: N rows of ceil(K/128) blocks x (16*bits code
    bytes + 512/group scale/bias bytes), the row padded to 16 bytes."""
    for N, K in [(512, 256), (262144, 5376), (17, 96 if group == 32 else 2 * group), (1, group), (0, 0)]:
        if K % group:
            continue
        kb = -(-K // 128)
        stride = -(-(kb * (16 * bits + 512 // group)) // 16) * 16
        assert api.rows_bytes(bits, group, N, K) == N * stride
    with pytest.raises(api.AffqmmError):
        api.rows_bytes(bits, group, 16, group + 16)


@pytest.mark.parametrize("bits,group,N,K,status", [
    (7, 64, 16, 128, "AFFQMM_E_BITS"), (1, 64, 16, 128, "AFFQMM_E_BITS"), (4, 16, 16, 128, "AFFQMM_E_GROUP"),
    (4, 256, 16, 256, "AFFQMM_E_GROUP"), (4, 64, 16, 96, "AFFQMM_E_SHAPE"), (4, 64, -1, 128, "AFFQMM_E_SHAPE"),
    (4, 64, 16, -64, "AFFQMM_E_SHAPE")])
def test_packed_bytes_refusals(bits, group, N, K, status):
    with pytest.raises(api.AffqmmError) as ei:
        api.packed_bytes(bits, group, N, K)
    assert ei.value.name == status


def _w(bits=4, group=64, N=32, K=256, packed=0x100000):
    return api.CWeight(bits, group, N, K, packed)


def _run(L, w, x=0x200000, M=1, y=0x300000, ws=None, nbytes=0):
    return L.affqmm_run(ctypes.byref(w) if w is not None else None, x, M, y, ws, nbytes, None)


def test_run_refusals_before_any_launch(L):
    names = api.STATUS_NAMES
    assert names[_run(L, None)] == "AFFQMM_E_NULL"
    assert names[_run(L, _w(bits=7))] == "AFFQMM_E_BITS"
    assert names[_run(L, _w(group=48))] == "AFFQMM_E_GROUP"
    assert names[_run(L, _w(K=100))] == "AFFQMM_E_SHAPE"
    assert names[_run(L, _w(packed=0))] == "AFFQMM_E_NULL"
    assert names[_run(L, _w(packed=0x100010))] == "AFFQMM_E_ALIGN"
    assert names[_run(L, _w(), M=-1)] == "AFFQMM_E_M"
    assert names[_run(L, _w(), M=(1 << 20) + 1)] == "AFFQMM_E_M"
    assert names[_run(L, _w(), x=0)] == "AFFQMM_E_NULL"
    assert names[_run(L, _w(), y=0)] == "AFFQMM_E_NULL"
    assert names[_run(L, _w(), x=0x200008)] == "AFFQMM_E_ALIGN"
    assert names[_run(L, _w(), y=0x300001)] == "AFFQMM_E_ALIGN"
    # M = 0 is a valid empty call: nothing to do, nothing launched.
    assert _run(L, _w(), M=0) == 0


def test_run_host_refusals_before_anything_is_enqueued(L):
    names = api.STATUS_NAMES
    w = _w()

    def run_host(wp, x=0x10000, M=1, y=0x20000, x_dev=0x200000, y_dev=0x300000):
        return L.affqmm_run_host(wp, x, M, y, x_dev, y_dev, None, 0, None)

    assert names[run_host(None)] == "AFFQMM_E_NULL"
    assert names[run_host(ctypes.byref(_w(bits=7)))] == "AFFQMM_E_BITS"
    assert names[run_host(ctypes.byref(w), M=-1)] == "AFFQMM_E_M"
    assert names[run_host(ctypes.byref(w), x=0)] == "AFFQMM_E_NULL"
    assert names[run_host(ctypes.byref(w), y=0)] == "AFFQMM_E_NULL"
    assert names[run_host(ctypes.byref(w), x_dev=0)] == "AFFQMM_E_NULL"
    assert names[run_host(ctypes.byref(w), y_dev=0)] == "AFFQMM_E_NULL"
    assert names[run_host(ctypes.byref(w), x_dev=0x200008)] == "AFFQMM_E_ALIGN"
    assert names[run_host(ctypes.byref(w), y_dev=0x300001)] == "AFFQMM_E_ALIGN"
    assert run_host(ctypes.byref(w), M=0) == 0


def test_run_exact_refusals_before_any_launch(L):
    names = api.STATUS_NAMES
    w = _w()
    run = lambda wp, M=1, x=0x200000, y=0x300000: L.affqmm_run_exact(wp, x, M, y, None, 0, None)
    assert names[run(None)] == "AFFQMM_E_NULL"
    assert names[run(ctypes.byref(_w(group=48)))] == "AFFQMM_E_GROUP"
    assert names[run(ctypes.byref(w), M=17)] == "AFFQMM_E_M"   # the exact-codes form is the decode path only
    assert names[run(ctypes.byref(w), M=-1)] == "AFFQMM_E_M"
    assert names[run(ctypes.byref(w), x=0)] == "AFFQMM_E_NULL"
    assert names[run(ctypes.byref(w), y=0x300001)] == "AFFQMM_E_ALIGN"
    assert run(ctypes.byref(w), M=0) == 0


def test_stacked_refusals(L):
    names = api.STATUS_NAMES
    arr = (api.CWeight * 2)(_w(), _w(K=512))
    ys = (ctypes.c_void_p * 2)(0x300000, 0x400000)
    rc = L.affqmm_run_stacked(2, arr, 0x200000, 1, ys, None, 0, None)
    assert names[rc] == "AFFQMM_E_ARG"         # mismatched K
    arr = (api.CWeight * 2)(_w(), _w(bits=8))
    assert names[L.affqmm_run_stacked(2, arr, 0x200000, 1, ys, None, 0, None)] == "AFFQMM_E_ARG"
    assert names[L.affqmm_run_stacked(0, arr, 0x200000, 1, ys, None, 0, None)] == "AFFQMM_E_ARG"
    assert names[L.affqmm_run_stacked(9, arr, 0x200000, 1, ys, None, 0, None)] == "AFFQMM_E_ARG"
    assert names[L.affqmm_run_stacked(1, arr, 0x200000, 1, None, None, 0, None)] == "AFFQMM_E_NULL"


def test_pack_and_dequant_refusals(L):
    names = api.STATUS_NAMES
    assert names[L.affqmm_pack(4, 64, 16, 128, 1, 2, 3, None, None)] == "AFFQMM_E_NULL"
    assert names[L.affqmm_pack(4, 64, 16, 128, 0, 2, 3, 0x100000, None)] == "AFFQMM_E_NULL"
    assert names[L.affqmm_pack(4, 64, 16, 128, 1, 2, 3, 0x100040, None)] == "AFFQMM_E_ALIGN"
    assert names[L.affqmm_pack(9, 64, 16, 128, 1, 2, 3, 0x100000, None)] == "AFFQMM_E_BITS"
    # an empty table packs to zero bytes: nothing to do
    assert L.affqmm_pack(4, 64, 0, 128, 0, 0, 0, None, None) == 0
    w = _w()
    assert names[L.affqmm_dequant(ctypes.byref(w), None, None)] == "AFFQMM_E_NULL"
    assert names[L.affqmm_dequant(ctypes.byref(w), 0x300001, None)] == "AFFQMM_E_ALIGN"
    assert names[L.affqmm_workspace_status(None, None)] == "AFFQMM_E_NULL"


def test_embed_rows_refusals_before_any_launch(L):
    w = _w()
    rc = L.affqmm_embed_rows(ctypes.byref(w), 0x200000, -1, 1, 0x4000, 0x300000, None, None)
    assert api.STATUS_NAMES[rc] == "AFFQMM_E_ARG"
    bad = _w(bits=7)
    rc = L.affqmm_embed_rows(ctypes.byref(bad), 0x200000, 4, 1, 0x4000, 0x300000, None, None)
    assert api.STATUS_NAMES[rc] == "AFFQMM_E_BITS"
    rc = L.affqmm_embed_rows(ctypes.byref(w), None, 4, 1, 0x4000, 0x300000, None, None)
    assert api.STATUS_NAMES[rc] == "AFFQMM_E_NULL"
    rc = L.affqmm_embed_rows(ctypes.byref(w), 0x200000, 4, 1, 0x4000, 0x300008, None, None)
    assert api.STATUS_NAMES[rc] == "AFFQMM_E_ALIGN"


def test_row_copy_refusals_before_any_launch(L):
    names = api.STATUS_NAMES
    w = _w()
    assert names[L.affqmm_pack_rows(ctypes.byref(w), None, None)] == "AFFQMM_E_NULL"
    assert names[L.affqmm_pack_rows(ctypes.byref(w), 0x400010, None)] == "AFFQMM_E_ALIGN"
    assert names[L.affqmm_pack_rows(ctypes.byref(_w(bits=7)), 0x400000, None)] == "AFFQMM_E_BITS"
    assert L.affqmm_pack_rows(ctypes.byref(_w(N=0)), None, None) == 0     # nothing to copy
    copy = lambda rows, ids=0x200000, out=0x300000, T=4: L.affqmm_embed_rows_copy(
        ctypes.byref(w), rows, ids, T, 1, 0x4000, out, None, None)
    assert names[copy(None)] == "AFFQMM_E_NULL"
    assert names[copy(0x400010)] == "AFFQMM_E_ALIGN"
    assert names[copy(0x400000, T=-1)] == "AFFQMM_E_ARG"
    assert names[copy(0x400000, out=0x300008)] == "AFFQMM_E_ALIGN"
    assert copy(None, T=0) == 0


def test_fault_wait_hook_refusal_and_reset(L):
    assert api.STATUS_NAMES[L.affqmm_test_fault_wait(-5)] == "AFFQMM_E_ARG"
    assert L.affqmm_test_fault_wait(0) == 0
