"""Python binding of libaffqmm (include/affqmm.h): argument marshalling only.

Every step of the projection runs in the library's CUDA kernels; this module
turns torch tensors into pointers, sizes and the current CUDA stream, and
turns status codes into exceptions.  PyTorch supplies device memory and
streams.  There is no fallback: if libaffqmm.so is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("AFFQMM_LIB_PATH") or os.path.join(_PKG, "libaffqmm.so")   # the in-tree build unless overridden

MAX_STACK = 8
MAX_M = 1 << 20
NOALLOC_MAX_M = 16                   # rows affqmm_run_noalloc takes
WORKSPACE_ZEROED = 256 + 65536 * 4   # leading workspace bytes kept zero between calls

STATUS_NAMES = {
    0: "AFFQMM_OK", 1: "AFFQMM_E_NULL", 2: "AFFQMM_E_BITS", 3: "AFFQMM_E_GROUP",
    4: "AFFQMM_E_SHAPE", 5: "AFFQMM_E_ALIGN", 6: "AFFQMM_E_M", 7: "AFFQMM_E_WORKSPACE",
    8: "AFFQMM_E_TIMEOUT", 9: "AFFQMM_E_CUDA", 10: "AFFQMM_E_ARG", 11: "AFFQMM_E_DEVICE",
    12: "AFFQMM_E_SCRATCH",
}


class AffqmmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{what}: {self.name} ({strerror(status)})")


class CWeight(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group", ctypes.c_int32), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("packed", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libaffqmm.so (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libaffqmm.so is not built ({LIB_PATH}); run group_affine_bit_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, szp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)
        wp = ctypes.POINTER(CWeight)
        sig = {
            "affqmm_strerror": (ctypes.c_char_p, [i32]),
            "affqmm_version": (i32, []),
            "affqmm_packed_bytes": (i32, [i32, i32, i64, i64, szp]),
            "affqmm_pack": (i32, [i32, i32, i64, i64, vp, vp, vp, vp, vp]),
            "affqmm_workspace_bytes": (i32, [wp, i64, szp]),
            "affqmm_workspace_bytes_stacked": (i32, [i32, wp, i64, szp]),
            "affqmm_run": (i32, [wp, vp, i64, vp, vp, ctypes.c_size_t, vp]),
            "affqmm_run_stacked": (i32, [i32, wp, vp, i64, ctypes.POINTER(vp), vp, ctypes.c_size_t, vp]),
            "affqmm_dequant": (i32, [wp, vp, vp]),
            "affqmm_workspace_status": (i32, [vp, vp]),
            "affqmm_run_noalloc": (i32, [wp, vp, i64, vp, vp]),
            "affqmm_run_host": (i32, [wp, vp, i64, vp, vp, vp, vp, ctypes.c_size_t, vp]),
            "affqmm_run_exact": (i32, [wp, vp, i64, vp, vp, ctypes.c_size_t, vp]),
            "affqmm_embed_rows": (i32, [wp, vp, i64, i32, ctypes.c_uint16, vp, vp, vp]),
            "affqmm_test_fault_wait": (i32, [i64]),
            "affqmm_run_exact_sums": (i32, [wp, vp, vp, i64, vp, vp, ctypes.c_size_t, vp]),
            "affqmm_run_geglu": (i32, [wp, vp, vp, i64, i32, vp, vp, ctypes.c_size_t, vp]),
            "affqmm_rows_bytes": (i32, [i32, i32, i64, i64, szp]),
            "affqmm_pack_rows": (i32, [wp, vp, vp]),
            "affqmm_embed_rows_copy": (i32, [wp, vp, vp, i64, i32, ctypes.c_uint16, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().affqmm_strerror(int(status)).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise AffqmmError(rc, what)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)   # cheap current-stream lookup, when present


def _stream_ptr(stream, device_index: int | None = None) -> int:
    if stream is None:
        if _raw_stream is not None:
            return int(_raw_stream(torch.cuda.current_device() if device_index is None else device_index))
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


@dataclass
class PackedWeight:
    """A packed affine table (device memory owned by the torch tensor `packed`)."""
    bits: int
    group: int
    N: int
    K: int
    packed: torch.Tensor
    _c: CWeight | None = field(default=None, repr=False, compare=False)
    _ws: dict = field(default_factory=dict, repr=False, compare=False)   # (M, device) -> workspace bytes

    def cstruct(self) -> CWeight:
        """The C view of this weight (built once: the storage never moves)."""
        if self._c is None:
            self._c = CWeight(self.bits, self.group, self.N, self.K,
                              self.packed.data_ptr() if self.packed.numel() else None)
        return self._c


def packed_bytes(bits: int, group: int, N: int, K: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().affqmm_packed_bytes(bits, group, N, K, ctypes.byref(out)), "affqmm_packed_bytes")
    return out.value


def pack(codes: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor, bits: int, group: int,
         stream=None) -> PackedWeight:
    """codes uint8 [N,K]; scales, biases bf16 [N,K/group]; all on one CUDA device."""
    N, K = codes.shape
    for t in (codes, scales, biases):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("pack wants contiguous CUDA tensors")
    if codes.dtype != torch.uint8 or scales.dtype != torch.bfloat16 or biases.dtype != torch.bfloat16:
        raise ValueError("pack wants uint8 codes and bf16 scales and biases")
    nbytes = packed_bytes(bits, group, N, K)
    packed = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=codes.device)
    _check(lib().affqmm_pack(bits, group, N, K, codes.data_ptr(), scales.data_ptr(), biases.data_ptr(),
                             packed.data_ptr(), _stream_ptr(stream)), "affqmm_pack")
    return PackedWeight(bits, group, N, K, packed)


def workspace_bytes(w: PackedWeight, M: int) -> int:
    key = (M, torch.cuda.current_device())
    got = w._ws.get(key)
    if got is None:
        out = ctypes.c_size_t(0)
        cw = w.cstruct()
        _check(lib().affqmm_workspace_bytes(ctypes.byref(cw), M, ctypes.byref(out)), "affqmm_workspace_bytes")
        got = w._ws[key] = out.value
    return got


def _warray(ws):
    arr = (CWeight * len(ws))()
    for i, w in enumerate(ws):
        arr[i] = w.cstruct()
    return arr


def workspace_bytes_stacked(ws, M: int) -> int:
    out = ctypes.c_size_t(0)
    arr = _warray(ws)
    _check(lib().affqmm_workspace_bytes_stacked(len(ws), arr, M, ctypes.byref(out)),
           "affqmm_workspace_bytes_stacked")
    return out.value


class Workspace:
    """A zero-filled device buffer that grows on demand.  The library leaves it
    zeroed after every call; calls sharing one must be stream-ordered."""

    def __init__(self, device=None):
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.buf = torch.zeros(0, dtype=torch.uint8, device=self.device)

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf


_workspaces: dict = {}


def default_workspace(device, stream_ptr: int | None = None) -> Workspace:
    """One workspace per (device, stream): calls on one stream never overlap."""
    index = torch.device(device).index if not isinstance(device, int) else device
    if stream_ptr is None:
        stream_ptr = _stream_ptr(None, index)
    key = (index, stream_ptr)
    ws = _workspaces.get(key)
    if ws is None:
        ws = _workspaces[key] = Workspace(torch.device("cuda", index))
    return ws


def _check_x(x: torch.Tensor, K: int):
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != K or not x.is_contiguous():
        raise ValueError(f"x must be a contiguous CUDA bf16 [M, {K}] tensor")


def run(w: PackedWeight, x: torch.Tensor, y: torch.Tensor | None = None, workspace: Workspace | None = None,
        stream=None) -> torch.Tensor:
    """y[M, N] = bf16(x @ dequant(W)^T) with fp32 accumulation."""
    _check_x(x, w.K)
    M = x.shape[0]
    dev = x.get_device()
    if y is None:
        y = torch.empty(M, w.N, dtype=torch.bfloat16, device=x.device)
    sp = _stream_ptr(stream, dev)
    ws = workspace or default_workspace(dev, sp)
    need = workspace_bytes(w, M)
    buf = ws.get(need)
    cw = w.cstruct()
    _check(lib().affqmm_run(ctypes.byref(cw), x.data_ptr(), M, y.data_ptr(), buf.data_ptr() if need else None,
                            buf.numel(), sp), "affqmm_run")
    return y


def run_exact(w: PackedWeight, x: torch.Tensor, y: torch.Tensor | None = None, workspace: Workspace | None = None,
              stream=None) -> torch.Tensor:
    """affqmm_run_exact (M <= 16): y = bf16(sum_g s_g * sum q x + b_g * sum x), the
    exact-codes form (the weights are not rounded to bf16)."""
    _check_x(x, w.K)
    M = x.shape[0]
    dev = x.get_device()
    if y is None:
        y = torch.empty(M, w.N, dtype=torch.bfloat16, device=x.device)
    sp = _stream_ptr(stream, dev)
    ws = workspace or default_workspace(dev, sp)
    need = workspace_bytes(w, M)
    buf = ws.get(need)
    cw = w.cstruct()
    _check(lib().affqmm_run_exact(ctypes.byref(cw), x.data_ptr(), M, y.data_ptr(), buf.data_ptr() if need else None,
                                  buf.numel(), sp), "affqmm_run_exact")
    return y


FORM_ROUNDED, FORM_EXACT, FORM_EXACT_SUMS = 0, 1, 2


def _check_xsums(xsums: torch.Tensor, M: int, w: PackedWeight, x: torch.Tensor):
    G = w.K // w.group
    if (not xsums.is_cuda or xsums.dtype != torch.float32 or tuple(xsums.shape) != (M, G)
            or not xsums.is_contiguous() or xsums.device != x.device):
        raise ValueError(f"xsums must be a contiguous CUDA float32 [{M}, {G}] tensor on {x.device}")


def run_exact_sums(w: PackedWeight, x: torch.Tensor, xsums: torch.Tensor, y: torch.Tensor | None = None,
                   workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """affqmm_run_exact_sums (M <= 16): the exact-codes form with the group sums
    of x (float32 [M, K/group]) as the kernel that produced x wrote them."""
    _check_x(x, w.K)
    M = x.shape[0]
    _check_xsums(xsums, M, w, x)
    dev = x.get_device()
    if y is None:
        y = torch.empty(M, w.N, dtype=torch.bfloat16, device=x.device)
    sp = _stream_ptr(stream, dev)
    ws = workspace or default_workspace(dev, sp)
    need = workspace_bytes(w, M)
    buf = ws.get(need)
    cw = w.cstruct()
    _check(lib().affqmm_run_exact_sums(ctypes.byref(cw), x.data_ptr(), xsums.data_ptr(), M, y.data_ptr(),
                                       buf.data_ptr() if need else None, buf.numel(), sp), "affqmm_run_exact_sums")
    return y


def run_geglu(w: PackedWeight, x: torch.Tensor, form: int = FORM_ROUNDED, xsums: torch.Tensor | None = None,
              h: torch.Tensor | None = None, workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """affqmm_run_geglu (M <= 16): a gate/up stack (rows interleaved in 16-row
    blocks) with GeGLU as its epilogue; returns h bf16 [M, N/2]."""
    _check_x(x, w.K)
    M = x.shape[0]
    if form == FORM_EXACT_SUMS:
        _check_xsums(xsums, M, w, x)
    dev = x.get_device()
    if h is None:
        h = torch.empty(M, w.N // 2, dtype=torch.bfloat16, device=x.device)
    sp = _stream_ptr(stream, dev)
    ws = workspace or default_workspace(dev, sp)
    need = workspace_bytes(w, M)
    buf = ws.get(need)
    cw = w.cstruct()
    xs = xsums.data_ptr() if (form == FORM_EXACT_SUMS and xsums is not None) else None
    _check(lib().affqmm_run_geglu(ctypes.byref(cw), x.data_ptr(), xs, M, int(form), h.data_ptr(),
                                  buf.data_ptr() if need else None, buf.numel(), sp), "affqmm_run_geglu")
    return h


def run_host(w: PackedWeight, x: torch.Tensor, y: torch.Tensor, x_dev: torch.Tensor, y_dev: torch.Tensor,
             workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """affqmm_run_host: x (host, bf16 [M, K]) is copied into x_dev, the projection
    runs into y_dev, and y_dev is copied back into y (host, bf16 [M, N]), all on
    the stream.  Pinned host tensors keep the copies asynchronous; y is complete
    once the stream has passed the call."""
    M = x.shape[0]
    if (x.is_cuda or y.is_cuda or x.dtype != torch.bfloat16 or y.dtype != torch.bfloat16
            or tuple(x.shape) != (M, w.K) or tuple(y.shape) != (M, w.N)
            or not x.is_contiguous() or not y.is_contiguous()):
        raise ValueError(f"x and y must be contiguous host bf16 tensors [M, {w.K}] and [M, {w.N}]")
    _check_x(x_dev, w.K)
    if (x_dev.shape[0] != M or y_dev.dtype != torch.bfloat16 or tuple(y_dev.shape) != (M, w.N)
            or not y_dev.is_contiguous() or y_dev.device != x_dev.device):
        raise ValueError(f"x_dev and y_dev must be contiguous bf16 [M, {w.K}] and [M, {w.N}] on one device")
    dev = x_dev.get_device()
    sp = _stream_ptr(stream, dev)
    ws = workspace or default_workspace(dev, sp)
    need = workspace_bytes(w, M)
    buf = ws.get(need)
    cw = w.cstruct()
    _check(lib().affqmm_run_host(ctypes.byref(cw), x.data_ptr(), M, y.data_ptr(), x_dev.data_ptr(), y_dev.data_ptr(),
                                 buf.data_ptr() if need else None, buf.numel(), sp), "affqmm_run_host")
    return y


def run_stacked(ws_list, x: torch.Tensor, ys=None, workspace: Workspace | None = None, stream=None):
    """Several projections of the same x in one launch; returns a list of y."""
    K = ws_list[0].K
    _check_x(x, K)
    M = x.shape[0]
    if ys is None:
        ys = [torch.empty(M, w.N, dtype=torch.bfloat16, device=x.device) for w in ws_list]
    sp = _stream_ptr(stream, x.get_device())
    wsp = workspace or default_workspace(x.get_device(), sp)
    need = workspace_bytes_stacked(ws_list, M)
    buf = wsp.get(need)
    arr = _warray(ws_list)
    yp = (ctypes.c_void_p * len(ys))(*[y.data_ptr() for y in ys])
    _check(lib().affqmm_run_stacked(len(ws_list), arr, x.data_ptr(), M, yp, buf.data_ptr() if need else None,
                                    buf.numel(), sp), "affqmm_run_stacked")
    return ys


def dequant(w: PackedWeight, stream=None) -> torch.Tensor:
    """The bf16 [N, K] weights as the run kernels dequantize them (test hook)."""
    out = torch.empty(w.N, w.K, dtype=torch.bfloat16, device=w.packed.device)
    cw = w.cstruct()
    _check(lib().affqmm_dequant(ctypes.byref(cw), out.data_ptr(), _stream_ptr(stream)), "affqmm_dequant")
    return out


def workspace_status(buf: torch.Tensor, stream=None) -> int:
    """Read a workspace's device status word (0 = ok; after a timeout the
    library zeroes the status word and the merge counters again)."""
    return int(lib().affqmm_workspace_status(buf.data_ptr(), _stream_ptr(stream)))


def test_fault_wait(cycles: int) -> None:
    """Test hook: while cycles > 0, decode launches (M <= 16) first wait, at
    most `cycles` SM clock cycles, on a barrier nothing completes, so the
    bounded wait runs out and the workspace status reports a timeout."""
    _check(lib().affqmm_test_fault_wait(int(cycles)), "affqmm_test_fault_wait")


def run_noalloc(w: PackedWeight, x: torch.Tensor, y: torch.Tensor, stream=None) -> torch.Tensor:
    """affqmm_run_noalloc: y = bf16(x @ dequant(W)^T) for M <= 16 rows, with no
    workspace.  For callers that cannot allocate device memory; the library
    works in its own fixed 8 MiB scratch array instead, shared by every call on
    the device, so calls must not overlap on the GPU.  `y` must be given: this
    wrapper allocates nothing either."""
    _check_x(x, w.K)
    M = x.shape[0]
    if y.dtype != torch.bfloat16 or tuple(y.shape) != (M, w.N) or not y.is_contiguous() or y.device != x.device:
        raise ValueError(f"y must be a contiguous bf16 [{M}, {w.N}] tensor on {x.device}")
    cw = w.cstruct()
    _check(lib().affqmm_run_noalloc(ctypes.byref(cw), x.data_ptr(), M, y.data_ptr(), _stream_ptr(stream)),
           "affqmm_run_noalloc")
    return y


def _embed_args(w: PackedWeight, ids: torch.Tensor, scale, out):
    if not ids.is_cuda or ids.dtype != torch.int32 or ids.dim() != 1 or not ids.is_contiguous():
        raise ValueError("ids must be a contiguous int32 CUDA vector")
    T = ids.shape[0]
    if out is None:
        out = torch.empty(T, w.K, dtype=torch.bfloat16, device=ids.device)
    if out.dtype != torch.bfloat16 or tuple(out.shape) != (T, w.K) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous bf16 [{T}, {w.K}] tensor")
    sbits = 0 if scale is None else int(torch.tensor([scale], dtype=torch.bfloat16).view(torch.int16).item()) & 0xFFFF
    return T, out, sbits


def embed_rows(w: PackedWeight, ids: torch.Tensor, scale: float | None = None, out: torch.Tensor | None = None,
               status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[t, k] = bf16(W[ids[t], k] * bf16(scale)) (or W's rows when scale is None),
    W = bf16(s*q + b): rows gathered from the packed table.  ids: int32 CUDA [T]."""
    T, out, sbits = _embed_args(w, ids, scale, out)
    cw = w.cstruct()
    _check(lib().affqmm_embed_rows(ctypes.byref(cw), ids.data_ptr(), T, 0 if scale is None else 1, sbits,
                                   out.data_ptr(), status.data_ptr() if status is not None else None,
                                   _stream_ptr(stream)), "affqmm_embed_rows")
    return out


def rows_bytes(bits: int, group: int, N: int, K: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().affqmm_rows_bytes(bits, group, N, K, ctypes.byref(out)), "affqmm_rows_bytes")
    return out.value


def pack_rows(w: PackedWeight, stream=None) -> torch.Tensor:
    """The row-contiguous copy of a packed table that embed_rows_copy gathers from."""
    nbytes = rows_bytes(w.bits, w.group, w.N, w.K)
    rows = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=w.packed.device)
    cw = w.cstruct()
    _check(lib().affqmm_pack_rows(ctypes.byref(cw), rows.data_ptr(), _stream_ptr(stream)), "affqmm_pack_rows")
    return rows


def embed_rows_copy(w: PackedWeight, rows: torch.Tensor, ids: torch.Tensor, scale: float | None = None,
                    out: torch.Tensor | None = None, status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """embed_rows, reading the rows from `rows` = pack_rows(w) (the same values)."""
    T, out, sbits = _embed_args(w, ids, scale, out)
    if not rows.is_cuda or rows.dtype != torch.uint8 or rows.numel() < rows_bytes(w.bits, w.group, w.N, w.K):
        raise ValueError("rows must be the uint8 CUDA copy made by pack_rows(w)")
    cw = w.cstruct()
    _check(lib().affqmm_embed_rows_copy(ctypes.byref(cw), rows.data_ptr(), ids.data_ptr(), T,
                                        0 if scale is None else 1, sbits, out.data_ptr(),
                                        status.data_ptr() if status is not None else None, _stream_ptr(stream)),
           "affqmm_embed_rows_copy")
    return out
