"""Test infrastructure: ctypes wrapper around the float64 CPU oracle (oracle.c).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may
import this package.  The product path (``group_affine_bit_gb300`` and
``libaffqmm``) never does; it fails loudly when its own CUDA library is
missing instead of falling back to anything here.

All arrays are numpy: codes uint8 [N,K]; scales, biases uint16 (bf16 bit
patterns) [N,K/g]; x uint16 [M,K].  See oracle.h for the arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def compile_oracle(src: str = SRC, out: str = LIB) -> str:
    """Compile oracle.c (or a copy of it) into a shared library with gcc."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", "-I", HERE, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


class Oracle:
    """Typed calls into one compiled oracle library."""

    def __init__(self, path: str = LIB):
        if path == LIB and (not os.path.exists(LIB) or
                            os.path.getmtime(LIB) < os.path.getmtime(SRC)):
            compile_oracle()
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_from_f32_bits.restype = None
        lib.oracle_bf16_from_f32_bits.argtypes = [_u32p, _u16p, ctypes.c_size_t]
        lib.oracle_dequant_one.restype = ctypes.c_uint16
        lib.oracle_dequant_one.argtypes = [ctypes.c_uint32, ctypes.c_uint16, ctypes.c_uint16]
        lib.oracle_dequant.restype = ctypes.c_int
        lib.oracle_dequant.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64,
                                       _u8p, _u16p, _u16p, _u16p]
        lib.oracle_qmm.restype = ctypes.c_int
        lib.oracle_qmm.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64,
                                   _u16p, _u8p, _u16p, _u16p, _f64p, ctypes.c_int]
        lib.oracle_qmm_groupsum.restype = ctypes.c_int
        lib.oracle_qmm_groupsum.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64,
                                            _u16p, _u8p, _u16p, _u16p, _f64p, _f64p]
        lib.oracle_qmm_groupsum_given.restype = ctypes.c_int
        lib.oracle_qmm_groupsum_given.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, _u16p,
                                                  ctypes.POINTER(ctypes.c_float), _u8p, _u16p, _u16p, _f64p]
        lib.oracle_geglu.restype = None
        lib.oracle_geglu.argtypes = [_i64, _u16p, _u16p, ctypes.c_int, _u16p, _u16p]
        lib.oracle_embed_rows.restype = ctypes.c_int
        lib.oracle_embed_rows.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _u8p, _u16p, _u16p,
                                          ctypes.POINTER(ctypes.c_int32), _i64, ctypes.c_int, ctypes.c_uint16, _u16p]
        self.lib = lib

    # -- bf16 -----------------------------------------------------------
    def bf16_from_double(self, v: float) -> int:
        return int(self.lib.oracle_bf16_from_double(float(v)))

    def bf16_to_double(self, h: int) -> float:
        return float(self.lib.oracle_bf16_to_double(int(h) & 0xFFFF))

    def bf16_from_f32_bits(self, bits: np.ndarray) -> np.ndarray:
        bits = np.ascontiguousarray(bits, dtype=np.uint32)
        out = np.empty(bits.shape, dtype=np.uint16)
        self.lib.oracle_bf16_from_f32_bits(_ptr(bits, _u32p), _ptr(out, _u16p), bits.size)
        return out

    # -- dequant ----------------------------------------------------------
    def dequant_one(self, q: int, s: int, b: int) -> int:
        return int(self.lib.oracle_dequant_one(int(q), int(s) & 0xFFFF, int(b) & 0xFFFF))

    def dequant(self, bits, group, codes, scales, biases) -> np.ndarray:
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        biases = np.ascontiguousarray(biases, dtype=np.uint16)
        N, K = codes.shape
        out = np.empty((N, K), dtype=np.uint16)
        rc = self.lib.oracle_dequant(bits, group, N, K, _ptr(codes, _u8p),
                                     _ptr(scales, _u16p), _ptr(biases, _u16p), _ptr(out, _u16p))
        if rc:
            raise ValueError(f"oracle_dequant rejected its arguments (rc={rc})")
        return out

    # -- projection ---------------------------------------------------------
    def qmm(self, bits, group, x, codes, scales, biases, nthreads: int = 1) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.uint16)
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        biases = np.ascontiguousarray(biases, dtype=np.uint16)
        M, K = x.shape
        N, K2 = codes.shape
        if K != K2:
            raise ValueError("x and codes disagree on K")
        y = np.empty((M, N), dtype=np.float64)
        rc = self.lib.oracle_qmm(bits, group, M, N, K, _ptr(x, _u16p), _ptr(codes, _u8p),
                                 _ptr(scales, _u16p), _ptr(biases, _u16p), _ptr(y, _f64p),
                                 int(nthreads))
        if rc:
            raise ValueError(f"oracle_qmm rejected its arguments (rc={rc})")
        return y

    def qmm_groupsum(self, bits, group, x, codes, scales, biases, nthreads: int = 1):
        """The exact-codes form.  nthreads > 1 splits the output rows n into
        contiguous slices, one C call per slice from a thread pool (ctypes
        releases the GIL); every output is the same single C computation."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        biases = np.ascontiguousarray(biases, dtype=np.uint16)
        M, K = x.shape
        N = codes.shape[0]
        y = np.empty((M, N), dtype=np.float64)
        mag = np.empty((M, N), dtype=np.float64)

        def rows(n0, n1):
            yy = np.empty((M, n1 - n0), dtype=np.float64)
            mm = np.empty((M, n1 - n0), dtype=np.float64)
            rc = self.lib.oracle_qmm_groupsum(bits, group, M, n1 - n0, K, _ptr(x, _u16p),
                                              _ptr(codes[n0:n1], _u8p), _ptr(scales[n0:n1], _u16p),
                                              _ptr(biases[n0:n1], _u16p), _ptr(yy, _f64p), _ptr(mm, _f64p))
            if rc:
                raise ValueError(f"oracle_qmm_groupsum rejected its arguments (rc={rc})")
            y[:, n0:n1] = yy
            mag[:, n0:n1] = mm

        nthreads = max(1, min(int(nthreads), N))
        if nthreads == 1:
            rows(0, N)
        else:
            from concurrent.futures import ThreadPoolExecutor
            cuts = [N * t // nthreads for t in range(nthreads + 1)]
            with ThreadPoolExecutor(nthreads) as ex:
                list(ex.map(lambda t: rows(cuts[t], cuts[t + 1]), range(nthreads)))
        return y, mag

    def qmm_groupsum_given(self, bits, group, x, xsums, codes, scales, biases, nthreads: int = 1):
        """The exact-codes form with the group sums of x given: xsums float32
        [M, K/g].  nthreads > 1 splits the output rows n into slices, one C call
        per slice from a thread pool."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        xsums = np.ascontiguousarray(xsums, dtype=np.float32)
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        biases = np.ascontiguousarray(biases, dtype=np.uint16)
        M, K = x.shape
        N = codes.shape[0]
        if xsums.shape != (M, K // group):
            raise ValueError("xsums must be [M, K/group]")
        y = np.empty((M, N), dtype=np.float64)

        def rows(n0, n1):
            yy = np.empty((M, n1 - n0), dtype=np.float64)
            rc = self.lib.oracle_qmm_groupsum_given(bits, group, M, n1 - n0, K, _ptr(x, _u16p),
                                                    xsums.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                                    _ptr(codes[n0:n1], _u8p), _ptr(scales[n0:n1], _u16p),
                                                    _ptr(biases[n0:n1], _u16p), _ptr(yy, _f64p))
            if rc:
                raise ValueError(f"oracle_qmm_groupsum_given rejected its arguments (rc={rc})")
            y[:, n0:n1] = yy

        nthreads = max(1, min(int(nthreads), N))
        if nthreads == 1:
            rows(0, N)
        else:
            from concurrent.futures import ThreadPoolExecutor
            cuts = [N * t // nthreads for t in range(nthreads + 1)]
            with ThreadPoolExecutor(nthreads) as ex:
                list(ex.map(lambda t: rows(cuts[t], cuts[t + 1]), range(nthreads)))
        return y

    # -- GeGLU ---------------------------------------------------------------------
    def geglu(self, gate, up, tanh_ulps: int = 4):
        """h = gelu_approx(gate) * up as bf16 operations (bit patterns in, bit
        patterns out): returns (h_lo, h_hi), the results for the bf16 roundings
        of tanh on either side of an fp32 tanh within tanh_ulps ulps."""
        gate = np.ascontiguousarray(gate, dtype=np.uint16)
        up = np.ascontiguousarray(up, dtype=np.uint16)
        if gate.shape != up.shape:
            raise ValueError("gate and up differ in shape")
        lo = np.empty(gate.shape, dtype=np.uint16)
        hi = np.empty(gate.shape, dtype=np.uint16)
        self.lib.oracle_geglu(gate.size, _ptr(gate, _u16p), _ptr(up, _u16p), int(tanh_ulps), _ptr(lo, _u16p),
                              _ptr(hi, _u16p))
        return lo, hi

    # -- scaled embedding rows -------------------------------------------------
    def embed_rows(self, bits, group, codes, scales, biases, ids, scale=None) -> np.ndarray:
        """out[t,k] = bf16(bf16(s*q + b) * scale) of table row ids[t]; scale is a
        bf16 bit pattern, or None for the weight row itself."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        biases = np.ascontiguousarray(biases, dtype=np.uint16)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        N, K = codes.shape
        T = ids.shape[0]
        out = np.empty((T, K), dtype=np.uint16)
        rc = self.lib.oracle_embed_rows(bits, group, N, K, _ptr(codes, _u8p), _ptr(scales, _u16p),
                                        _ptr(biases, _u16p), ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), T,
                                        0 if scale is None else 1, 0 if scale is None else int(scale), _ptr(out, _u16p))
        if rc:
            raise ValueError(f"oracle_embed_rows rejected its arguments (rc={rc})")
        return out


_DEFAULT = None


def load() -> Oracle:
    """The oracle built from oracle.c in this directory (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
