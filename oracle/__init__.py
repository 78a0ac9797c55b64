"""CPU oracle for the packed-Trellis decode and decode-and-multiply.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``trellis_quantized_weight_gb300``) never imports it.

The arithmetic lives in ``trellis_oracle.c`` (plain single-threaded C99, built
with ``gcc -ffp-contract=off``); this module compiles it on demand and exposes
it on numpy arrays through ctypes.  It follows the Metal kernel source on the
page "mlx-bun 0.2.0 -> 0.4.0", package/src/model/trellis-wide-prefill.ts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "trellis_oracle.c")
_DEFAULT_LIB = os.path.join(_HERE, "_build", "liboracle.so")
CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fexcess-precision=standard", "-Wall", "-Wextra"]

_lock = threading.Lock()
_cached = None


def compile_source(src_path: str, out_path: str) -> str:
    """Compile an oracle C source into a shared library at ``out_path``."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-I", _HERE, src_path, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile the oracle library if it is missing or older than its source."""
    if (force or not os.path.exists(_DEFAULT_LIB)
            or os.path.getmtime(_DEFAULT_LIB) < os.path.getmtime(_SRC)
            or os.path.getmtime(_DEFAULT_LIB) < os.path.getmtime(os.path.join(_HERE, "trellis_oracle.h"))):
        compile_source(_SRC, _DEFAULT_LIB)
    return _DEFAULT_LIB


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i64 = ctypes.c_int64
        lib.oracle_window.restype = ctypes.c_uint32
        lib.oracle_window.argtypes = [u32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_code.restype = ctypes.c_int32
        lib.oracle_code.argtypes = [ctypes.c_uint32]
        lib.oracle_value.restype = ctypes.c_float
        lib.oracle_value.argtypes = [ctypes.c_int32]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_weight.restype = ctypes.c_uint16
        lib.oracle_weight.argtypes = [u32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_uint16]
        lib.oracle_check_geometry.restype = ctypes.c_int
        lib.oracle_check_geometry.argtypes = [i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_decode_rows.restype = ctypes.c_int
        lib.oracle_decode_rows.argtypes = [u32p, u16p, i64, i64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, i64, i64, u16p]
        lib.oracle_silu_mul.restype = None
        lib.oracle_silu_mul.argtypes = [u16p, u16p, i64, u16p]
        lib.oracle_gemm_dense.restype = ctypes.c_int
        lib.oracle_gemm_dense.argtypes = [u16p, u16p, i64, i64, i64,
                                          ctypes.POINTER(ctypes.c_float),
                                          ctypes.POINTER(ctypes.c_double)]
        self.lib = lib

    # -- scalar steps ---------------------------------------------------------
    def window(self, blk: np.ndarray, t: int, k: int, L: int, T: int) -> int:
        blk = np.ascontiguousarray(blk, dtype=np.uint32)
        return int(self.lib.oracle_window(_ptr(blk, ctypes.c_uint32), t, k, L, T))

    def code(self, win: int) -> int:
        return int(self.lib.oracle_code(win))

    def value(self, code: int) -> np.float32:
        return np.float32(self.lib.oracle_value(code))

    def bf16_to_f32(self, h: int) -> np.float32:
        return np.float32(self.lib.oracle_bf16_to_f32(h))

    def f32_to_bf16(self, f) -> int:
        return int(self.lib.oracle_f32_to_bf16(float(np.float32(f))))

    def weight(self, blk: np.ndarray, t: int, k: int, L: int, T: int, scale_bf16: int) -> int:
        blk = np.ascontiguousarray(blk, dtype=np.uint32)
        return int(self.lib.oracle_weight(_ptr(blk, ctypes.c_uint32), t, k, L, T, scale_bf16))

    # -- whole arrays ---------------------------------------------------------
    def decode(self, codes: np.ndarray, scales_bf16: np.ndarray, K: int, N: int, k: int,
               L: int = 12, T: int = 256, rows: tuple[int, int] | None = None) -> np.ndarray:
        """bf16 bits (uint16) of rows [n0, n1) of the dense [N, K] weight matrix."""
        n0, n1 = rows if rows is not None else (0, N)
        codes = np.ascontiguousarray(codes, dtype=np.uint32)
        scales_bf16 = np.ascontiguousarray(scales_bf16, dtype=np.uint16)
        assert codes.size == N * K * k // 32 and scales_bf16.size == N
        out = np.empty((n1 - n0, K), dtype=np.uint16)
        rc = self.lib.oracle_decode_rows(_ptr(codes, ctypes.c_uint32), _ptr(scales_bf16, ctypes.c_uint16),
                                         K, N, k, L, T, n0, n1, _ptr(out, ctypes.c_uint16))
        if rc != 0:
            raise ValueError(f"oracle_decode_rows rejected the geometry (status {rc})")
        return out

    def gemm_dense(self, x_bf16: np.ndarray, w_bf16: np.ndarray):
        """(ref fp32 [M, nrows], refabs f64 [M, nrows]) for x [M, K] and dense rows W [nrows, K]."""
        x_bf16 = np.ascontiguousarray(x_bf16, dtype=np.uint16)
        w_bf16 = np.ascontiguousarray(w_bf16, dtype=np.uint16)
        M, K = x_bf16.shape
        nrows = w_bf16.shape[0]
        assert w_bf16.shape[1] == K
        ref = np.empty((M, nrows), dtype=np.float32)
        refabs = np.empty((M, nrows), dtype=np.float64)
        rc = self.lib.oracle_gemm_dense(_ptr(x_bf16, ctypes.c_uint16), _ptr(w_bf16, ctypes.c_uint16),
                                        M, K, nrows, _ptr(ref, ctypes.c_float), _ptr(refabs, ctypes.c_double))
        if rc != 0:
            raise ValueError(f"oracle_gemm_dense rejected the shape (status {rc})")
        return ref, refabs

    def gemm(self, x_bf16: np.ndarray, codes: np.ndarray, scales_bf16: np.ndarray, K: int, N: int,
             k: int, L: int = 12, T: int = 256, rows: tuple[int, int] | None = None):
        """Decode rows [n0, n1) then multiply: (ref [M, n1-n0], refabs [M, n1-n0])."""
        w = self.decode(codes, scales_bf16, K, N, k, L, T, rows)
        return self.gemm_dense(x_bf16, w)

    def silu_mul(self, g_bf16: np.ndarray, u_bf16: np.ndarray) -> np.ndarray:
        """act = bf16(silu(g) * u) elementwise on bf16 bit arrays of one shape."""
        g = np.ascontiguousarray(g_bf16, dtype=np.uint16)
        u = np.ascontiguousarray(u_bf16, dtype=np.uint16)
        if g.shape != u.shape:
            raise ValueError("g and u must have one shape")
        act = np.empty_like(g)
        self.lib.oracle_silu_mul(_ptr(g, ctypes.c_uint16), _ptr(u, ctypes.c_uint16), g.size,
                                 _ptr(act, ctypes.c_uint16))
        return act


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def get() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _cached
    with _lock:
        if _cached is None:
            _cached = Oracle(build())
        return _cached


def ulp_bf16(ref: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |ref| (the min-normal spacing for tiny values)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def gemm_tolerance(ref: np.ndarray, refabs: np.ndarray) -> np.ndarray:
    """Allowed |gpu - ref|: max(2 bf16 ulp of ref, 1e-4 * sum_k |w_k x_k|)."""
    return np.maximum(2.0 * ulp_bf16(ref), 1e-4 * np.asarray(refabs, dtype=np.float64))
