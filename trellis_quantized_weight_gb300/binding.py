"""Thin ctypes binding of libtrellis_gb300.so (the C ABI in include/trellis.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their data pointers and the current CUDA stream are handed to the
library, and a non-zero status raises ``TrellisError``.  Every step of the
decode and product runs in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

STATUS = {
    0: "TRELLIS_OK", -1: "TRELLIS_ERR_NULL", -2: "TRELLIS_ERR_SHAPE", -3: "TRELLIS_ERR_UNSUPPORTED",
    -4: "TRELLIS_ERR_ALIGN", -5: "TRELLIS_ERR_CUDA", -6: "TRELLIS_ERR_TIMEOUT", -7: "TRELLIS_ERR_WORKSPACE",
}

# Exported functions: name -> (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
SIGNATURES = {
    "trellis_abi_version": (_I, []),
    "trellis_status_string": (ctypes.c_char_p, [_I]),
    "trellis_decode": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "trellis_gemm": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "trellis_gemm_workspace_size": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "trellis_gemm_ws": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "trellis_gemm_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "trellis_device_status": (_I, [_P]),
    "trellis_selftest_wait_timeout": (_I, [_P]),
    "trellis_gemm_gateup": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "trellis_gemm_gateup_workspace_size": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "trellis_gemm_packed": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "trellis_gemm_packed_workspace_size": (_I, [_P, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
}


class TrellisError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: the CUDA library has not been built "
                    "(run trellis_quantized_weight_gb300.build.build())")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def status_string(status: int) -> str:
    try:
        return load().trellis_status_string(status).decode()
    except Exception:  # the message is only decoration
        return STATUS.get(status, "TRELLIS_ERR_UNKNOWN")


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise TrellisError(rc, where)


# ---- raw ABI calls (integer pointers; used by tests and the benchmark) ----
def abi_decode(codes_ptr, scales_ptr, K, N, k, L, T, out_ptr, stream) -> int:
    return load().trellis_decode(codes_ptr, scales_ptr, K, N, k, L, T, out_ptr, stream)


def abi_gemm(x_ptr, codes_ptr, scales_ptr, M, K, N, k, L, T, out_ptr, stream) -> int:
    return load().trellis_gemm(x_ptr, codes_ptr, scales_ptr, M, K, N, k, L, T, out_ptr, stream)


def abi_gemm_ws(x_ptr, codes_ptr, scales_ptr, M, K, N, k, L, T, out_ptr, ws_ptr, ws_bytes, stream) -> int:
    return load().trellis_gemm_ws(x_ptr, codes_ptr, scales_ptr, M, K, N, k, L, T, out_ptr, ws_ptr,
                                  ws_bytes, stream)


def gemm_workspace_bytes(M, K, N, k, L=12, T=256) -> int:
    n = ctypes.c_size_t(0)
    _check(load().trellis_gemm_workspace_size(M, K, N, k, L, T, ctypes.byref(n)),
           "trellis_gemm_workspace_size")
    return int(n.value)


def gemm_gateup_workspace_bytes(M, K, N, k, L=12, T=256) -> int:
    n = ctypes.c_size_t(0)
    _check(load().trellis_gemm_gateup_workspace_size(M, K, N, k, L, T, ctypes.byref(n)),
           "trellis_gemm_gateup_workspace_size")
    return int(n.value)


def gemm_packed_workspace_bytes(rows, K, N, k, L=12, T=256) -> int:
    r = (ctypes.c_int * len(rows))(*rows)
    n = ctypes.c_size_t(0)
    _check(load().trellis_gemm_packed_workspace_size(r, len(rows), K, N, k, L, T, ctypes.byref(n)),
           "trellis_gemm_packed_workspace_size")
    return int(n.value)


# ---- torch-facing API ------------------------------------------------------
def _torch():
    import torch
    return torch


def _stream_handle(device, stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _require(t, name, dtypes, ndim):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


_ws_cache: dict = {}
_ws_lock = threading.Lock()


def _workspace(device, nbytes: int, stream=None):
    """A zero-filled torch buffer per (device, stream), reused across calls and grown
    as needed.  It is allocated and zero-filled on the stream the calls run on, so
    stream order alone makes the fill land first and lets torch's caching allocator
    recycle an outgrown buffer once the calls enqueued before it are done: no host
    synchronisation.  One buffer per stream also keeps calls on different streams
    off each other's split-K counters."""
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (torch.device(device).index, s.cuda_stream)
    with _ws_lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < nbytes:
            with torch.cuda.stream(s):
                buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws_cache[key] = buf
    return buf


def decode(codes, scales, K: int, k: int, L: int = 12, T: int = 256, out=None, stream=None):
    """Dense bf16 weights [N, K] from packed codes [N, K*k/32] and bf16 scales [N]."""
    torch = _torch()
    _require(codes, "codes", (torch.int32, torch.uint32), 2)
    _require(scales, "scales", (torch.bfloat16,), 1)
    N = codes.shape[0]
    if codes.shape[1] * 32 != K * k or scales.numel() != N:
        raise ValueError("codes must be [N, K*k/32] and scales [N]")
    if out is None:
        out = torch.empty((N, K), dtype=torch.bfloat16, device=codes.device)
    _require(out, "out", (torch.bfloat16,), 2)
    if tuple(out.shape) != (N, K):
        raise ValueError("out must be [N, K]")
    rc = abi_decode(codes.data_ptr(), scales.data_ptr(), K, N, k, L, T, out.data_ptr(),
                    _stream_handle(codes.device, stream))
    _check(rc, "trellis_decode")
    return out


def gemm(x, codes, scales, k: int, L: int = 12, T: int = 256, out=None, stream=None):
    """out [M, N] bf16 = x [M, K] times the decoded weights [N, K] transposed."""
    torch = _torch()
    _require(x, "x", (torch.bfloat16,), 2)
    _require(codes, "codes", (torch.int32, torch.uint32), 2)
    _require(scales, "scales", (torch.bfloat16,), 1)
    M, K = x.shape
    N = codes.shape[0]
    if codes.shape[1] * 32 != K * k or scales.numel() != N:
        raise ValueError("codes must be [N, K*k/32] and scales [N]")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _require(out, "out", (torch.bfloat16,), 2)
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be [M, N]")
    nbytes = gemm_workspace_bytes(M, K, N, k, L, T)
    ws = _workspace(x.device, max(nbytes, 256), stream)
    rc = abi_gemm_ws(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), M, K, N, k, L, T,
                     out.data_ptr(), ws.data_ptr(), ws.numel(), _stream_handle(x.device, stream))
    _check(rc, "trellis_gemm_ws")
    return out


def gemm_gateup(x, codes_gate, scales_gate, codes_up, scales_up, k: int, act: bool = True, L: int = 12,
                T: int = 256, stream=None):
    """The two projections that share x: returns (gate [M, N], up [M, N], act [M, N] or None)
    with act = bf16(silu(gate) * up)."""
    torch = _torch()
    _require(x, "x", (torch.bfloat16,), 2)
    for name, c, sc in (("gate", codes_gate, scales_gate), ("up", codes_up, scales_up)):
        _require(c, f"codes_{name}", (torch.int32, torch.uint32), 2)
        _require(sc, f"scales_{name}", (torch.bfloat16,), 1)
    M, K = x.shape
    N = codes_gate.shape[0]
    if tuple(codes_up.shape) != tuple(codes_gate.shape) or codes_gate.shape[1] * 32 != K * k:
        raise ValueError("codes_gate and codes_up must both be [N, K*k/32]")
    if scales_gate.numel() != N or scales_up.numel() != N:
        raise ValueError("scales must be [N]")
    g = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    u = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    a = torch.empty((M, N), dtype=torch.bfloat16, device=x.device) if act else None
    nbytes = gemm_gateup_workspace_bytes(M, K, N, k, L, T)
    ws = _workspace(x.device, max(nbytes, 256), stream)
    rc = load().trellis_gemm_gateup(x.data_ptr(), codes_gate.data_ptr(), scales_gate.data_ptr(),
                                    codes_up.data_ptr(), scales_up.data_ptr(), M, K, N, k, L, T,
                                    g.data_ptr(), u.data_ptr(), a.data_ptr() if act else None,
                                    ws.data_ptr(), ws.numel(), _stream_handle(x.device, stream))
    _check(rc, "trellis_gemm_gateup")
    return g, u, a



def gemm_packed(xs, codes, scales, k: int, L: int = 12, T: int = 256, outs=None, stream=None):
    """Token packing: one product for several groups of activation rows sharing the
    weights.  xs: list of bf16 [rows_g, K]; returns the list of bf16 [rows_g, N]."""
    torch = _torch()
    xs = list(xs)
    if not xs:
        raise ValueError("xs must hold at least one group")
    for i, x in enumerate(xs):
        _require(x, f"xs[{i}]", (torch.bfloat16,), 2)
    _require(codes, "codes", (torch.int32, torch.uint32), 2)
    _require(scales, "scales", (torch.bfloat16,), 1)
    K = xs[0].shape[1]
    N = codes.shape[0]
    if any(x.shape[1] != K for x in xs) or codes.shape[1] * 32 != K * k or scales.numel() != N:
        raise ValueError("every x must be [rows, K] with codes [N, K*k/32] and scales [N]")
    rows = [int(x.shape[0]) for x in xs]
    if outs is None:
        outs = [torch.empty((r, N), dtype=torch.bfloat16, device=xs[0].device) for r in rows]
    for i, (o, r) in enumerate(zip(outs, rows)):
        _require(o, f"outs[{i}]", (torch.bfloat16,), 2)
        if tuple(o.shape) != (r, N):
            raise ValueError(f"outs[{i}] must be [{r}, {N}]")
    nbytes = gemm_packed_workspace_bytes(rows, K, N, k, L, T)
    ws = _workspace(xs[0].device, max(nbytes, 256), stream)
    xp = (ctypes.c_void_p * len(xs))(*[x.data_ptr() for x in xs])
    op = (ctypes.c_void_p * len(outs))(*[o.data_ptr() for o in outs])
    rp = (ctypes.c_int * len(rows))(*rows)
    rc = load().trellis_gemm_packed(xp, rp, len(rows), codes.data_ptr(), scales.data_ptr(), K, N, k, L, T, op,
                                    ws.data_ptr(), ws.numel(), _stream_handle(xs[0].device, stream))
    _check(rc, "trellis_gemm_packed")
    return outs
