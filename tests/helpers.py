"""Shared test plumbing: host<->device copies and a row-parallel oracle driver.

The row-parallel driver only splits the oracle's row range over threads (the
ctypes calls release the GIL); every row is still computed by the unchanged
single-threaded oracle function.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle


def dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_codes(words: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(words).view(np.int32)).cuda()


def host_bits(t) -> np.ndarray:
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


# the spacing of bf16 values at |v| (the smallest normal spacing below 2^-126):
# the oracle's, pinned in test_tolerance_pins.py
ulp_bf16_of = oracle.ulp_bf16


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def oracle_decode_par(o, codes, scales, K, N, k, rows=None, L=12):
    n0, n1 = rows if rows is not None else (0, N)
    nt = _threads()
    edges = np.linspace(n0, n1, nt + 1).astype(int)
    parts = [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:]) if b > a]
    with cf.ThreadPoolExecutor(nt) as ex:
        outs = list(ex.map(lambda r: o.decode(codes, scales, K, N, k, L=L, rows=r), parts))
    return np.concatenate(outs, axis=0) if outs else np.empty((0, K), np.uint16)


def oracle_gemm_par(o, x, w_rows):
    nt = _threads()
    n = w_rows.shape[0]
    edges = np.linspace(0, n, nt + 1).astype(int)
    parts = [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:]) if b > a]
    with cf.ThreadPoolExecutor(nt) as ex:
        res = list(ex.map(lambda r: o.gemm_dense(x, w_rows[r[0]:r[1]]), parts))
    ref = np.concatenate([r[0] for r in res], axis=1)
    refabs = np.concatenate([r[1] for r in res], axis=1)
    return ref, refabs


def assert_gemm_close(got_bits: np.ndarray, ref: np.ndarray, refabs: np.ndarray, what: str = ""):
    """|gpu - ref| <= max(2 bf16 ulp of ref, 1e-4 * sum_k |w x|), element by element."""
    got = bf16_to_f32(got_bits).astype(np.float64)
    tol = oracle.gemm_tolerance(ref, refabs)
    err = np.abs(got - ref.astype(np.float64))
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs out of tolerance; first at {tuple(i)}: "
            f"gpu={got[tuple(i)]!r} ref={ref[tuple(i)]!r} tol={tol[tuple(i)]!r}")
