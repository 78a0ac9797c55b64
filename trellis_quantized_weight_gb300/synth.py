"""Seeded synthetic inputs for the packed-Trellis decode and product.

This module only draws random numbers and lays them out; it holds none of the
decode or product arithmetic, and both the CUDA path and the CPU oracle are fed
from it.  Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), one independent stream per
tensor, all derived from one per-workload seed.

Inputs follow the shapes and distributions of the quantised-linear workloads:
  codes  uint32 [N, K*k/32]  uniform random words (every bit pattern is a valid
                             code, so random words exercise exactly the work of
                             trained codes);
  scales bf16 [N]            U(0.005, 0.02);
  x      bf16 [M, K]         N(0, sigma^2) by Box-Muller on 53-bit uniforms.
bf16 rounding of the drawn float32 values is torch's round-to-nearest-even
conversion.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)

TAG_CODES, TAG_SCALES, TAG_X = 1, 2, 3


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset+1 .. offset+n of splitmix64 started from ``seed`` (uint64 array)."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
        return z ^ (z >> np.uint64(31))


def _stream_seed(seed: int, tag: int) -> int:
    return ((seed & 0xFFFFFFFF) << 8 | tag) & 0xFFFFFFFFFFFFFFFF


def uniform01(seed: int, n: int) -> np.ndarray:
    """float64 uniforms in [0, 1) from the top 53 bits of each output."""
    return (splitmix64(seed, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def to_bf16_bits(a) -> np.ndarray:
    """Round float values to bf16 (nearest, ties to even) and return the uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def codes_words(seed: int, N: int, K: int, k: int) -> np.ndarray:
    words = N * K * k // 32
    raw = splitmix64(_stream_seed(seed, TAG_CODES), (words + 1) // 2)
    return raw.view(np.uint32)[:words].reshape(N, K * k // 32).copy()


def scales_bf16(seed: int, N: int, lo: float = 0.005, hi: float = 0.02) -> np.ndarray:
    u = uniform01(_stream_seed(seed, TAG_SCALES), N)
    return to_bf16_bits(lo + (hi - lo) * u)


def x_bf16(seed: int, M: int, K: int, sigma: float = 1.0) -> np.ndarray:
    n = M * K
    u = uniform01(_stream_seed(seed, TAG_X), 2 * n)
    u1 = 1.0 - u[0::2]          # (0, 1]
    u2 = u[1::2]
    g = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return to_bf16_bits(sigma * g).reshape(M, K)


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    k: int
    sigma: float
    seed: int
    L: int = 12
    T: int = 256

    @property
    def row_words(self) -> int:
        return self.K * self.k // 32

    @property
    def weights(self) -> int:
        return self.N * self.K

    @property
    def code_bytes(self) -> int:
        return self.N * self.row_words * 4

    def generate(self):
        """(x [M,K] uint16 bf16 bits, codes [N, K*k/32] uint32, scales [N] uint16 bf16 bits)."""
        return (x_bf16(self.seed, self.M, self.K, self.sigma),
                codes_words(self.seed, self.N, self.K, self.k),
                scales_bf16(self.seed, self.N))


def _wl(i, name, M, K, N, k, sigma):
    return Workload(name=name, M=M, K=K, N=N, k=k, sigma=sigma, seed=0x5EED0000 + i)


# The five quantised-linear shapes: MLP gate/up projections of a 5120-wide
# model at three bit widths, its down projection at M=1, and a 64-token
# prefill chunk.
WORKLOADS = {
    w.name: w for w in [
        _wl(0, "gemm_m5_k5120_n17408_k2", 5, 5120, 17408, 2, 1.0),
        _wl(1, "gemm_m8_k5120_n17408_k3", 8, 5120, 17408, 3, 1.0),
        _wl(2, "gemm_m15_k5120_n17408_k4", 15, 5120, 17408, 4, 1.0),
        _wl(3, "gemv_m1_k17408_n5120_k4", 1, 17408, 5120, 4, 0.5),
        _wl(4, "prefill_m64_k5120_n17408_k4", 64, 5120, 17408, 4, 1.0),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)


def small(M: int, K: int, N: int, k: int, seed: int, sigma: float = 1.0) -> Workload:
    """A small seeded case of the same distributions (for parity at several tiles)."""
    return Workload(name=f"small_m{M}_k{K}_n{N}_k{k}", M=M, K=K, N=N, k=k, sigma=sigma, seed=seed)
