"""GPU parity for the general geometry: k = 1..8 bits per weight and window
widths k < L <= 24 (T = 256).  The page's wrapper accepts only k in {2,3,4}
with L = 12; the same definition (window at bit (T-1-t)*k, wrapping to word 0
of the block, hash, byte sum, quotient, scale) is taken for the rest.  These
run on the kernels built for a run-time window width, with the computed
quotient.

Decode must match the oracle bit for bit; the product stays within
max(2 bf16 ulp, 1e-4 * sum_k |w_k x_k|) of the oracle's fp32 result, on the
CUDA-core path (M <= 16) and on the tensor cores (M > 16).
"""
import numpy as np
import pytest

from helpers import (assert_gemm_close, bf16_to_f32, dev_bf16, dev_codes, host_bits, oracle_decode_par,
                     oracle_gemm_par, ulp_bf16_of)

pytestmark = pytest.mark.gpu

# every k with its smallest, a middle and the largest window width
GEOMETRIES = [(k, L) for k in range(1, 9) for L in sorted({k + 1, max(k + 1, 12), 16, 24})]


@pytest.fixture(scope="module")
def tq():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from trellis_quantized_weight_gb300 import build
    build.build()
    import trellis_quantized_weight_gb300 as tq
    tq.load()
    return tq


def _inputs(M, K, N, k, seed, sigma=1.0):
    from trellis_quantized_weight_gb300 import synth
    return synth.small(M, K, N, k, seed, sigma).generate()


@pytest.mark.parametrize("k,L", GEOMETRIES)
def test_decode_general_geometry_bitexact(tq, oracle_lib, k, L):
    N, K = 45, 768    # 3 blocks a row, a ragged number of rows
    _, codes, scales = _inputs(1, K, N, k, seed=31 * k + L)
    got = host_bits(tq.decode(dev_codes(codes), dev_bf16(scales), K, k, L=L))
    want = oracle_decode_par(oracle_lib, codes, scales, K, N, k, L=L)
    assert np.array_equal(got, want), f"k={k} L={L}: {int((got != want).sum())} weights differ"


@pytest.mark.parametrize("k,L", [(1, 2), (1, 12), (2, 16), (3, 7), (4, 24), (5, 12), (6, 9), (7, 20), (8, 24)])
@pytest.mark.parametrize("M", [1, 3, 8, 13, 16, 17, 64, 100, 200])
def test_gemm_general_geometry(tq, oracle_lib, k, L, M):
    import torch
    from trellis_quantized_weight_gb300 import binding
    N, K = 300, 512
    x, codes, scales = _inputs(M, K, N, k, seed=4000 + 97 * k + 7 * L + M)
    dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
    pad = 4
    out = torch.full(((M + pad) * N,), 0x7FC1, dtype=torch.int16, device="cuda")
    rc = binding.abi_gemm(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, L, 256, out.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    assert rc == 0, binding.status_string(rc)
    torch.cuda.synchronize()
    assert binding.load().trellis_device_status(None) == 0
    bits = out.cpu().numpy().view(np.uint16)
    assert np.all(bits[M * N:] == 0x7FC1), "rows beyond M were written"
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k, L=L)
    ref, refabs = oracle_gemm_par(oracle_lib, x, w)
    assert_gemm_close(bits[: M * N].reshape(M, N), ref, refabs, f"M={M} k={k} L={L}")


@pytest.mark.parametrize("k,L,M", [(8, 16, 15), (4, 16, 16), (6, 20, 16), (7, 12, 16), (8, 9, 14)])
def test_gemm_general_two_row_shapes(tq, oracle_lib, k, L, M):
    """General-geometry shapes at the top of the small-M range (M = 14 .. 16, the
    most registers a lane, and the shapes that once ran two rows a lane), on
    several tile-groups, a ragged N and K-ranges split over CTAs."""
    N, K = 1001, 2048
    x, codes, scales = _inputs(M, K, N, k, seed=9000 + 17 * M + k + L)
    got = host_bits(tq.gemm(dev_bf16(x), dev_codes(codes), dev_bf16(scales), k, L=L))
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k, L=L)
    ref, refabs = oracle_gemm_par(oracle_lib, x, w)
    assert_gemm_close(got, ref, refabs, f"M={M} k={k} L={L}")


@pytest.mark.parametrize("k,L,M", [(1, 24, 16), (5, 16, 9), (8, 10, 40), (6, 16, 100), (7, 12, 256)])
def test_gemm_general_one_hot_rows_are_exact(tq, oracle_lib, k, L, M):
    """Row i of x selects weight column j_i: each output row is that decoded
    column bit for bit (one exact product plus zeros)."""
    N, K = 200, 1024
    _, codes, scales = _inputs(1, K, N, k, seed=5100 + k + L)
    w = oracle_lib.decode(codes, scales, K, N, k, L=L)
    cols = [(37 * i + 5) % K for i in range(M)]
    e = np.zeros((M, K), np.uint16)
    for i, j in enumerate(cols):
        e[i, j] = 0x3F80
    got = host_bits(tq.gemm(dev_bf16(e), dev_codes(codes), dev_bf16(scales), k, L=L))
    for i, j in enumerate(cols):
        assert np.array_equal(got[i], w[:, j]), (i, j)


@pytest.mark.parametrize("k,L,M", [(5, 16, 8), (1, 12, 3), (6, 20, 64)])
def test_gemm_gateup_general_geometry(tq, oracle_lib, k, L, M):
    """Gate/up outside the fast geometry: the two products run as two launches
    through one workspace, then the activation."""
    from trellis_quantized_weight_gb300 import binding
    N, K = 260, 768
    x, cg, sg = _inputs(M, K, N, k, seed=6100 + 3 * k + L)
    _, cu, su = _inputs(M, K, N, k, seed=6200 + 3 * k + L)
    g, u, a = binding.gemm_gateup(dev_bf16(x), dev_codes(cg), dev_bf16(sg), dev_codes(cu), dev_bf16(su), k,
                                  act=True, L=L)
    g, u, a = host_bits(g), host_bits(u), host_bits(a)
    for got, codes, scales, what in ((g, cg, sg, "gate"), (u, cu, su, "up")):
        w = oracle_decode_par(oracle_lib, codes, scales, K, N, k, L=L)
        ref, refabs = oracle_gemm_par(oracle_lib, x, w)
        assert_gemm_close(got, ref, refabs, f"{what} M={M} k={k} L={L}")
    ref_act = bf16_to_f32(oracle_lib.silu_mul(g, u)).astype(np.float64)
    err = np.abs(bf16_to_f32(a).astype(np.float64) - ref_act)
    assert np.all(err <= ulp_bf16_of(ref_act))


def test_general_geometry_full_size_sampled_rows(tq, oracle_lib):
    """k = 8, L = 16 at the headline shape (M = 8, K = 5120, N = 17408): decode
    bit-exact and product rows checked on a sample of output rows."""
    M, K, N, k, L = 8, 5120, 17408, 8, 16
    x, codes, scales = _inputs(M, K, N, k, seed=7001)
    dc, ds = dev_codes(codes), dev_bf16(scales)
    dec = host_bits(tq.decode(dc, ds, K, k, L=L))
    out = host_bits(tq.gemm(dev_bf16(x), dc, ds, k, L=L))
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([rng.integers(0, N, 48), [0, N - 1]]))
    for n in rows:
        w = oracle_lib.decode(codes, scales, K, N, k, L=L, rows=(int(n), int(n) + 1))
        assert np.array_equal(dec[n], w[0]), n
        ref, refabs = oracle_lib.gemm_dense(x, w)
        assert_gemm_close(out[:, n:n + 1], ref, refabs, f"row {n}")
