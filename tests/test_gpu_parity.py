"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Decode must match bit for bit.  The product must stay within
max(2 bf16 ulp, 1e-4 * sum_k |w_k x_k|) of the oracle's exactly summed fp32
result, element by element.  Shapes span several tiles, ragged tails, single
blocks, splits of one row's K-range over many CTAs and CTAs that own whole
tile-groups, plus the full-size quantised-linear workloads.
"""
import ctypes

import numpy as np
import pytest

from helpers import (assert_gemm_close, bf16_to_f32, dev_bf16, dev_codes, host_bits,
                     oracle_decode_par, oracle_gemm_par)

pytestmark = pytest.mark.gpu


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


# ------------------------------------------------------------------ decode --
@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("N,K", [(1, 256), (3, 256), (33, 512), (1000, 1024), (77, 256 * 13)])
def test_decode_bitexact(tq, oracle_lib, k, N, K):
    _, codes, scales = _inputs(1, K, N, k, seed=1000 * k + N + K)
    got = host_bits(tq.decode(dev_codes(codes), dev_bf16(scales), K, k))
    want = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("k", [2, 3, 4])
def test_decode_crafted_blocks(tq, oracle_lib, k):
    """Blocks that light up the wrap from the last word to word 0 and every word edge."""
    T, wpb = 256, 256 * k // 32
    rows = []
    for bit in list(range(0, 32)) + [T * k - 1 - i for i in range(32)] + [32 * i + 31 for i in range(wpb)]:
        r = np.zeros(wpb, np.uint32)
        r[bit // 32] |= np.uint32(1 << (bit % 32))
        rows.append(r)
    rows.append(np.full(wpb, 0xFFFFFFFF, np.uint32))
    rows.append(np.zeros(wpb, np.uint32))
    codes = np.stack(rows)
    N = codes.shape[0]
    scales = np.full(N, 0x3F80, np.uint16)       # 1.0: weights are bf16(value) directly
    got = host_bits(tq.decode(dev_codes(codes), dev_bf16(scales), T, k))
    want = oracle_lib.decode(codes, scales, T, N, k)
    assert np.array_equal(got, want)
    assert np.all(got[-2] == 0x3FA3) and np.all(got[-1] == 0xBFA0)   # hand-worked values


# -------------------------------------------------------------------- gemm --
@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 16])
def test_gemm_small(tq, oracle_lib, M, k):
    N, K = 1000, 1024
    x, codes, scales = _inputs(M, K, N, k, seed=77 * M + k)
    got = host_bits(tq.gemm(dev_bf16(x), dev_codes(codes), dev_bf16(scales), k))
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
    ref, refabs = oracle_gemm_par(oracle_lib, x, w)
    assert_gemm_close(got, ref, refabs, f"M={M} k={k}")


@pytest.mark.parametrize("M,K,N,k", [
    (1, 256, 1, 2), (3, 256, 5, 3), (5, 512, 33, 4), (16, 256 * 7, 129, 2),
    (8, 256, 40000, 3),          # many tile-groups, K of one block
    (2, 256, 200000, 4),         # CTAs owning whole tile-groups (no split)
    (9, 256, 90000, 2),          # same with the 8-warp shape
    (1, 256 * 70, 64, 4),        # one tile-group split over every CTA
])
def test_gemm_shapes(tq, oracle_lib, M, K, N, k):
    x, codes, scales = _inputs(M, K, N, k, seed=M * 131 + K + N + k)
    got = host_bits(tq.gemm(dev_bf16(x), dev_codes(codes), dev_bf16(scales), k))
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
    ref, refabs = oracle_gemm_par(oracle_lib, x, w)
    assert_gemm_close(got, ref, refabs, f"M={M} K={K} N={N} k={k}")


@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("N,K", [(128, 256), (300, 512), (1000, 1024), (129, 256 * 9)])
def test_gemm_m64_tensor_cores(tq, oracle_lib, k, N, K):
    """M = 64 runs on tcgen05 (decoded bf16 tiles, fp32 accumulation in tensor memory)."""
    from trellis_quantized_weight_gb300 import binding
    M = 64
    x, codes, scales = _inputs(M, K, N, k, seed=640 + 7 * k + N + K)
    got = host_bits(tq.gemm(dev_bf16(x), dev_codes(codes), dev_bf16(scales), k))
    assert binding.load().trellis_device_status(None) == 0
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
    ref, refabs = oracle_gemm_par(oracle_lib, x, w)
    assert_gemm_close(got, ref, refabs, f"M=64 N={N} K={K} k={k}")


@pytest.mark.parametrize("M", [17, 33, 63, 65, 100, 128, 129, 200, 256, 257, 300, 513])
@pytest.mark.parametrize("k", [2, 3, 4])
def test_gemm_general_m_tensor_cores(tq, oracle_lib, M, k):
    """M > 16 runs on tcgen05 with the MMA's N = 64, 128 or 256 (chunks of 256
    rows above that, the last one overlapping); a partial chunk's missing rows
    are zero-filled or never loaded and never stored: the rows after the output
    (sentinel-filled) stay untouched."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    N, K = 300, 512
    x, codes, scales = _inputs(M, K, N, k, seed=1700 + 3 * M + k)
    dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
    pad = 8
    out = torch.full(((M + pad) * N,), 0x7FC1, dtype=torch.int16, device="cuda")
    rc = binding.abi_gemm(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256,
                          out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, binding.status_string(rc)
    torch.cuda.synchronize()
    assert binding.load().trellis_device_status(None) == 0
    bits = out.cpu().numpy().view(np.uint16)
    got = bits[: M * N].reshape(M, N)
    assert np.all(bits[M * N:] == 0x7FC1), "rows beyond M were written"
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
    ref, refabs = oracle_gemm_par(oracle_lib, x, w)
    assert_gemm_close(got, ref, refabs, f"M={M} N={N} K={K} k={k}")


@pytest.mark.parametrize("M", [100, 300])
def test_gemm_one_hot_rows_are_exact(tq, oracle_lib, M):
    """Each row of x selects a weight column, bit for bit: at M = 100 one
    128-row launch with a partial tile, at M = 300 two overlapping 256-row
    chunks."""
    N, K, k = 256, 1024, 3
    _, codes, scales = _inputs(1, K, N, k, seed=642)
    w = oracle_lib.decode(codes, scales, K, N, k)
    cols = [(53 * i + 11) % K for i in range(M)]
    e = np.zeros((M, K), np.uint16)
    for i, j in enumerate(cols):
        e[i, j] = 0x3F80
    got = host_bits(tq.gemm(dev_bf16(e), dev_codes(codes), dev_bf16(scales), k))
    for i, j in enumerate(cols):
        assert np.array_equal(got[i], w[:, j]), i


@pytest.mark.parametrize("M", [1, 5, 8, 15, 16, 17, 64, 100])
@pytest.mark.parametrize("k", [2, 4])
def test_gemm_gateup(tq, oracle_lib, M, k):
    """Gate and up projections sharing x in one call: each output against the
    oracle product, act = bf16(silu(gate) * up) against the oracle's activation
    of the GPU's own gate/up outputs (within 1 bf16 ulp: fp32 exp on the GPU),
    and nothing written past either [M, N] output (sentinel rows)."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    from helpers import ulp_bf16_of
    N, K = 300, 1024
    x, cg, sg = _inputs(M, K, N, k, seed=2100 + 5 * M + k)
    _, cu, su = _inputs(M, K, N, k, seed=2200 + 5 * M + k)
    dx, dcg, dsg, dcu, dsu = dev_bf16(x), dev_codes(cg), dev_bf16(sg), dev_codes(cu), dev_bf16(su)
    pad = 4
    bufs = [torch.full(((M + pad) * N,), 0x7FC1, dtype=torch.int16, device="cuda") for _ in range(3)]
    need = binding.gemm_gateup_workspace_bytes(M, K, N, k)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    rc = binding.load().trellis_gemm_gateup(dx.data_ptr(), dcg.data_ptr(), dsg.data_ptr(), dcu.data_ptr(),
                                            dsu.data_ptr(), M, K, N, k, 12, 256, bufs[0].data_ptr(),
                                            bufs[1].data_ptr(), bufs[2].data_ptr(), ws.data_ptr(), ws.numel(),
                                            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, binding.status_string(rc)
    torch.cuda.synchronize()
    assert binding.load().trellis_device_status(None) == 0
    host = [b.cpu().numpy().view(np.uint16) for b in bufs]
    for h in host:
        assert np.all(h[M * N:] == 0x7FC1), "rows beyond M were written"
    g, u, a = (h[: M * N].reshape(M, N) for h in host)
    for got, codes, scales, what in ((g, cg, sg, "gate"), (u, cu, su, "up")):
        w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
        ref, refabs = oracle_gemm_par(oracle_lib, x, w)
        assert_gemm_close(got, ref, refabs, f"{what} M={M} k={k}")
    ref_act = bf16_to_f32(oracle_lib.silu_mul(g, u)).astype(np.float64)
    err = np.abs(bf16_to_f32(a).astype(np.float64) - ref_act)
    assert np.all(err <= ulp_bf16_of(ref_act)), f"act: max excess {float((err - ulp_bf16_of(ref_act)).max())}"


@pytest.mark.parametrize("M,N,k", [(8, 1300, 3), (15, 870, 4), (5, 1740, 2)])
def test_gemm_gateup_dead_tile_before_second_matrix(tq, oracle_lib, M, N, k):
    """A CTA's range runs from the first matrix's last tile-group, where whole
    tiles lie past N, into the second matrix's first tile-group: the tiles
    past N request nothing for their next segment, which must then load its
    own codes and scales (K long enough that CTAs take several units)."""
    K = 5120
    x, cg, sg = _inputs(M, K, N, k, seed=2400 + M)
    _, cu, su = _inputs(M, K, N, k, seed=2500 + M)
    g, u, a = tq.gemm_gateup(dev_bf16(x), dev_codes(cg), dev_bf16(sg), dev_codes(cu), dev_bf16(su), k,
                             act=False)
    for got, codes, scales, what in ((g, cg, sg, "gate"), (u, cu, su, "up")):
        w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
        ref, refabs = oracle_gemm_par(oracle_lib, x, w)
        assert_gemm_close(host_bits(got), ref, refabs, f"{what} M={M} N={N} k={k}")


def test_gemm_gateup_without_activation(tq, oracle_lib):
    """act=False returns no third output; gate and up, over a K long enough to be
    split across CTAs, match the oracle products."""
    M, K, N, k = 8, 5120, 2000, 3
    x, cg, sg = _inputs(M, K, N, k, seed=2301)
    _, cu, su = _inputs(M, K, N, k, seed=2302)
    g, u, a = tq.gemm_gateup(dev_bf16(x), dev_codes(cg), dev_bf16(sg), dev_codes(cu), dev_bf16(su), k,
                             act=False)
    assert a is None
    for got, codes, scales, what in ((g, cg, sg, "gate"), (u, cu, su, "up")):
        w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
        ref, refabs = oracle_gemm_par(oracle_lib, x, w)
        assert_gemm_close(host_bits(got), ref, refabs, what)


@pytest.mark.parametrize("k", [2, 3, 4])
def test_gemm_m64_one_hot_is_exact(tq, oracle_lib, k):
    """Each of the 64 rows of x selects a different weight column, bit for bit
    (every k, so every code-word layout of the tensor-core decode)."""
    N, K = 256, 1024
    _, codes, scales = _inputs(1, K, N, k, seed=641 + k)
    w = oracle_lib.decode(codes, scales, K, N, k)
    cols = [(37 * i + 5) % K for i in range(64)]
    e = np.zeros((64, K), np.uint16)
    for i, j in enumerate(cols):
        e[i, j] = 0x3F80
    got = host_bits(tq.gemm(dev_bf16(e), dev_codes(codes), dev_bf16(scales), k))
    for i, j in enumerate(cols):
        assert np.array_equal(got[i], w[:, j]), i


def test_gemm_one_hot_is_exact(tq, oracle_lib):
    """x = e_j picks column j of the decoded weights, bit for bit."""
    N, K, k = 700, 1280, 3
    _, codes, scales = _inputs(1, K, N, k, seed=5)
    w = oracle_lib.decode(codes, scales, K, N, k)
    for j in (0, 255, 256, 777, K - 1):
        e = np.zeros((1, K), np.uint16)
        e[0, j] = 0x3F80
        got = host_bits(tq.gemm(dev_bf16(e), dev_codes(codes), dev_bf16(scales), k))
        assert np.array_equal(got[0], w[:, j])


def test_gemm_deterministic(tq):
    x, codes, scales = _inputs(15, 5120, 3000, 4, seed=9)
    dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
    a = host_bits(tq.gemm(dx, dc, ds, 4))
    b = host_bits(tq.gemm(dx, dc, ds, 4))
    assert np.array_equal(a, b)


def test_gemm_library_workspace_matches(tq):
    """trellis_gemm (the library's static scratch) equals trellis_gemm_ws (caller's)."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    M, K, N, k = 5, 2048, 2000, 2
    x, codes, scales = _inputs(M, K, N, k, seed=12)
    dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
    a = host_bits(tq.gemm(dx, dc, ds, k))
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    rc = binding.abi_gemm(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256,
                          out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert np.array_equal(a, host_bits(out))


def test_gemm_workspace_reuse_across_geometries(tq, oracle_lib):
    """One workspace serves a sequence of geometries without clearing: the tile
    counters sit at a fixed place and every call leaves them at zero."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    cases = [(8, 256, 40000, 3), (2, 256, 100000, 4), (1, 256 * 70, 64, 4), (15, 1024, 3000, 2),
             (8, 256, 40000, 3)]
    need = max(binding.gemm_workspace_bytes(M, K, N, k) for M, K, N, k in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for i, (M, K, N, k) in enumerate(cases):
        x, codes, scales = _inputs(M, K, N, k, seed=900 + i)
        dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert binding.abi_gemm_ws(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256,
                                   out.data_ptr(), ws.data_ptr(), need, s) == 0
        torch.cuda.synchronize()
        w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
        ref, refabs = oracle_gemm_par(oracle_lib, x, w)
        assert_gemm_close(host_bits(out), ref, refabs, f"case {i}")
        assert int(ws[: 1 << 20].count_nonzero()) == 0, "tile counters not left at zero"


def test_gemm_back_to_back_chain(tq, oracle_lib):
    """Calls queued back to back on one stream with no synchronisation between
    them: each layer's output is the next layer's activations, and all share one
    workspace.  A launch may begin while the previous one drains, so this checks
    that every input a call reads, and the workspace, are complete before use."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    M = 8
    layers = [(512, 768, 3), (768, 1280, 4), (1280, 256, 2), (256, 5120, 3), (5120, 512, 4)]
    weights = [_inputs(M, K, N, k, seed=1300 + i)[1:] for i, (K, N, k) in enumerate(layers)]
    x0 = _inputs(M, layers[0][0], 1, 2, seed=1299)[0]
    need = max(binding.gemm_workspace_bytes(M, K, N, k) for K, N, k in layers)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    acts = [dev_bf16(x0)] + [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _, N, _ in layers]
    dev_w = [(dev_codes(c), dev_bf16(sc)) for c, sc in weights]
    torch.cuda.synchronize()
    for i, ((K, N, k), (dc, ds)) in enumerate(zip(layers, dev_w)):
        assert binding.abi_gemm_ws(acts[i].data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256,
                                   acts[i + 1].data_ptr(), ws.data_ptr(), need, s) == 0
    torch.cuda.synchronize()
    for i, ((K, N, k), (codes, scales)) in enumerate(zip(layers, weights)):
        x = host_bits(acts[i])           # the GPU's own input to this layer
        w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
        ref, refabs = oracle_gemm_par(oracle_lib, x, w)
        assert_gemm_close(host_bits(acts[i + 1]), ref, refabs, f"layer {i}")
    assert int(ws[: 1 << 20].count_nonzero()) == 0, "tile counters not left at zero"


def test_gemm_workspace_errors(tq):
    import torch
    from trellis_quantized_weight_gb300 import binding
    M, K, N, k = 4, 1024, 5000, 4
    x, codes, scales = _inputs(M, K, N, k, seed=3)
    dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    need = binding.gemm_workspace_bytes(M, K, N, k)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = (dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256, out.data_ptr())
    assert binding.abi_gemm_ws(*args, ws.data_ptr(), need - 1, s) == -7
    assert binding.abi_gemm_ws(*args, 0, need, s) == -7
    assert binding.abi_gemm_ws(*args, ws.data_ptr() + 4, need - 4, s) in (-4, -7)
    assert binding.abi_gemm_ws(*args, ws.data_ptr(), need, s) == 0
    # misaligned x (2-byte offset into a bf16 buffer)
    big = torch.zeros(M * K + 8, dtype=torch.bfloat16, device="cuda")
    assert binding.abi_gemm_ws(big.data_ptr() + 2, *args[1:], ws.data_ptr(), need, s) == -4
    torch.cuda.synchronize()


# ----------------------------------------------- full-size quantised-linear --
ALL_WORKLOADS = ["gemm_m5_k5120_n17408_k2", "gemm_m8_k5120_n17408_k3", "gemm_m15_k5120_n17408_k4",
                 "gemv_m1_k17408_n5120_k4", "prefill_m64_k5120_n17408_k4"]


@pytest.fixture(scope="module")
def full_inputs():
    from trellis_quantized_weight_gb300 import synth
    cache = {}

    def get(name):
        if name not in cache:
            cache.clear()
            wl = synth.WORKLOADS[name]
            cache[name] = (wl, *wl.generate())
        return cache[name]
    return get


@pytest.mark.parametrize("name", ALL_WORKLOADS)
def test_full_decode_bitexact(tq, oracle_lib, full_inputs, name):
    wl, x, codes, scales = full_inputs(name)
    got = host_bits(tq.decode(dev_codes(codes), dev_bf16(scales), wl.K, wl.k))
    want = oracle_decode_par(oracle_lib, codes, scales, wl.K, wl.N, wl.k)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("name", ALL_WORKLOADS)
def test_full_gemm(tq, oracle_lib, full_inputs, name):
    """Both product entries at full size against the oracle: trellis_gemm_ws (the
    caller's workspace, through the Python API) and trellis_gemm (no workspace
    argument, the library's static scratch), which must also agree bit for bit."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    wl, x, codes, scales = full_inputs(name)
    dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
    got = host_bits(tq.gemm(dx, dc, ds, wl.k))
    out = torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device="cuda")
    rc = binding.abi_gemm(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), wl.M, wl.K, wl.N, wl.k, 12, 256,
                          out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, binding.status_string(rc)
    got_abi = host_bits(out)
    w = oracle_decode_par(oracle_lib, codes, scales, wl.K, wl.N, wl.k)
    ref, refabs = oracle_gemm_par(oracle_lib, x, w)
    assert_gemm_close(got, ref, refabs, name)
    assert_gemm_close(got_abi, ref, refabs, name + " (trellis_gemm)")
    assert np.array_equal(got, got_abi)


def test_gemm_largest_m(tq, oracle_lib):
    """M = 65536, the largest accepted: 256 tensor-core launches of 256 rows.
    Checked against the oracle on sampled activation rows (the first and last
    rows, both sides of several launch boundaries, and random rows), with the
    rows after the output left untouched."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    M, K, N, k = 65536, 256, 130, 3
    x, codes, scales = _inputs(M, K, N, k, seed=9901)
    dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
    pad = 2
    out = torch.full(((M + pad) * N,), 0x7FC1, dtype=torch.int16, device="cuda")
    ws = torch.zeros(max(binding.gemm_workspace_bytes(M, K, N, k), 256), dtype=torch.uint8, device="cuda")
    rc = binding.abi_gemm_ws(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256, out.data_ptr(),
                             ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, binding.status_string(rc)
    torch.cuda.synchronize()
    assert binding.load().trellis_device_status(None) == 0
    bits = out.cpu().numpy().view(np.uint16)
    assert np.all(bits[M * N:] == 0x7FC1)
    got = bits[: M * N].reshape(M, N)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 255, 256, 257, 32767, 32768, 65279, 65280, 65535],
                                     rng.integers(0, M, 100)]))
    w = oracle_lib.decode(codes, scales, K, N, k)
    ref, refabs = oracle_lib.gemm_dense(x[rows], w)
    assert_gemm_close(got[rows], ref, refabs, "M=65536 sampled rows")


@pytest.mark.parametrize("M", [8, 64])
def test_gemm_long_k(tq, oracle_lib, M):
    """K = 51200 (200 blocks a row, 400 tensor-core stages): long reductions on
    both paths."""
    N, K, k = 200, 256 * 200, 2
    x, codes, scales = _inputs(M, K, N, k, seed=9911 + M)
    got = host_bits(tq.gemm(dev_bf16(x), dev_codes(codes), dev_bf16(scales), k))
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
    ref, refabs = oracle_gemm_par(oracle_lib, x, w)
    assert_gemm_close(got, ref, refabs, f"M={M} K={K}")


def test_wait_timeout_is_reported_and_the_context_stays_usable(tq, oracle_lib):
    """A bounded device-side wait that runs out (the self-test kernel waits on a
    barrier that nothing arrives on) is reported by trellis_device_status as
    TRELLIS_ERR_TIMEOUT once, the flag clears, and the next product is correct."""
    from trellis_quantized_weight_gb300 import binding
    lib = binding.load()
    assert lib.trellis_device_status(None) == 0
    assert lib.trellis_selftest_wait_timeout(None) == 0
    assert lib.trellis_device_status(None) == -6
    assert lib.trellis_device_status(None) == 0
    M, K, N, k = 64, 512, 300, 4
    x, codes, scales = _inputs(M, K, N, k, seed=9950)
    got = host_bits(tq.gemm(dev_bf16(x), dev_codes(codes), dev_bf16(scales), k))
    assert lib.trellis_device_status(None) == 0
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
    ref, refabs = oracle_gemm_par(oracle_lib, x, w)
    assert_gemm_close(got, ref, refabs, "after the self-test")


def test_concurrent_streams_give_the_sequential_bits(tq):
    """Calls on different streams, each with its own workspace, may overlap on
    the GPU: small-M products on two streams and a tensor-core product on a
    third, issued interleaved, give exactly the bits of the same calls run one
    at a time (each product's summation order is fixed by its launch shape)."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    lib = binding.load()
    cases = [(8, 1024, 3000, 3), (5, 2048, 1500, 2), (64, 1024, 2000, 4)]
    data = []
    for i, (M, K, N, k) in enumerate(cases):
        x, codes, scales = _inputs(M, K, N, k, seed=9960 + i)
        ws = torch.zeros(max(binding.gemm_workspace_bytes(M, K, N, k), 256), dtype=torch.uint8, device="cuda")
        data.append((M, K, N, k, dev_bf16(x), dev_codes(codes), dev_bf16(scales), ws))

    def call(d, out, stream):
        M, K, N, k, dx, dc, ds, ws = d
        rc = lib.trellis_gemm_ws(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256, out.data_ptr(),
                                 ws.data_ptr(), ws.numel(), stream.cuda_stream)
        assert rc == 0, binding.status_string(rc)

    main = torch.cuda.current_stream()
    want = []
    for d in data:
        o = torch.empty((d[0], d[2]), dtype=torch.bfloat16, device="cuda")
        call(d, o, main)
        torch.cuda.synchronize()
        want.append(o.view(torch.int16).cpu().numpy())
    streams = [torch.cuda.Stream() for _ in data]
    outs = [[torch.empty((d[0], d[2]), dtype=torch.bfloat16, device="cuda") for _ in range(6)] for d in data]
    torch.cuda.synchronize()
    for rep in range(6):
        for d, s, o in zip(data, streams, outs):
            call(d, o[rep], s)
    torch.cuda.synchronize()
    assert lib.trellis_device_status(None) == 0
    for i, o in enumerate(outs):
        for rep in range(6):
            assert np.array_equal(o[rep].view(torch.int16).cpu().numpy(), want[i]), (i, rep)


def test_host_threads_on_their_own_streams(tq):
    """Several host threads, each with its own stream and workspace, call the
    library at once: every result equals the single-threaded one."""
    import threading
    import torch
    from trellis_quantized_weight_gb300 import binding
    lib = binding.load()
    M, K, N, k = 8, 1024, 2500, 3
    x, codes, scales = _inputs(M, K, N, k, seed=9970)
    dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
    need = max(binding.gemm_workspace_bytes(M, K, N, k), 256)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws0 = torch.zeros(need, dtype=torch.uint8, device="cuda")
    assert lib.trellis_gemm_ws(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256, ref.data_ptr(),
                               ws0.data_ptr(), need, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    want = ref.view(torch.int16).cpu().numpy()
    nthreads, reps = 4, 5
    wss = [torch.zeros(need, dtype=torch.uint8, device="cuda") for _ in range(nthreads)]
    outs = [[torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(reps)] for _ in range(nthreads)]
    streams = [torch.cuda.Stream() for _ in range(nthreads)]
    torch.cuda.synchronize()
    errors = []

    def worker(t):
        try:
            torch.cuda.set_device(0)
            for r in range(reps):
                rc = lib.trellis_gemm_ws(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256,
                                         outs[t][r].data_ptr(), wss[t].data_ptr(), need, streams[t].cuda_stream)
                if rc != 0:
                    errors.append(rc)
        except Exception as e:   # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(nthreads)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for t in range(nthreads):
        for r in range(reps):
            assert np.array_equal(outs[t][r].view(torch.int16).cpu().numpy(), want), (t, r)


@pytest.mark.parametrize("M,K,N,k", [(8, 1024, 3000, 3), (64, 1024, 2000, 4), (300, 512, 700, 2)])
def test_cuda_graph_capture_replays_the_eager_bits(tq, M, K, N, k):
    """trellis_gemm_ws captured into a CUDA graph (no allocation or host sync
    inside the call; programmatic launches become graph edges) replays to the
    bits of the eager call, on the CUDA-core and the tensor-core paths."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    lib = binding.load()
    x, codes, scales = _inputs(M, K, N, k, seed=9980 + M)
    dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
    ws = torch.zeros(max(binding.gemm_workspace_bytes(M, K, N, k), 256), dtype=torch.uint8, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def call(stream_handle):
        return lib.trellis_gemm_ws(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256,
                                   out.data_ptr(), ws.data_ptr(), ws.numel(), stream_handle)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert call(s.cuda_stream) == 0
    torch.cuda.synchronize()
    want = out.view(torch.int16).cpu().numpy().copy()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        assert call(torch.cuda.current_stream().cuda_stream) == 0
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.view(torch.int16).cpu().numpy(), want)
    assert lib.trellis_device_status(None) == 0


def test_two_copies_of_the_library_in_one_process(tq, tmp_path):
    """A second copy of the library (another file, as when two versions are
    loaded into one process) keeps its own per-device state: both copies
    launch the shared-memory-heavy small-M kernel and give the same bits."""
    import shutil
    import torch
    from trellis_quantized_weight_gb300 import binding, build
    copy_path = str(tmp_path / "libtrellis_copy.so")
    shutil.copy(build.LIB_PATH, copy_path)
    libs = [binding.load(), ctypes.CDLL(copy_path)]
    M, K, N, k = 15, 1024, 1000, 4
    x, codes, scales = _inputs(M, K, N, k, seed=4711)
    dx, dc, ds = dev_bf16(x), dev_codes(codes), dev_bf16(scales)
    s = torch.cuda.current_stream().cuda_stream
    outs = []
    for lib in libs:
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        rc = lib.trellis_gemm(ctypes.c_void_p(dx.data_ptr()), ctypes.c_void_p(dc.data_ptr()),
                              ctypes.c_void_p(ds.data_ptr()), M, K, N, k, 12, 256, ctypes.c_void_p(out.data_ptr()),
                              ctypes.c_void_p(s))
        assert rc == 0, binding.status_string(rc)
        outs.append(host_bits(out))
    torch.cuda.synchronize()
    assert np.array_equal(outs[0], outs[1])
