"""GPU parity of token packing (trellis_gemm_packed): each group's output
against the oracle product of that group's rows (product tolerance), and bit
for bit against the rows of one trellis_gemm call on the concatenated x (the
same product, so the same bits).  Nothing is written past a group's rows."""
import ctypes

import numpy as np
import pytest

from helpers import assert_gemm_close, dev_bf16, dev_codes, oracle_decode_par, oracle_gemm_par

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


def _inputs(M, K, N, k, seed):
    from trellis_quantized_weight_gb300 import synth
    return synth.small(M, K, N, k, seed).generate()


def _run_packed(lib, xs, rows, dc, ds, K, N, k, L, ws, pad=3):
    """Raw ABI call with sentinel-padded outputs; returns the host bits of each group's rows."""
    import torch
    outs = [torch.full(((r + pad) * N,), 0x7FC1, dtype=torch.int16, device="cuda") for r in rows]
    xp = (ctypes.c_void_p * len(xs))(*[x.data_ptr() for x in xs])
    op = (ctypes.c_void_p * len(outs))(*[o.data_ptr() for o in outs])
    rp = (ctypes.c_int * len(rows))(*rows)
    rc = lib.trellis_gemm_packed(xp, rp, len(rows), dc.data_ptr(), ds.data_ptr(), K, N, k, L, 256, op,
                                 ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.trellis_status_string(rc).decode()
    torch.cuda.synchronize()
    got = []
    for o, r in zip(outs, rows):
        bits = o.cpu().numpy().view(np.uint16)
        assert np.all(bits[r * N:] == 0x7FC1), "rows beyond the group were written"
        got.append(bits[: r * N].reshape(r, N))
    return got


@pytest.mark.parametrize("rows,k,L", [
    ([3, 5, 1, 7], 3, 12),     # M = 16 on the CUDA cores
    ([1, 1], 4, 12),           # two single-token sequences
    ([20, 40, 4], 4, 12),      # M = 64 on the tensor cores
    ([100, 50, 150, 3], 2, 12),  # M = 303: two 256-row launches
    ([6], 4, 12),              # one group: in place
    ([2, 3], 5, 16),           # another geometry
])
def test_packed_matches_oracle_and_concatenated_product(tq, oracle_lib, rows, k, L):
    import torch
    from trellis_quantized_weight_gb300 import binding
    lib = binding.load()
    N, K = 300, 512
    M = sum(rows)
    x, codes, scales = _inputs(M, K, N, k, seed=8100 + M + 10 * k + L)
    dx = dev_bf16(x)
    xs = [dx[a:b].contiguous() for a, b in zip(np.cumsum([0] + rows[:-1]), np.cumsum(rows))]
    dc, ds = dev_codes(codes), dev_bf16(scales)
    ws = torch.zeros(max(binding.gemm_packed_workspace_bytes(rows, K, N, k, L), 256), dtype=torch.uint8,
                     device="cuda")
    got = _run_packed(lib, xs, rows, dc, ds, K, N, k, L, ws)
    whole = tq.gemm(dx, dc, ds, k, L=L).view(torch.int16).cpu().numpy().view(np.uint16)
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k, L=L)
    pos = 0
    for g, r in enumerate(rows):
        assert np.array_equal(got[g], whole[pos:pos + r]), f"group {g} differs from the concatenated product"
        ref, refabs = oracle_gemm_par(oracle_lib, x[pos:pos + r], w)
        assert_gemm_close(got[g], ref, refabs, f"group {g} rows {r}")
        pos += r


def test_packed_workspace_reused_across_group_shapes(tq, oracle_lib):
    """One zero-filled workspace serves calls whose packed M moves between the
    CUDA-core path (counters in use) and the tensor cores (packed copies only)."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    lib = binding.load()
    N, K, k = 260, 1024, 4
    shapes = [[3, 5], [30, 40, 10], [2, 2, 2, 2], [16], [7, 9], [50, 1]]
    need = max(binding.gemm_packed_workspace_bytes(r, K, N, k) for r in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    _, codes, scales = _inputs(1, K, N, k, seed=8200)
    dc, ds = dev_codes(codes), dev_bf16(scales)
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
    for i, rows in enumerate(shapes):
        x, _, _ = _inputs(sum(rows), K, N, k, seed=8300 + i)
        dx = dev_bf16(x)
        xs = [dx[a:b].contiguous() for a, b in zip(np.cumsum([0] + rows[:-1]), np.cumsum(rows))]
        got = _run_packed(lib, xs, rows, dc, ds, K, N, k, 12, ws)
        pos = 0
        for g, r in enumerate(rows):
            ref, refabs = oracle_gemm_par(oracle_lib, x[pos:pos + r], w)
            assert_gemm_close(got[g], ref, refabs, f"call {i} group {g}")
            pos += r


def test_packed_python_api(tq, oracle_lib):
    """binding.gemm_packed returns one [rows_g, N] tensor per group."""
    from trellis_quantized_weight_gb300 import gemm_packed
    N, K, k, rows = 200, 768, 3, [4, 1, 6]
    x, codes, scales = _inputs(sum(rows), K, N, k, seed=8400)
    dx = dev_bf16(x)
    xs = [dx[0:4].contiguous(), dx[4:5].contiguous(), dx[5:11].contiguous()]
    outs = gemm_packed(xs, dev_codes(codes), dev_bf16(scales), k)
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
    pos = 0
    for o, r in zip(outs, rows):
        assert tuple(o.shape) == (r, N)
        bits = o.view(__import__("torch").int16).cpu().numpy().view(np.uint16)
        ref, refabs = oracle_gemm_par(oracle_lib, x[pos:pos + r], w)
        assert_gemm_close(bits, ref, refabs)
        pos += r


def test_packed_many_groups(tq, oracle_lib):
    """100 groups (two gather and two scatter launches of at most 64 groups),
    mostly single rows: every group matches the concatenated product bit for bit."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    lib = binding.load()
    rng = np.random.default_rng(11)
    rows = [int(r) for r in rng.integers(1, 4, 100)]
    rows[:60] = [1] * 60
    N, K, k = 220, 512, 3
    M = sum(rows)
    x, codes, scales = _inputs(M, K, N, k, seed=8500)
    dx = dev_bf16(x)
    offs = np.cumsum([0] + rows)
    xs = [dx[a:b].contiguous() for a, b in zip(offs[:-1], offs[1:])]
    dc, ds = dev_codes(codes), dev_bf16(scales)
    ws = torch.zeros(binding.gemm_packed_workspace_bytes(rows, K, N, k), dtype=torch.uint8, device="cuda")
    got = _run_packed(lib, xs, rows, dc, ds, K, N, k, 12, ws)
    whole = tq.gemm(dx, dc, ds, k).view(torch.int16).cpu().numpy().view(np.uint16)
    for g, (a, b) in enumerate(zip(offs[:-1], offs[1:])):
        assert np.array_equal(got[g], whole[a:b]), g
