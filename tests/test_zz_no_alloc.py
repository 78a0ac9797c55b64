"""trellis_gemm_noalloc: the decode-and-multiply for callers that cannot allocate.

Some callers may not call cudaMalloc: code running inside an allocator or a
memory-pool callback (allocating there would re-enter the allocator), processes
that reserve all device memory up front (nothing is left to allocate), or
runtimes that forbid allocation on their hot path (an allocation can
synchronise the device).  trellis_gemm_noalloc serves them by taking its
split-K scratch from a fixed array inside the library.

Each case calls it twice in a row through the C ABI (the second call finds the
scratch exactly as the first left it).  Both calls run the same kernel, plan and
fixed reduction order as trellis_gemm_ws, so both outputs must equal its output
bit for bit; one case is also checked against the CPU oracle within the product
tolerance max(2 bf16 ulp, 1e-4 * sum_k |w_k x_k|), and one checks that calls
after the first leave the device's free memory unchanged.  This file is
collected last and also passes on its own in a fresh process.
"""
import numpy as np
import pytest

from helpers import assert_gemm_close, host_bits, oracle_decode_par, oracle_gemm_par

pytestmark = pytest.mark.gpu

FAKE = 0x10000   # aligned, never dereferenced: only in calls that validation rejects before any
                 # launch (a call that could pass validation must use real device buffers)
SCRATCH_LIMIT = 16 << 20


@pytest.fixture(scope="module")
def lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from trellis_quantized_weight_gb300 import binding, build
    build.build()
    return binding.load()


def _dev(a, torch, bf16):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if bf16 else np.int32)).cuda()
    return t.view(torch.bfloat16) if bf16 else t


def _inputs(M, K, N, k, seed, torch):
    from trellis_quantized_weight_gb300 import synth
    x, codes, scales = synth.small(M, K, N, k, seed=seed).generate()
    return (x, codes, scales), (_dev(x, torch, True), _dev(codes, torch, False), _dev(scales, torch, True))


def _gemm_ws(lib, dx, dc, ds, M, K, N, k, L, s, torch):
    from trellis_quantized_weight_gb300 import binding
    need = binding.gemm_workspace_bytes(M, K, N, k, L)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert lib.trellis_gemm_ws(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, L, 256,
                               ref.data_ptr(), ws.data_ptr(), ws.numel(), s) == 0
    return ref


def _noalloc_twice(lib, dx, dc, ds, M, K, N, k, L, s, torch):
    from trellis_quantized_weight_gb300 import binding
    outs = []
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.trellis_gemm_noalloc(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, L, 256,
                                      out.data_ptr(), s)
        assert rc == 0, binding.status_string(rc)
        torch.cuda.synchronize()
        outs.append(out)
    return outs


@pytest.mark.parametrize("M,K,N,k", [
    (8, 5120, 17408, 3),       # the M = 8 quantised-linear shape
    (15, 5120, 6000, 4),
    (1, 17408, 5120, 4),
    (5, 256, 40000, 2),
])
def test_noalloc_matches_gemm_ws_bit_for_bit(lib, M, K, N, k):
    import torch
    _, (dx, dc, ds) = _inputs(M, K, N, k, 4242 + M + k, torch)
    s = torch.cuda.current_stream().cuda_stream
    ref = _gemm_ws(lib, dx, dc, ds, M, K, N, k, 12, s, torch)
    for call, out in enumerate(_noalloc_twice(lib, dx, dc, ds, M, K, N, k, 12, s, torch)):
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call} differs"


def test_noalloc_against_the_oracle(lib, oracle_lib):
    """Both calls within the product tolerance of the CPU oracle (several tiles, ragged N)."""
    import torch
    M, K, N, k = 8, 1024, 3001, 3
    (x, codes, scales), (dx, dc, ds) = _inputs(M, K, N, k, 4400, torch)
    s = torch.cuda.current_stream().cuda_stream
    w = oracle_decode_par(oracle_lib, codes, scales, K, N, k)
    ref, refabs = oracle_gemm_par(oracle_lib, x, w)
    for call, out in enumerate(_noalloc_twice(lib, dx, dc, ds, M, K, N, k, 12, s, torch)):
        assert_gemm_close(host_bits(out), ref, refabs, f"noalloc call {call}")


def test_noalloc_allocates_nothing_after_its_first_call(lib):
    """After the first call on this device (set-up, module loading) further calls,
    on another geometry served by the same kernel, change neither torch's
    allocations nor the device's free memory."""
    import torch
    from trellis_quantized_weight_gb300 import binding
    s = torch.cuda.current_stream().cuda_stream
    M, k = 8, 3
    _, a = _inputs(M, 2048, 3000, k, 4500, torch)
    _, b = _inputs(M, 5120, 17408, k, 4501, torch)
    outs = [torch.empty((M, 3000), dtype=torch.bfloat16, device="cuda"),
            torch.empty((M, 17408), dtype=torch.bfloat16, device="cuda")]
    assert lib.trellis_gemm_noalloc(a[0].data_ptr(), a[1].data_ptr(), a[2].data_ptr(), M, 2048, 3000, k, 12,
                                    256, outs[0].data_ptr(), s) == 0
    torch.cuda.synchronize()

    def free_bytes():   # cudaMemGetInfo
        return torch.cuda.mem_get_info()[0]

    before = (torch.cuda.memory_allocated(), free_bytes())
    for _ in range(3):
        rc = lib.trellis_gemm_noalloc(b[0].data_ptr(), b[1].data_ptr(), b[2].data_ptr(), M, 5120, 17408, k, 12,
                                      256, outs[1].data_ptr(), s)
        assert rc == 0, binding.status_string(rc)
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(), free_bytes())
    assert after == before


def test_noalloc_rejects_bad_arguments(lib):
    """Same checks, in the same order, as trellis_gemm (nothing is launched)."""
    for fn in (lib.trellis_gemm_noalloc, lib.trellis_gemm):
        assert fn(0, FAKE, FAKE, 8, 5120, 64, 3, 12, 256, FAKE, None) == -1
        assert fn(FAKE + 2, FAKE, FAKE, 8, 5120, 64, 3, 12, 256, FAKE, None) == -4
        # M outside 1..65536 (every M inside it is accepted and would launch)
        assert fn(FAKE, FAKE, FAKE, 0, 5120, 64, 3, 12, 256, FAKE, None) == -3
        assert fn(FAKE, FAKE, FAKE, 65537, 5120, 64, 3, 12, 256, FAKE, None) == -3
        assert fn(FAKE, FAKE, FAKE, 8, 5000, 64, 3, 12, 256, FAKE, None) == -2
        # two faults at once: the unsupported M is reported before the misaligned x
        assert fn(FAKE + 2, FAKE, FAKE, 0, 5120, 64, 3, 12, 256, FAKE, None) == -3
        # a bad geometry is reported before a misaligned output
        assert fn(FAKE, FAKE, FAKE, 8, 5000, 64, 3, 12, 256, FAKE + 1, None) == -2


def test_every_accepted_geometry_fits_the_fixed_scratch(lib):
    """On this device the scratch of every geometry the product accepts, for every
    M on the split-K path and every bit width, stays within the 16 MiB array (it
    depends on the SM count, not on N or K), so the entry's too-large check only
    guards larger devices."""
    from trellis_quantized_weight_gb300 import binding
    largest = 0
    for M in range(1, 17):
        for k, L in [(2, 12), (3, 12), (4, 12), (1, 9), (5, 16), (8, 24)]:
            for K, N in [(256, 1), (5120, 17408), (17408, 5120), (256, 200000)]:
                largest = max(largest, binding.gemm_workspace_bytes(M, K, N, k, L))
    assert 0 < largest <= SCRATCH_LIMIT


def test_every_accepted_geometry_fits_trellis_gemm_scratch(lib):
    """The same for trellis_gemm's 4 MiB static scratch: on this device no
    single-matrix geometry it accepts needs more, so it never answers
    TRELLIS_ERR_WORKSPACE here."""
    from trellis_quantized_weight_gb300 import binding
    largest = 0
    for M in range(1, 17):
        for k, L in [(2, 12), (3, 12), (4, 12), (1, 9), (5, 16), (8, 24)]:
            for K, N in [(256, 1), (5120, 17408), (17408, 5120), (256, 200000)]:
                largest = max(largest, binding.gemm_workspace_bytes(M, K, N, k, L))
    assert 0 < largest <= 4 << 20


@pytest.mark.parametrize("M,K,N,k,L", [(6, 1024, 3000, 5, 16), (40, 512, 1000, 1, 9)])
def test_noalloc_general_geometry(lib, M, K, N, k, L):
    """The no-allocation entry on a geometry outside k in {2,3,4}, L = 12, on
    both paths, bit for bit against trellis_gemm_ws."""
    import torch
    _, (dx, dc, ds) = _inputs(M, K, N, k, 4300 + M + k, torch)
    s = torch.cuda.current_stream().cuda_stream
    ref = _gemm_ws(lib, dx, dc, ds, M, K, N, k, L, s, torch)
    for call, out in enumerate(_noalloc_twice(lib, dx, dc, ds, M, K, N, k, L, s, torch)):
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call} differs"
