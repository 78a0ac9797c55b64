"""The trace build of the library (-DTRELLIS_TRACE, trellis_quantized_weight_gb300/trace.py).

Its stamps must not change a single output bit, and they must describe one
launch consistently: every CTA stamped its entry, its loop end and its unit
count; every warp left the loop before its tickets were answered, before its
reduction's sums were complete and before its end.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def traced():
    from trellis_quantized_weight_gb300 import trace
    return trace.load_traced(trace.build_traced())


@pytest.mark.parametrize("M,K,N,k", [(15, 2560, 3001, 4), (5, 5120, 2000, 2), (8, 1024, 777, 3), (1, 4096, 1500, 4)])
def test_trace_build_is_bit_identical_and_consistent(traced, M, K, N, k):
    from trellis_quantized_weight_gb300 import binding, synth, trace
    lib = binding.load()
    x, c, sc = synth.small(M, K, N, k, seed=31 * M + k).generate()
    dx = torch.from_numpy(x.view(np.int16)).cuda()
    dc = torch.from_numpy(c.view(np.int32)).cuda()
    ds = torch.from_numpy(sc.view(np.int16)).cuda()
    s = torch.cuda.current_stream().cuda_stream
    ref = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    got = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    assert lib.trellis_gemm(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256, ref.data_ptr(), s) == 0
    buf = torch.zeros(trace.MAX_CTAS * trace.CTA_WORDS, dtype=torch.int64, device="cuda")
    assert traced.trellis_trace_attach(buf.data_ptr(), buf.numel() * 8) == 0
    try:
        assert traced.trellis_gemm(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256,
                                   got.data_ptr(), s) == 0
        torch.cuda.synchronize()
        assert traced.trellis_device_status(None) == 0
    finally:
        traced.trellis_trace_attach(None, 0)
    assert torch.equal(got, ref)

    rec = buf.view(trace.MAX_CTAS, trace.CTA_WORDS).cpu().numpy()
    ctas = int(np.count_nonzero(rec[:, 1]))
    assert ctas > 0 and np.all(rec[:ctas, 1] != 0) and np.all(rec[ctas:, 1] == 0)
    assert np.all(rec[:ctas, 2] >= rec[:ctas, 1])
    units = rec[:ctas, 3]
    # the units of all CTAs cover every (tile-group, block) once
    nblocks = K // 256
    assert units.sum() % nblocks == 0 and units.min() >= 0
    w = rec[:ctas, 8:].reshape(ctas, 16, 8)
    left = w[:, :, 0] != 0
    assert left.any()
    for field in (1, 2, 3):
        v = w[:, :, field]
        set_ = left & (v != 0)
        assert np.all(v[set_] >= w[:, :, 0][set_])
    both = left & (w[:, :, 1] != 0) & (w[:, :, 2] != 0)
    assert np.all(w[:, :, 2][both] >= w[:, :, 1][both])
    assert np.all(w[:, :, 3][left] != 0)
    summary = trace.summarise(rec)
    assert summary["ctas"] == ctas
