"""trellis_gemm neither allocates nor synchronises.

trellis_gemm takes no workspace: the split-K scratch of the small-M product is
a static region of the library image.  These tests run in a fresh process
(the first call on a device is the one that used to allocate and synchronise):

* with the library's modules loaded eagerly, the device's free memory and
  torch's allocations are the same before and after the process's first
  trellis_gemm call, and after later calls on other geometries, and the first
  call returns while a long kernel enqueued before it on another stream is
  still running, so it did not synchronise the device;
* under the default lazy module loading the same holds for every call after
  the one that made the driver load the library's modules (that load itself
  can wait for work in flight: the driver's doing, not the call's);
* the result is bit for bit the one of trellis_gemm_ws.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import json, sys
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    from trellis_quantized_weight_gb300 import binding, synth

    torch.zeros(1, device="cuda")
    lib = binding.load()
    wl = synth.WORKLOADS["gemm_m8_k5120_n17408_k3"]
    x, codes, scales = wl.generate()
    dx = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    dc = torch.from_numpy(codes.view(np.int32)).cuda()
    ds = torch.from_numpy(scales.view(np.int16)).cuda().view(torch.bfloat16)
    M, K, N, k = wl.M, wl.K, wl.N, wl.k
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    small = [torch.from_numpy(a.view(np.int16 if i != 1 else np.int32)).cuda()
             for i, a in enumerate(synth.small(8, 1024, 3000, 3, seed=77).generate())]
    out_small = torch.empty((8, 3000), dtype=torch.bfloat16, device="cuda")
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    if WARM:
        # one call first: the driver loads the library's modules (under lazy
        # loading that load can wait for work in flight on the device)
        assert lib.trellis_gemm(small[0].data_ptr(), small[1].data_ptr(), small[2].data_ptr(), 8, 1024, 3000, 3,
                                12, 256, out_small.data_ptr(), main.cuda_stream) == 0
    torch.cuda.synchronize()
    res = {}

    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    # a kernel of about a second on another stream, enqueued before the first call
    with torch.cuda.stream(side):
        torch.cuda._sleep(int(2.5e9))
        busy = torch.cuda.Event()
        busy.record(side)
    rc = lib.trellis_gemm(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256,
                          out.data_ptr(), main.cuda_stream)
    res["rc"] = rc
    res["side_still_running"] = not busy.query()
    torch.cuda.synchronize()
    res["free_delta_first_call"] = torch.cuda.mem_get_info()[0] - free0
    res["alloc_delta_first_call"] = torch.cuda.memory_allocated() - alloc0
    for _ in range(2):
        rc2 = lib.trellis_gemm(small[0].data_ptr(), small[1].data_ptr(), small[2].data_ptr(), 8, 1024, 3000, 3,
                               12, 256, out_small.data_ptr(), main.cuda_stream)
        res["rc"] = res["rc"] or rc2
    torch.cuda.synchronize()
    res["free_delta_later_calls"] = torch.cuda.mem_get_info()[0] - free0
    ref = torch.empty_like(out)
    ws = torch.zeros(binding.gemm_workspace_bytes(M, K, N, k), dtype=torch.uint8, device="cuda")
    assert lib.trellis_gemm_ws(dx.data_ptr(), dc.data_ptr(), ds.data_ptr(), M, K, N, k, 12, 256,
                               ref.data_ptr(), ws.data_ptr(), ws.numel(), main.cuda_stream) == 0
    torch.cuda.synchronize()
    res["equal_to_ws"] = bool(torch.equal(out.view(torch.int16), ref.view(torch.int16)))
    print("RESULT " + json.dumps(res))
""")


def _run_child(module_loading: str, warm: bool) -> dict:
    import json
    env = dict(os.environ, CUDA_MODULE_LOADING=module_loading)
    src = "ROOT = " + repr(ROOT) + "\nWARM = " + repr(warm) + "\n" + CHILD
    r = subprocess.run([sys.executable, "-c", src], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    return json.loads(line[len("RESULT "):])


def test_first_call_allocates_nothing_and_does_not_synchronise():
    """With the modules loaded eagerly, the process's first call allocates nothing
    and does not wait for other streams."""
    res = _run_child("EAGER", warm=False)
    assert res["rc"] == 0
    assert res["side_still_running"], "the first trellis_gemm call waited for other streams' work"
    assert res["alloc_delta_first_call"] == 0
    assert res["free_delta_first_call"] == 0, f"device free memory changed by {res['free_delta_first_call']}"
    assert res["free_delta_later_calls"] == 0
    assert res["equal_to_ws"]


def test_calls_after_module_loading_under_lazy_loading():
    """Under the default lazy module loading the driver places the library's code
    and static scratch in device memory when a call first needs them, and that
    load can wait for work in flight.  Once loaded, calls (here on a new
    geometry served by the same kernel) allocate nothing and do not wait for
    other streams."""
    res = _run_child("LAZY", warm=True)
    assert res["rc"] == 0
    assert res["side_still_running"], "trellis_gemm waited for other streams' work"
    assert res["alloc_delta_first_call"] == 0
    assert res["free_delta_first_call"] == 0
    assert res["free_delta_later_calls"] == 0
    assert res["equal_to_ws"]
